// decode.cuh - split-KV attention for short query lengths (decode), the
// HBM-bound path of the AttentionPlugin ("TensorRT Plugins Guide":
// vanilla decoding attention) with the TRT_Attention semantics of
// "TensorRT Custom Operator Schemas".
//
// Work: pairs (batch b, KV head g, chunk of 8 or 16 query rows), each with
// the 32-key tiles of the batch's key extent.  The query rows of a pair are
// the (token, head) pairs of the G heads of g, 8 at a time: the N = 8 of the
// m16n8k16 MMA in the transposed products S^T = K Q^T and O^T = V^T P^T
// (keys, then head dims, on M), so no MMA row is wasted at G = 8 and K and
// V are read once from HBM for all G query heads of the KV head.  Where a
// (batch, KV head) holds more than 8 rows (tree decoding, G = 16), the
// 16-bit tile takes 16 rows per pair as two N-blocks that share every K and
// V fragment, so the keys are streamed half as often.
// All tiles of all pairs form one batch-major line that is cut into equal
// contiguous ranges, one per warp of the persistent grid, so that every
// warp streams the same number of tiles and none is left finishing a long
// unit alone at the end.  Each CTA validates the lengths and lays out the
// line itself (no scheduler launch).  A warp streams its range's K/V tiles
// with TMA through its own ring of a few stages (128-byte swizzle), straight
// across pair boundaries, and keeps an online softmax in fp32 registers.
// A pair inside one range is written to Y by its warp; a pair cut by range
// ends leaves a partial (O, m, l) per warp, and the last of its warps to
// finish (atomic ticket) merges them in warp order and writes Y.
//
// FP8 KV cache ("TensorRT Plugins Guide", AttentionPlugin: kv_cache_type
// FP8): K and V hold OCP E4M3FN codes with one dequantisation scale each.
// The tiles arrive as bytes (half the HBM traffic), each thread converts its
// MMA operand fragments to f16/bf16 in registers (exactly: every E4M3 value
// is an f16 and a bf16 value), the K scale is folded into the softmax scale
// and the V scale into the final 1/l.  An fp8 CTA runs 8 warps, since a
// tile carries half the bytes and more arithmetic per byte.
#pragma once
#include <type_traits>
#include <cuda.h>
#include "device_common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace rga {

// KV8: K and V are E4M3 codes (one byte per element).
template <int D, bool KV8>
struct DecLayout {
    static constexpr int NW = KV8 ? DEC_WARPS_KV8 : DEC_WARPS;   // warps per CTA
    static constexpr int THREADS = NW * 32;
    static constexpr int STAGES = KV8 ? DEC_STAGES_KV8 : DEC_STAGES;
    static constexpr int BLK = DEC_KEYS * 128;          // 16-bit: 32 rows x 64 columns x 2 bytes
    static constexpr int TILE = KV8 ? DEC_KEYS * D : (D / 64) * BLK;   // one K or V tile
    static constexpr int STAGE = 2 * TILE;               // K + V
    static constexpr int WARP_RING = STAGES * STAGE;
    static constexpr int RING = NW * WARP_RING;
    static constexpr int BAR_OFF = RING;
    static constexpr int SCR_OFF = BAR_OFF + NW * STAGES * 8 + 64;   // prefix scratch
    static constexpr int TPRE_OFF = SCR_OFF + (THREADS + 1) * 4 + 12;
    static constexpr int PPRE_OFF = TPRE_OFF + (DEC_MAX_B + 1) * 4;
    static constexpr int BYTES = PPRE_OFF + (DEC_MAX_B + 1) * 4 + 64;
    static constexpr int ALLOC = BYTES + 1024;
    static_assert(ALLOC <= 232448, "shared memory per CTA");
};

template <bool BF16>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    if constexpr (BF16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
            "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
            "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                        uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                          uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// Byte offset of 16-byte chunk `ch` (8 elements) of row `row` in a
// 128-byte-swizzled tile made of 64-column blocks of `blk` bytes.
__device__ __forceinline__ uint32_t swz(int row, int ch, int blk) {
    return (ch >> 3) * blk + row * 128 + (((ch & 7) ^ (row & 7)) << 4);
}

// Loads the K and V tiles of keys [j0, j0 + DEC_KEYS) of batch b, KV head
// g.  Paged cache: the tile lies in one page (page_size is a multiple of
// DEC_KEYS); pk / pv are its K and V pages, looked up by the caller, and
// the pools' tensor maps are [num_pages, Hkv, page_size, D].
template <bool KV8, bool PAGED>
__device__ __forceinline__ void dec_tma(const AttnParams &p, const TensorMaps &tm,
                                        const SeqInfo &s, int b, int g, int j0, uint8_t *dst,
                                        uint64_t *bar, int D, int pk, int pv) {
    int rk = j0, rv = j0, zk = b, zv = b;   // padded / paged coordinates (row, outer)
    if constexpr (PAGED) {
        rk = rv = j0 % p.page_size;
        zk = pk;
        zv = pv;
    }
    // (debug checks) the tile starts inside the sequence, in the cache or in
    // pages of the pools; a skipped load still completes its transactions
    if (!dbg_ok(j0 >= 0 && j0 < s.kv_len && g >= 0 && g < p.Hkv &&
                (PAGED ? pk >= 0 && pk < p.num_pages && pv >= 0 && pv < p.num_pages
                       : p.kv_packed ? s.kv_off + j0 < p.kv_seq : j0 < p.kv_seq && b < p.B),
                p.status)) {
        const uint32_t bytes = 2 * (KV8 ? DEC_KEYS * D : (D / 64) * DEC_KEYS * 128);
        mbar_arrive_expect_tx(bar, bytes);
        mbar_complete_tx(bar, bytes);
        return;
    }
    if constexpr (KV8) {   // one box of DEC_KEYS rows x D bytes per tensor
        const int tile = DEC_KEYS * D;
        mbar_arrive_expect_tx(bar, 2 * tile);
        if (p.kv_packed) {
            tma_load_3d(dst, &tm.k, bar, 0, g, s.kv_off + j0);
            tma_load_3d(dst + tile, &tm.v, bar, 0, g, s.kv_off + j0);
        } else {
            tma_load_4d(dst, &tm.k, bar, 0, rk, g, zk);
            tma_load_4d(dst + tile, &tm.v, bar, 0, rv, g, zv);
        }
        return;
    }
    const int tile = (D / 64) * DEC_KEYS * 128;
    mbar_arrive_expect_tx(bar, 2 * tile);
    for (int blk = 0; blk < D / 64; ++blk) {
        uint8_t *kd = dst + blk * DEC_KEYS * 128;
        uint8_t *vd = dst + tile + blk * DEC_KEYS * 128;
        if (p.kv_packed) {
            tma_load_3d(kd, &tm.k, bar, blk * 64, g, s.kv_off + j0);
            tma_load_3d(vd, &tm.v, bar, blk * 64, g, s.kv_off + j0);
        } else {
            tma_load_4d(kd, &tm.k, bar, blk * 64, rk, g, zk);
            tma_load_4d(vd, &tm.v, bar, blk * 64, rv, g, zv);
        }
    }
}

// One row: the query token/head it stands for, and its limits.
struct DecRow {
    bool valid;
    int i, h, lim;
    long long qoff, mrow;
};

__device__ __forceinline__ DecRow dec_row(const AttnParams &p, const SeqInfo &s, int b, int g,
                                          int R, int rows, int k1) {
    DecRow r;
    r.valid = R < rows;
    const int t = r.valid ? R / p.G : 0, hh = r.valid ? R % p.G : 0;
    r.i = t;
    r.h = g * p.G + hh;
    r.lim = r.valid ? min(causal_limit(p.causal, t, s), k1 - 1) : -1;
    r.qoff = p.q_packed ? ((long long)(s.q_off + t) * p.Hq + r.h) * p.D
                        : (((long long)b * p.Hq + r.h) * p.q_seq + t) * p.D;
    r.mrow = (p.mask && r.valid) ? mask_row(p, b, r.h, t) : 0;
    return r;
}

// Byte offset of 16-byte chunk `ch` of key row `row` in an fp8 tile of
// D-byte rows as the TMA writes it: 128-byte swizzle for D = 128 (chunk
// XOR row % 8), 64-byte swizzle for D = 64 (chunk XOR (row / 2) % 4).
template <int D>
__device__ __forceinline__ uint32_t off8(int row, int ch) {
    if constexpr (D == 128) return row * 128 + ((ch ^ (row & 7)) << 4);
    else return row * 64 + ((ch ^ ((row >> 1) & 3)) << 4);
}

__device__ __forceinline__ void lds128(uint32_t addr, uint32_t (&w)[4]) {
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(addr));
}
__device__ __forceinline__ void lds64(uint32_t addr, uint32_t &w0, uint32_t &w1) {
    asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(w0), "=r"(w1) : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// Scale, mask and online softmax ('none': scale and mask only) of one
// 32-key tile of a transposed product S^T (keys on M, the pair's 8 query
// rows on N): element (mb, e) is key j0 + 16 mb + lane/4 + 8 (e / 2) of row
// rr[e % 2] (rows 2c and 2c + 1, c = lane % 4).  Leaves P^T in sacc and
// rescales O^T (o[m][e] belongs to row rr[e % 2]) and l.
template <int D, bool SOFTMAX>
__device__ __forceinline__ void dec_normalize_t(const AttnParams &p, const DecRow (&rr)[2],
                                                float (&sacc)[2][4], int j0,
                                                float (&o)[D / 16][4], float (&m_r)[2],
                                                float (&l_r)[2], float sc) {
    constexpr int NO = D / 16;
    const int r = (threadIdx.x & 31) >> 2;
    float mx[2] = {-INFINITY, -INFINITY};
    // one copy of the loop per mask type (MK: -1 none, else the rga_dtype),
    // so that no iteration carries the loads of the other types
    auto scores = [&](auto mk) {
        constexpr int MK = decltype(mk)::value;
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const DecRow &R = rr[e & 1];
                const int j = j0 + 16 * mb + r + 8 * (e >> 1);
                bool ok = j <= R.lim;
                float add = 0.f;
                if constexpr (MK >= 0)
                    if (ok) ok = mask_at_t<MK>(p, p.md[3] == 1 ? R.mrow : R.mrow + j, add);
                const float v = sacc[mb][e] * sc + (SOFTMAX ? add * 1.4426950408889634f : add);
                sacc[mb][e] = ok ? v : (SOFTMAX ? -INFINITY : 0.f);
                mx[e & 1] = fmaxf(mx[e & 1], sacc[mb][e]);
            }
    };
    if (!p.mask) scores(std::integral_constant<int, -1>{});
    else if (p.mask_dtype == 3) scores(std::integral_constant<int, 3>{});
    else if (p.mask_dtype == 0) scores(std::integral_constant<int, 0>{});
    else if (p.mask_dtype == 1) scores(std::integral_constant<int, 1>{});
    else scores(std::integral_constant<int, 2>{});
    if (SOFTMAX) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int m = 4; m < 32; m <<= 1) mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], m));
        // O and l need rescaling only when a row's running max grew (alpha
        // is exactly 1 otherwise); the test is warp-uniform
        const float mn0 = fmaxf(m_r[0], mx[0]), mn1 = fmaxf(m_r[1], mx[1]);
        if (__any_sync(0xffffffffu, mn0 > m_r[0] || mn1 > m_r[1])) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float m_new = i ? mn1 : mn0;
                const float mu = (m_new == -INFINITY) ? 0.f : m_new;
                const float alpha = ex2(m_r[i] - mu);
                l_r[i] *= alpha;
#pragma unroll
                for (int m = 0; m < NO; ++m) { o[m][i] *= alpha; o[m][i + 2] *= alpha; }
            }
        }
        m_r[0] = mn0;
        m_r[1] = mn1;
        const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sacc[mb][e] = ex2(sacc[mb][e] - ((e & 1) ? mu1 : mu0));
                l_r[e & 1] += sacc[mb][e];
            }
    }
}

// dec_tile for an fp8 KV cache, kb/vb holding E4M3 codes that each thread
// converts in registers.  Both products are transposed so that the MMA's
// 8-wide N dimension holds the pair's 8 query rows and nothing is wasted:
//   S^T = K Q^T:  M = keys (two blocks of 16), N = rows, K = head dims;
//   O^T = V^T P^T: M = head dims (D/16 blocks), N = rows, K = keys.
// S^T is an f16 product whatever the input type: qb holds Q as f16 (bf16
// queries were scaled by a power of two into f16 range when the pair
// started) and a single cvt converts two key codes exactly.  The head dims
// of the S^T contraction are permuted (lane c = lane % 4 takes dims
// [c D/4, (c+1) D/4) of its key rows, four per k-step; Q was loaded the
// same way) so that a thread's K codes are contiguous.  P^T reaches the B
// fragment layout by an 8x8 transpose (movmatrix) of the S^T accumulator.
// V^T's M rows are permuted too: in dim block m, M-row r stands for dim
// (D/8) r + 2m and M-row r + 8 for dim (D/8) r + 2m + 1, so a thread reads
// D/8 contiguous codes from each of four key rows and pairs keys with byte
// permutes.  Accumulator o[m][e] therefore holds row 2c + e % 2, dim
// (D/8) (lane / 4) + 2m + e / 2.  Rows rr[0..1] are rows 2c and 2c + 1.
// With softmax, P (in [0, 1]) and V enter the P V product as f16 whatever
// the input type (every E4M3 value is an f16; f16 holds P more finely than
// bf16; P below 2^-24 flushes to zero, far inside the tolerance); 'none'
// leaves P unbounded and keeps the input type.
template <int D, bool BF16, bool SOFTMAX>
__device__ __forceinline__ void dec_tile8(const AttnParams &p, const DecRow (&rr)[2],
                                          const uint32_t (&qb)[D / 16][2], uint32_t kb,
                                          uint32_t vb, int j0, float (&o)[D / 16][4],
                                          float (&m_r)[2], float (&l_r)[2], float sc) {
    constexpr int KS = D / 16, CH = D / 64, VW = D / 8;
    constexpr bool PV_BF16 = BF16 && !SOFTMAX;   // type of P and V in the P V product
    const int lane = threadIdx.x & 31, c = lane & 3, r = lane >> 2;
    // V codes of keys 0..15 (rows 2c, 2c+1, 2c+8, 2c+9), loaded before the
    // S^T product so that their latency hides behind it
    uint32_t pv0[VW / 4], pv1[VW / 4], pv8[VW / 4], pv9[VW / 4];
    if constexpr (D == 128) {
        uint32_t w[4];
        lds128(vb + off8<D>(2 * c, r), w);
#pragma unroll
        for (int i = 0; i < 4; ++i) pv0[i] = w[i];
        lds128(vb + off8<D>(2 * c + 1, r), w);
#pragma unroll
        for (int i = 0; i < 4; ++i) pv1[i] = w[i];
        lds128(vb + off8<D>(2 * c + 8, r), w);
#pragma unroll
        for (int i = 0; i < 4; ++i) pv8[i] = w[i];
        lds128(vb + off8<D>(2 * c + 9, r), w);
#pragma unroll
        for (int i = 0; i < 4; ++i) pv9[i] = w[i];
    } else {
        const int ch = r >> 1, half = (r & 1) * 8;
        lds64(vb + off8<D>(2 * c, ch) + half, pv0[0], pv0[1]);
        lds64(vb + off8<D>(2 * c + 1, ch) + half, pv1[0], pv1[1]);
        lds64(vb + off8<D>(2 * c + 8, ch) + half, pv8[0], pv8[1]);
        lds64(vb + off8<D>(2 * c + 9, ch) + half, pv9[0], pv9[1]);
    }
    float sacc[2][4];
#pragma unroll
    for (int mb = 0; mb < 2; ++mb) {
        sacc[mb][0] = sacc[mb][1] = sacc[mb][2] = sacc[mb][3] = 0.f;
        uint32_t k0[KS], k8[KS];   // key rows 16 mb + r and 16 mb + r + 8
#pragma unroll
        for (int h = 0; h < CH; ++h) {
            uint32_t w[4];
            lds128(kb + off8<D>(16 * mb + r, c * CH + h), w);
#pragma unroll
            for (int i = 0; i < 4; ++i) k0[4 * h + i] = w[i];
            lds128(kb + off8<D>(16 * mb + r + 8, c * CH + h), w);
#pragma unroll
            for (int i = 0; i < 4; ++i) k8[4 * h + i] = w[i];
        }
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint32_t a[4];
            e4m3x4_to_x2<false>(k0[ks], a[0], a[2]);
            e4m3x4_to_x2<false>(k8[ks], a[1], a[3]);
            mma16816<false>(sacc[mb], a, qb[ks][0], qb[ks][1]);
        }
    }
    dec_normalize_t<D, SOFTMAX>(p, rr, sacc, j0, o, m_r, l_r, sc);
    // O^T += V^T P^T over the tile's two 16-key halves
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
        const uint32_t b0 = movmatrix_trans(pack2<PV_BF16>(sacc[kk][0], sacc[kk][1]));
        const uint32_t b1 = movmatrix_trans(pack2<PV_BF16>(sacc[kk][2], sacc[kk][3]));
        // key rows k0, k0 + 1 (a0, a1) and k0 + 8, k0 + 9 (a2, a3); codes [VW r, VW r + VW)
        const int k0 = kk * 16 + 2 * c;
        uint32_t v0[VW / 4], v1[VW / 4], v8[VW / 4], v9[VW / 4];
        if (kk == 0) {
#pragma unroll
            for (int i = 0; i < VW / 4; ++i) {
                v0[i] = pv0[i]; v1[i] = pv1[i]; v8[i] = pv8[i]; v9[i] = pv9[i];
            }
        } else if constexpr (D == 128) {
            uint32_t w[4];
            lds128(vb + off8<D>(k0, r), w);
#pragma unroll
            for (int i = 0; i < 4; ++i) v0[i] = w[i];
            lds128(vb + off8<D>(k0 + 1, r), w);
#pragma unroll
            for (int i = 0; i < 4; ++i) v1[i] = w[i];
            lds128(vb + off8<D>(k0 + 8, r), w);
#pragma unroll
            for (int i = 0; i < 4; ++i) v8[i] = w[i];
            lds128(vb + off8<D>(k0 + 9, r), w);
#pragma unroll
            for (int i = 0; i < 4; ++i) v9[i] = w[i];
        } else {
            const int ch = r >> 1, half = (r & 1) * 8;
            lds64(vb + off8<D>(k0, ch) + half, v0[0], v0[1]);
            lds64(vb + off8<D>(k0 + 1, ch) + half, v1[0], v1[1]);
            lds64(vb + off8<D>(k0 + 8, ch) + half, v8[0], v8[1]);
            lds64(vb + off8<D>(k0 + 9, ch) + half, v9[0], v9[1]);
        }
#pragma unroll
        for (int w = 0; w < VW / 4; ++w) {
            uint32_t x[4], y[4];   // dims VW r + 4w .. + 3: keys (k0, k0 + 1) in x, (k0 + 8, k0 + 9) in y
            e4m3x4_to_x2<PV_BF16>(__byte_perm(v0[w], v1[w], 0x5140), x[0], x[1]);
            e4m3x4_to_x2<PV_BF16>(__byte_perm(v0[w], v1[w], 0x7362), x[2], x[3]);
            e4m3x4_to_x2<PV_BF16>(__byte_perm(v8[w], v9[w], 0x5140), y[0], y[1]);
            e4m3x4_to_x2<PV_BF16>(__byte_perm(v8[w], v9[w], 0x7362), y[2], y[3]);
            const uint32_t a0[4] = {x[0], x[1], y[0], y[1]};   // dim block 2w
            const uint32_t a1[4] = {x[2], x[3], y[2], y[3]};   // dim block 2w + 1
            mma16816<PV_BF16>(o[2 * w], a0, b0, b1);
            mma16816<PV_BF16>(o[2 * w + 1], a1, b0, b1);
        }
    }
}

// The 16-bit tile with the transposed products of dec_tile8 (S^T = K Q^T,
// O^T = V^T P^T; each N-block of 8 query rows is the MMA's N): K blocks are
// the A operand straight from ldmatrix, V^T blocks from ldmatrix.trans, P^T
// from movmatrix; Q (qb[nb]) is the B operand in the natural dim order.
// The NB N-blocks (8 NB rows of the pair) share every A fragment.
// Accumulator o[nb][m][e] holds row 8 nb + 2c + e % 2, dim 16 m + lane/4 +
// 8 (e / 2).
template <int D, bool BF16, bool SOFTMAX, int NB>
__device__ __forceinline__ void dec_tile16t(const AttnParams &p, const DecRow (&rr)[NB][2],
                                            const uint32_t (&qb)[NB][D / 16][2], uint32_t kb,
                                            uint32_t vb, int j0, float (&o)[NB][D / 16][4],
                                            float (&m_r)[NB][2], float (&l_r)[NB][2], float sc) {
    using L = DecLayout<D, false>;
    constexpr int KS = D / 16, NO = D / 16;
    const int lane = threadIdx.x & 31;
    float sacc[NB][2][4];
#pragma unroll
    for (int mb = 0; mb < 2; ++mb) {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
            sacc[nb][mb][0] = sacc[nb][mb][1] = sacc[nb][mb][2] = sacc[nb][mb][3] = 0.f;
        const int key = 16 * mb + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint32_t a[4];
            ldsm_x4(kb + swz(key, ks * 2 + (lane >> 4), L::BLK), a[0], a[1], a[2], a[3]);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) mma16816<BF16>(sacc[nb][mb], a, qb[nb][ks][0], qb[nb][ks][1]);
        }
    }
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
        dec_normalize_t<D, SOFTMAX>(p, rr[nb], sacc[nb], j0, o[nb], m_r[nb], l_r[nb], sc);
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
        uint32_t b0[NB], b1[NB];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            b0[nb] = movmatrix_trans(pack2<BF16>(sacc[nb][kk][0], sacc[nb][kk][1]));
            b1[nb] = movmatrix_trans(pack2<BF16>(sacc[nb][kk][2], sacc[nb][kk][3]));
        }
        const int key = 16 * kk + (lane & 7) + ((lane >> 4) & 1) * 8;
#pragma unroll
        for (int m = 0; m < NO; ++m) {
            uint32_t a[4];
            ldsm_x4_t(vb + swz(key, m * 2 + ((lane >> 3) & 1), L::BLK), a[0], a[1], a[2], a[3]);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) mma16816<BF16>(o[nb][m], a, b0[nb], b1[nb]);
        }
    }
}

// Accumulator layouts of the two tiles (DLAY), both with rows 2c and 2c+1
// (c = lane % 4): DLAY_FP8, dims [(D/8) (lane/4), +D/8) in order; DLAY_16T,
// dim 16 m + lane/4 + 8 (e / 2) of o[m][e].
constexpr int DLAY_FP8 = 1, DLAY_16T = 2;

// Y rows of this lane's output rows, scaled by f (rows outside are skipped).
template <int D, bool BF16, int DLAY>
__device__ __forceinline__ void dec_store_y(const AttnParams &p, const DecRow (&rr)[2],
                                            const float (&o)[D / 16][4], const float (&f)[2]) {
    const int lane = threadIdx.x & 31;
    uint16_t *y = static_cast<uint16_t *>(p.y);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        if (!rr[r].valid) continue;
        if (!dbg_ok(rr[r].qoff >= 0 && rr[r].qoff + D <= q_elems(p), p.status)) continue;
        if constexpr (DLAY == DLAY_FP8) {
            constexpr int NO = D / 16;
            uint4 *dst = reinterpret_cast<uint4 *>(y + rr[r].qoff + (D / 8) * (lane >> 2));
#pragma unroll
            for (int i = 0; i < NO / 4; ++i)
                dst[i] = make_uint4(pack2<BF16>(o[4 * i][r] * f[r], o[4 * i][r + 2] * f[r]),
                                    pack2<BF16>(o[4 * i + 1][r] * f[r], o[4 * i + 1][r + 2] * f[r]),
                                    pack2<BF16>(o[4 * i + 2][r] * f[r], o[4 * i + 2][r + 2] * f[r]),
                                    pack2<BF16>(o[4 * i + 3][r] * f[r], o[4 * i + 3][r + 2] * f[r]));
        } else {
            // dims 16 m + lane/4 and + 8: one 16-bit store each (once per pair)
#pragma unroll
            for (int m = 0; m < D / 16; ++m) {
                const uint32_t w = pack2<BF16>(o[m][r] * f[r], o[m][r + 2] * f[r]);
                y[rr[r].qoff + 16 * m + (lane >> 2)] = (uint16_t)(w & 0xffffu);
                y[rr[r].qoff + 16 * m + (lane >> 2) + 8] = (uint16_t)(w >> 16);
            }
        }
    }
}

// This lane's partial O rows (unnormalised) into one partial slot.
template <int D, int DLAY>
__device__ __forceinline__ void dec_store_part(float *slot_rows, const float (&o)[D / 16][4]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        if constexpr (DLAY == DLAY_FP8) {
            float *po = slot_rows + (2 * (lane & 3) + r) * D + (D / 8) * (lane >> 2);
#pragma unroll
            for (int i = 0; i < D / 32; ++i)
                *reinterpret_cast<float4 *>(po + 4 * i) =
                    make_float4(o[2 * i][r], o[2 * i][r + 2], o[2 * i + 1][r], o[2 * i + 1][r + 2]);
        } else {
            float *po = slot_rows + (2 * (lane & 3) + r) * D + (lane >> 2);
#pragma unroll
            for (int m = 0; m < D / 16; ++m) {
                po[16 * m] = o[m][r];
                po[16 * m + 8] = o[m][r + 2];
            }
        }
    }
}

// One lane's view of the pair being computed or loaded: a pair is
// (batch b, KV head g, row chunk rc of DR query rows); its key tiles
// are the 32-key tiles of [0, key extent of the batch).
struct DecCur {
    int b, pib;          // batch, pair within the batch (g * nrc + rc)
    int tile;            // tile within the pair
    int nt, nrc;         // tiles per pair, row chunks of the batch
    SeqInfo s;
};

// Batch b's row chunks of DR rows and key tiles per pair (0 chunks: no
// query rows).
template <int DR>
__device__ __forceinline__ void dec_batch_shape(const AttnParams &p, const SeqInfo &s, int &nrc,
                                                int &nt) {
    const int rows = s.q_len * p.G;
    nrc = (rows + DR - 1) / DR;
    const int kv_hi = rows > 0 ? key_extent(p.causal, s.q_len - 1, s) : 0;
    nt = (kv_hi + DEC_KEYS - 1) / DEC_KEYS;
}

// Block-wide exclusive prefix of v[0..n) in place (n <= DEC_MAX_B), with
// v[n] set to the total; every thread of the block (THREADS) calls it.
template <int THREADS>
__device__ __forceinline__ void dec_prefix(int *v, int n, int *scratch) {
    const int per = (n + THREADS - 1) / THREADS;
    const int lo = threadIdx.x * per, hi = min(n, lo + per);
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += v[i];
    scratch[threadIdx.x] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int t = 0; t < THREADS; ++t) {
            const int x = scratch[t];
            scratch[t] = run;
            run += x;
        }
        scratch[THREADS] = run;
    }
    __syncthreads();
    int run = scratch[threadIdx.x];
    for (int i = lo; i < hi; ++i) {
        const int x = v[i];
        v[i] = run;
        run += x;
    }
    if (threadIdx.x == 0) v[n] = scratch[THREADS];
    __syncthreads();
}

// PAGED: K and V come from page pools (a compile-time choice, so that the
// page lookups cost the linear-cache kernels nothing).  NB: N-blocks of 8
// query rows per pair (16-bit cache: 1 or 2; fp8 cache: 1); the launcher
// takes it from p.dec_rows, which also sized the partial slots.
template <int D, bool BF16, bool SOFTMAX, bool KV8, bool PAGED, int NB>
__global__ void __launch_bounds__(DecLayout<D, KV8>::THREADS, 1)
decode_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ TensorMaps tm) {
    static_assert(NB == 1 || (NB == 2 && !KV8), "N-blocks per pair");
    using L = DecLayout<D, KV8>;
    constexpr int NW = L::NW;
    constexpr int DR = 8 * NB;                     // query rows per pair
    constexpr int NS = L::STAGES;
    constexpr int DLAY = KV8 ? DLAY_FP8 : DLAY_16T;
    constexpr int NO = D / 16;                     // O^T accumulator blocks
    constexpr int QW = 2;                          // Q fragment words per k-step
    constexpr int KS = D / 16;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::BAR_OFF);
    volatile int *abort = reinterpret_cast<volatile int *>(sm + L::BAR_OFF + NW * NS * 8);
    int *flags = reinterpret_cast<int *>(sm + L::BAR_OFF + NW * NS * 8 + 4);
    int *scratch = reinterpret_cast<int *>(sm + L::SCR_OFF);
    int *tpre = reinterpret_cast<int *>(sm + L::TPRE_OFF);   // key tiles before batch b
    int *ppre = reinterpret_cast<int *>(sm + L::PPRE_OFF);   // pairs before batch b
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NW * NS; ++i) mbar_init(&bars[i], 1);
        *abort = 0;
        flags[0] = 0;   // bad lengths
        fence_mbar_init();
    }
    __syncthreads();
    // Every CTA validates the lengths and lays out the work itself.
    for (int b = threadIdx.x; b < p.B; b += L::THREADS) {
        const int32_t *ql = p.query_lengths, *kl = p.kv_lengths;
        const SeqInfo s = seq_info(p, b);
        bool ok = s.q_len >= 0 && s.kv_len >= 0;
        if (ql) ok = ok && ql[0] == 0;
        if (p.q_packed) ok = ok && ql[b + 1] <= p.q_seq;
        else ok = ok && s.q_len <= p.q_seq;
        if (p.kv_packed) ok = ok && kl[0] == 0 && kl[b + 1] <= p.kv_seq;
        else ok = ok && s.kv_len <= p.kv_seq;
        if (p.mask) {
            if (p.md[2] != 1 && p.md[2] < s.q_len) ok = false;
            if (p.md[3] != 1 && p.md[3] < s.kv_len) ok = false;
        }
        if (!ok) atomicOr(&flags[0], 1);
        int nrc = 0, nt = 0;
        if (ok) dec_batch_shape<DR>(p, s, nrc, nt);
        tpre[b] = p.Hkv * nrc * nt;
        ppre[b] = p.Hkv * nrc;
    }
    __syncthreads();
    if (flags[0]) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_status(p.status, 4);
        return;
    }
    dec_prefix<L::THREADS>(tpre, p.B, scratch);
    dec_prefix<L::THREADS>(ppre, p.B, scratch);
    pdl_wait();   // the tickets have been cleared (and, paged, the pages checked)
    if constexpr (PAGED) {
        const volatile int *pf = reinterpret_cast<const volatile int *>(p.ws) + WS_PAGE_FLAGS;
        const int bad = (int)threadIdx.x < dec_prep_blocks(p) ? pf[threadIdx.x] : 0;
        if (__syncthreads_or(bad)) {
            if (blockIdx.x == 0 && threadIdx.x == 0) set_status(p.status, 4);
            return;
        }
    }

    // Stream-K split of the work: all key tiles of all pairs, batch-major,
    // in one line of T tiles, cut into equal contiguous ranges, one per warp
    // of the grid.  A pair inside one range is finished by its warp; a pair
    // cut by range ends is finished by the last of its warps to arrive
    // (atomic ticket), which merges the others' partials in warp order.
    const int T = tpre[p.B];
    const int wg = blockIdx.x * NW + warp;
    // at most one warp per tile, so that every range holds at least one
    // (the merge counts a pair's warps from the range ends); later warps idle
    const int Wn = max(1, min((int)gridDim.x * NW, T));
    auto range_start = [&](int w) { return (int)((long long)w * T / Wn); };
    auto warp_of = [&](int x) { return (int)(((long long)(x + 1) * Wn - 1) / T); };
    int *tickets = reinterpret_cast<int *>(p.ws + dec_tickets_off(p));
    float *part = reinterpret_cast<float *>(p.ws + dec_part_off(p));
    float2 *pml = reinterpret_cast<float2 *>(p.ws + dec_ml_off(p));

    // batches with query rows but no key tile: their rows are zero
    for (int b = wg; b < p.B; b += gridDim.x * NW) {
        const SeqInfo s = seq_info(p, b);
        int nrc, nt;
        dec_batch_shape<DR>(p, s, nrc, nt);
        if (nrc == 0 || nt > 0) continue;
        const int rows = s.q_len * p.G;
        for (int r = lane; r < p.Hkv * rows; r += 32) {
            const DecRow R = dec_row(p, s, b, r / rows, r % rows, rows, 0);
            if (!dbg_ok(R.qoff >= 0 && R.qoff + D <= q_elems(p), p.status)) continue;
            uint4 *y = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.y) + R.qoff);
            for (int c = 0; c < D / 8; ++c) y[c] = make_uint4(0, 0, 0, 0);
        }
    }

    uint8_t *ring = sm + warp * L::WARP_RING;
    uint64_t *wbar = bars + warp * NS;
    const uint32_t ring_u32 = smem_u32(ring);
    uint32_t issued = 0, consumed = 0;
    const int t_begin = wg < Wn ? range_start(wg) : T, t_end = wg < Wn ? range_start(wg + 1) : T;

    auto locate = [&](int t, DecCur &c) {
        int lo = 0, hi = p.B;   // tpre[lo] <= t < tpre[lo + 1]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (tpre[mid] <= t) lo = mid; else hi = mid;
        }
        c.b = lo;
        c.s = seq_info(p, lo);
        dec_batch_shape<DR>(p, c.s, c.nrc, c.nt);
        const int r = t - tpre[lo];
        c.pib = r / c.nt;
        c.tile = r % c.nt;
    };
    auto advance = [&](DecCur &c) {   // the next tile of the line
        if (++c.tile < c.nt) return;
        c.tile = 0;
        if (++c.pib < p.Hkv * c.nrc) return;
        int b = c.b + 1;
        while (b < p.B && tpre[b + 1] == tpre[b]) ++b;   // batches without tiles
        if (b >= p.B) return;                              // past the end: never used
        c.b = b;
        c.pib = 0;
        c.s = seq_info(p, b);
        dec_batch_shape<DR>(p, c.s, c.nrc, c.nt);
    };
    // K and V pages of cursor c's tile (paged cache; lane 0 only)
    auto pages_of = [&](const DecCur &c, int &pk, int &pv) {
        pk = pv = 0;
        if (PAGED && lane == 0) {
            const int32_t *pt = p.page_table + (size_t)c.b * 2 * p.max_pages;
            const int pg = c.tile * DEC_KEYS / p.page_size;
            pk = __ldg(pt + pg);
            pv = __ldg(pt + p.max_pages + pg);
        }
    };
    auto issue = [&](const DecCur &c, int pk, int pv) {
        if (lane == 0) {
            fence_proxy_async_smem();   // the stage's previous tile was read by ldmatrix
            dec_tma<KV8, PAGED>(p, tm, c.s, c.b, c.pib / c.nrc, c.tile * DEC_KEYS,
                    ring + (issued % NS) * L::STAGE, &wbar[issued % NS], D, pk, pv);
        }
        ++issued;
    };

    // score scale (the K dequantisation scale folded in) and output factor
    // (the V dequantisation scale)
    const float sc = (SOFTMAX ? p.scale_log2 : p.scale) * (KV8 ? __ldg(p.k_scale) : 1.f);
    float sc_pair = sc;   // sc times the power of two taken out of Q (fp8 KV, bf16 Q)
    const float sv = KV8 ? __ldg(p.v_scale) : 1.f;
    bool ok = true;
    if (t_begin < t_end) {
        DecCur lc, cc;
        locate(t_begin, lc);
        cc = lc;
        int next_issue = t_begin;
        for (; next_issue < t_end && next_issue < t_begin + NS; ++next_issue) {
            int pk, pv;
            pages_of(lc, pk, pv);
            issue(lc, pk, pv);
            advance(lc);
        }
        DecRow rr[NB][2];   // this lane's two output rows of each N-block
        uint32_t qa[NB][KS][QW];
        float o[NB][NO][4];
        float m_r[NB][2], l_r[NB][2];
        int seg0 = t_begin;    // first tile of the current pair in this range
        int kv_hi = 0, rows = 0;
        auto start_pair = [&]() {
            const int g = cc.pib / cc.nrc, rc = cc.pib % cc.nrc;
            rows = cc.s.q_len * p.G;
            kv_hi = key_extent(p.causal, cc.s.q_len - 1, cc.s);
            const uint32_t *q32 = static_cast<const uint32_t *>(p.q);
            if constexpr (!KV8) {
                // N-block nb: output rows 8 nb + 2c, 8 nb + 2c + 1; Q row
                // 8 nb + lane / 4 is the B operand of S^T in the natural dim order
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
                    const int r0 = rc * DR + 8 * nb;
                    rr[nb][0] = dec_row(p, cc.s, cc.b, g, r0 + 2 * (lane & 3), rows, kv_hi);
                    rr[nb][1] = dec_row(p, cc.s, cc.b, g, r0 + 2 * (lane & 3) + 1, rows, kv_hi);
                    DecRow rq = dec_row(p, cc.s, cc.b, g, r0 + (lane >> 2), rows, kv_hi);
                    rq.valid = rq.valid &&
                               dbg_ok(rq.qoff >= 0 && rq.qoff + D <= q_elems(p), p.status);
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        qa[nb][ks][0] = rq.valid ? q32[(rq.qoff >> 1) + 8 * ks + (lane & 3)] : 0u;
                        qa[nb][ks][1] = rq.valid ? q32[(rq.qoff >> 1) + 8 * ks + 4 + (lane & 3)] : 0u;
                    }
                }
            } else if constexpr (KV8) {
                // output rows 2c, 2c + 1; Q row lane / 4 (the B operand of
                // S^T), dims [c D/4, (c+1) D/4), four per k-step (the
                // contraction order of dec_tile8)
                rr[0][0] = dec_row(p, cc.s, cc.b, g, rc * DR + 2 * (lane & 3), rows, kv_hi);
                rr[0][1] = dec_row(p, cc.s, cc.b, g, rc * DR + 2 * (lane & 3) + 1, rows, kv_hi);
                DecRow rq = dec_row(p, cc.s, cc.b, g, rc * DR + (lane >> 2), rows, kv_hi);
                rq.valid = rq.valid && dbg_ok(rq.qoff >= 0 && rq.qoff + D <= q_elems(p), p.status);
                uint32_t w[D / 8];
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    static_cast<const uint16_t *>(p.q) + rq.qoff + (lane & 3) * (D / 4));
#pragma unroll
                for (int k = 0; k < D / 32; ++k) {
                    const uint4 x = rq.valid ? src[k] : make_uint4(0, 0, 0, 0);
                    w[4 * k] = x.x; w[4 * k + 1] = x.y; w[4 * k + 2] = x.z; w[4 * k + 3] = x.w;
                }
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    qa[0][ks][0] = w[2 * ks];
                    qa[0][ks][1] = w[2 * ks + 1];
                }
                if constexpr (BF16) {
                    // bf16 -> f16 for the f16 S product: scale the warp's
                    // 8 rows by 2^-e so that their largest magnitude lies
                    // in [2^14, 2^15).  Every bf16 value (8 significant
                    // bits) at or above 2^-14 after scaling is then an exact
                    // f16; smaller ones (below 2^-28 of the largest) round
                    // to the f16 spacing 2^-24, a change far below the
                    // fp32 rounding of the dot product.  2^e goes back into
                    // the score scale.
                    float mx = 0.f;
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                        for (int i = 0; i < QW; ++i)
                            mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(qa[0][ks][i] << 16)),
                                                 fabsf(__uint_as_float(qa[0][ks][i] & 0xffff0000u))));
#pragma unroll
                    for (int m = 1; m < 32; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
                    int e = mx > 0.f ? (int)((__float_as_uint(mx) >> 23) & 0xff) - 127 - 14 : 0;
                    e = min(max(e, -100), 100);
                    const float down = __uint_as_float((uint32_t)(127 - e) << 23);
                    sc_pair = sc * __uint_as_float((uint32_t)(127 + e) << 23);
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                        for (int i = 0; i < QW; ++i)
                            qa[0][ks][i] = pack2<false>(__uint_as_float(qa[0][ks][i] << 16) * down,
                                                        __uint_as_float(qa[0][ks][i] & 0xffff0000u) * down);
                }
            }
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
                for (int n = 0; n < NO; ++n) o[nb][n][0] = o[nb][n][1] = o[nb][n][2] = o[nb][n][3] = 0.f;
                m_r[nb][0] = m_r[nb][1] = -INFINITY;
                l_r[nb][0] = l_r[nb][1] = 0.f;
            }
        };
        start_pair();

        for (int t = t_begin; t < t_end; ++t) {
            const uint32_t c = consumed;
            const int st = c % NS;
            if (!mbar_wait(&wbar[st], (c / NS) & 1, abort)) { ok = false; break; }
            ++consumed;
            // pages of the tile the refill below loads, read while this one computes
            int npk = 0, npv = 0;
            if (PAGED && next_issue < t_end) pages_of(lc, npk, npv);
            const int j0 = cc.tile * DEC_KEYS;
            const uint32_t kb = ring_u32 + st * L::STAGE, vb = kb + L::TILE;
            const int rem = cc.s.kv_len - j0;
            if (rem < DEC_KEYS) {   // rows past the sequence end may hold NaN: zero them
                uint8_t *vp = ring + st * L::STAGE + L::TILE;
                constexpr int CPR = KV8 ? D / 16 : D / 8;   // 16-byte chunks per row
                for (int idx = lane; idx < DEC_KEYS * CPR; idx += 32) {
                    const int row = idx / CPR, ch = idx % CPR;
                    if (row >= rem)
                        *reinterpret_cast<uint4 *>(vp + (KV8 ? off8<D>(row, ch) : swz(row, ch, L::BLK))) =
                            make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }
            if constexpr (KV8)
                dec_tile8<D, BF16, SOFTMAX>(p, rr[0], qa[0], kb, vb, j0, o[0], m_r[0], l_r[0], sc_pair);
            else dec_tile16t<D, BF16, SOFTMAX, NB>(p, rr, qa, kb, vb, j0, o, m_r, l_r, sc);
            __syncwarp();
            if (next_issue < t_end) {   // refill the stage just used
                issue(lc, npk, npv);
                advance(lc);
                ++next_issue;
            }
            const bool pair_end = cc.tile + 1 == cc.nt;
            if (pair_end || t + 1 == t_end) {
                // this range's share of the pair is done (the lanes
                // sharing a row differ in lane / 4)
                if (SOFTMAX)
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                        for (int r = 0; r < 2; ++r)
#pragma unroll
                            for (int m = 4; m < 32; m <<= 1)
                                l_r[nb][r] += __shfl_xor_sync(0xffffffffu, l_r[nb][r], m);
                const int b = cc.b, g = cc.pib / cc.nrc, rc = cc.pib % cc.nrc;
                const int ps = tpre[b] + cc.pib * cc.nt, pe = ps + cc.nt;
                if (seg0 == ps && t + 1 == pe) {   // the whole pair: write Y
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) {
                        float f[2];
#pragma unroll
                        for (int r = 0; r < 2; ++r)
                            f[r] = (SOFTMAX ? (l_r[nb][r] > 0.f ? 1.f / l_r[nb][r] : 0.f) : 1.f) * sv;
                        dec_store_y<D, BF16, DLAY>(p, rr[nb], o[nb], f);
                    }
                } else {
                    // partial (O, m, l): slot 0 for the first pair of the
                    // range, slot 1 for the last; N-block nb holds rows 8 nb ..
                    const size_t slot = (size_t)wg * 2 + (seg0 == t_begin ? 0 : 1);
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) {
                        if (!dbg_ok(slot < (size_t)p.dec_slots && DR == p.dec_rows, p.status)) break;
                        dec_store_part<D, DLAY>(part + (slot * DR + 8 * nb) * D, o[nb]);
                        if (lane < 4)
#pragma unroll
                            for (int r = 0; r < 2; ++r)
                                pml[slot * DR + 8 * nb + 2 * lane + r] = make_float2(m_r[nb][r], l_r[nb][r]);
                    }
                    __threadfence();
                    __syncwarp();
                    const int w_lo = warp_of(ps), w_hi = warp_of(pe - 1);
                    const int pidx = ppre[b] + cc.pib;
                    int tk = 0;
                    if (lane == 0 && dbg_ok(pidx >= 0 && pidx <= p.max_pairs, p.status))
                        tk = atomicAdd(&tickets[pidx], 1);
                    tk = __shfl_sync(0xffffffffu, tk, 0);
                    if (tk == w_hi - w_lo) {   // the last of the pair's warps: merge
                        __threadfence();
                        // LPR lanes per row, each with D / LPR dims, merged
                        // MC dims at a time
                        constexpr int LPR = 32 / DR, DL = D / LPR, MC = DL < 32 ? DL : 32;
                        const int row = lane / LPR, c0 = (lane % LPR) * DL;
                        // the first warp's share is its slot 1 unless the pair
                        // starts its range; every later warp's share is its slot 0
                        auto slot_of = [&](int w) -> size_t {
                            return (size_t)w * 2 + ((w == w_lo && range_start(w) != ps) ? 1 : 0);
                        };
                        float M = -INFINITY;
                        if (SOFTMAX)
                            for (int w = w_lo; w <= w_hi; ++w)
                                M = fmaxf(M, __ldcg(&pml[slot_of(w) * DR + row].x));
                        const DecRow R = dec_row(p, cc.s, b, g, rc * DR + row, rows, kv_hi);
#pragma unroll 1
                        for (int h = 0; h < DL / MC; ++h) {
                            float acc[MC];
#pragma unroll
                            for (int k = 0; k < MC; ++k) acc[k] = 0.f;
                            float Lsum = 0.f;
                            for (int w = w_lo; w <= w_hi; ++w) {
                                const size_t sl = slot_of(w);
                                float wt = 1.f;
                                if (SOFTMAX) {
                                    const float2 v = __ldcg(&pml[sl * DR + row]);
                                    wt = (v.x == -INFINITY) ? 0.f : ex2(v.x - M);
                                    Lsum += v.y * wt;
                                }
                                const float4 *src = reinterpret_cast<const float4 *>(
                                    part + (sl * DR + row) * D + c0 + h * MC);
#pragma unroll
                                for (int k = 0; k < MC / 4; ++k) {
                                    const float4 x4 = __ldcg(src + k);
                                    acc[4 * k] += x4.x * wt;
                                    acc[4 * k + 1] += x4.y * wt;
                                    acc[4 * k + 2] += x4.z * wt;
                                    acc[4 * k + 3] += x4.w * wt;
                                }
                            }
                            if (R.valid && dbg_ok(R.qoff >= 0 && R.qoff + D <= q_elems(p), p.status)) {
                                const float f = (SOFTMAX ? (Lsum > 0.f ? 1.f / Lsum : 0.f) : 1.f) * sv;
                                uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.y) +
                                                                       R.qoff + c0 + h * MC);
#pragma unroll
                                for (int k = 0; k < MC / 8; ++k)
                                    dst[k] = make_uint4(pack2<BF16>(acc[8 * k] * f, acc[8 * k + 1] * f),
                                                        pack2<BF16>(acc[8 * k + 2] * f, acc[8 * k + 3] * f),
                                                        pack2<BF16>(acc[8 * k + 4] * f, acc[8 * k + 5] * f),
                                                        pack2<BF16>(acc[8 * k + 6] * f, acc[8 * k + 7] * f));
                            }
                        }
                        if (lane == 0) tickets[pidx] = 0;   // ready for the next call
                    }
                }
            }
            advance(cc);
            if (pair_end && t + 1 < t_end) {
                start_pair();
                seg0 = t + 1;
            }
        }
    }
    // copies still in flight (only after an abort) land before the CTA exits
    while (consumed < issued) {
        mbar_wait_drain(&wbar[consumed % NS], (consumed / NS) & 1);
        ++consumed;
    }
    __syncwarp();
    if (lane == 0 && (!ok || *abort)) set_status(p.status, 5);
}

// Clears the merge tickets of a decode call.  With a paged cache every
// block also checks its slice of the page indices of every sequence's keys
// (all of [0, kv_len)) and writes to its own header word whether one lies
// outside the pools.  The decode kernel follows it as a programmatic
// dependent and reads those words after griddepcontrol.wait, before
// writing anything.
static __global__ void decode_prep_kernel(const __grid_constant__ AttnParams p, int n) {
    pdl_launch_dependents();
    int *tickets = reinterpret_cast<int *>(p.ws + dec_tickets_off(p));
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        tickets[i] = 0;
    if (p.paged) {
        const long long total = (long long)p.B * p.max_pages;
        const long long cap = (long long)p.max_pages * p.page_size;
        int bad = 0;
        for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
             i += (long long)gridDim.x * blockDim.x) {
            const int b = (int)(i / p.max_pages), k = (int)(i % p.max_pages);
            const long long len = min((long long)max(p.kv_lengths[b], 0), cap);
            if (k >= (len + p.page_size - 1) / p.page_size) continue;
            const int32_t *pt = p.page_table + (size_t)b * 2 * p.max_pages;
            const int a = pt[k], v = pt[p.max_pages + k];
            if (a < 0 || a >= p.num_pages || v < 0 || v >= p.num_pages) bad = 1;
        }
        bad = __syncthreads_or(bad);
        if (threadIdx.x == 0) reinterpret_cast<int *>(p.ws)[WS_PAGE_FLAGS + blockIdx.x] = bad;
    }
}

template <int D, bool BF16, bool SOFTMAX, bool KV8, bool PAGED, int NB>
static cudaError_t dec_launch(const AttnParams &p, const TensorMaps &m, cudaStream_t s) {
    using L = DecLayout<D, KV8>;
    static std::atomic<unsigned long long> configured{0};
    cudaError_t e = once_per_device(configured, [] {
        return cudaFuncSetAttribute(decode_kernel<D, BF16, SOFTMAX, KV8, PAGED, NB>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    });
    if (e != cudaSuccess) return e;
    const int n = p.max_pairs + 1;
    decode_prep_kernel<<<dec_prep_blocks(p), 256, 0, s>>>(p, n);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_dependent(decode_kernel<D, BF16, SOFTMAX, KV8, PAGED, NB>, p.grid, L::THREADS,
                            L::ALLOC, s, p, m);
}

template <bool KV8, bool PAGED, int NB>
static cudaError_t dec_launch_kp(const AttnParams &p, const TensorMaps &m, bool sm,
                                 cudaStream_t s, int bf16) {
    if (p.D == 64) {
        if (bf16) return sm ? dec_launch<64, true, true, KV8, PAGED, NB>(p, m, s)
                            : dec_launch<64, true, false, KV8, PAGED, NB>(p, m, s);
        return sm ? dec_launch<64, false, true, KV8, PAGED, NB>(p, m, s)
                  : dec_launch<64, false, false, KV8, PAGED, NB>(p, m, s);
    }
    if (bf16) return sm ? dec_launch<128, true, true, KV8, PAGED, NB>(p, m, s)
                        : dec_launch<128, true, false, KV8, PAGED, NB>(p, m, s);
    return sm ? dec_launch<128, false, true, KV8, PAGED, NB>(p, m, s)
              : dec_launch<128, false, false, KV8, PAGED, NB>(p, m, s);
}

// The decode kernels of one KV element type (KV8: E4M3 codes) and one
// number of N-blocks per pair, linear or paged; each instantiates in its own
// translation unit.  p.dec_rows (which sized the partial slots) must be 8 NB.
template <bool KV8, int NB>
cudaError_t launch_decode_kv(const AttnParams &p, const TensorMaps &m, int mode,
                             cudaStream_t s, int bf16) {
    if (p.dec_rows != 8 * NB) return cudaErrorInvalidValue;
    const bool sm = (mode == MODE_SOFTMAX);
    return p.paged ? dec_launch_kp<KV8, true, NB>(p, m, sm, s, bf16)
                   : dec_launch_kp<KV8, false, NB>(p, m, sm, s, bf16);
}

}  // namespace rga
