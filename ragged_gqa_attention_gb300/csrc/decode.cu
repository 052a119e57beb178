// decode.cu - split-KV attention for short query lengths (decode), the
// HBM-bound path of the AttentionPlugin ("TensorRT Plugins Guide":
// vanilla decoding attention) with the TRT_Attention semantics of
// "TensorRT Custom Operator Schemas".
//
// Work unit: (batch b, KV head g, split of DEC_SPLIT keys).  The grid is
// persistent; each CTA validates the lengths and lists the units itself
// (no scheduler launch), and every warp is an independent engine: it takes
// the next unit from an atomic counter, streams the unit's
// 32-key K/V tiles with TMA through its own DEC_STAGES-deep, 128-byte-
// swizzled ring, computes S = Q K^T and O += P V with m16n8k16 MMAs (K and
// V are read once from HBM for all G query heads of the KV head) and keeps
// an online softmax in fp32 registers.  The query rows of a unit are the
// (token, head) pairs of the G heads, 16 at a time (one MMA row block).
// A unit that covers its whole (b, g) pair writes Y; otherwise its partial
// (O, m, l) goes to the workspace and the last warp to finish a pair
// (atomic ticket) merges the splits and writes Y.
//
// A pair with more than 16 query rows (more than 16/G tokens) is one unit
// that loops over the row blocks.
#include <cuda.h>
#include "device_common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace rga {

constexpr int DEC_THREADS = DEC_WARPS * 32;

template <int D>
struct DecLayout {
    static constexpr int BLK = DEC_KEYS * 128;          // 32 rows x 64 columns x 2 bytes
    static constexpr int TILE = (D / 64) * BLK;          // one K or V tile
    static constexpr int STAGE = 2 * TILE;               // K + V
    static constexpr int WARP_RING = DEC_STAGES * STAGE;
    static constexpr int RING = DEC_WARPS * WARP_RING;
    static constexpr int BAR_OFF = RING;
    static constexpr int BOFF_OFF = BAR_OFF + DEC_WARPS * DEC_STAGES * 8 + 64;
    static constexpr int BYTES = BOFF_OFF + (DEC_MAX_B + 1) * 4 + 64;
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

__device__ __forceinline__ void dec_tma(const AttnParams &p, const TensorMaps &tm,
                                        const SeqInfo &s, int b, int g, int j0, uint8_t *dst,
                                        uint64_t *bar, int D) {
    const int tile = (D / 64) * DEC_KEYS * 128;
    mbar_arrive_expect_tx(bar, 2 * tile);
    for (int blk = 0; blk < D / 64; ++blk) {
        uint8_t *kd = dst + blk * DEC_KEYS * 128;
        uint8_t *vd = dst + tile + blk * DEC_KEYS * 128;
        if (p.kv_packed) {
            tma_load_3d(kd, &tm.k, bar, blk * 64, g, s.kv_off + j0);
            tma_load_3d(vd, &tm.v, bar, blk * 64, g, s.kv_off + j0);
        } else {
            tma_load_4d(kd, &tm.k, bar, blk * 64, j0, g, b);
            tma_load_4d(vd, &tm.v, bar, blk * 64, j0, g, b);
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

// One 32-key tile for the warp's 16 query rows: S = Q K^T, scale and mask,
// online softmax (or 'none'), O += P V.  Rows rr[0..1] are this lane's rows
// (lane/4 and lane/4 + 8); kb/vb: the tile's K and V in shared memory.
template <int D, bool BF16, bool SOFTMAX>
__device__ __forceinline__ void dec_tile(const AttnParams &p, const DecRow (&rr)[2],
                                         const uint32_t (&qa)[D / 16][4], uint32_t kb,
                                         uint32_t vb, int j0, float (&o)[D / 8][4],
                                         float (&m_r)[2], float (&l_r)[2]) {
    using L = DecLayout<D>;
    constexpr int NT = D / 8, KS = D / 16;
    const int lane = threadIdx.x & 31;
    const float sc = SOFTMAX ? p.scale_log2 : p.scale;
    float sacc[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ks += 2) {
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4(kb + swz(nt * 8 + (lane & 7), ks * 2 + (lane >> 3), L::BLK), r0, r1, r2, r3);
            mma16816<BF16>(sacc[nt], qa[ks], r0, r1);
            mma16816<BF16>(sacc[nt], qa[ks + 1], r2, r3);
        }
    }
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const DecRow &R = rr[e >> 1];
            const int j = j0 + nt * 8 + (lane & 3) * 2 + (e & 1);
            bool ok = j <= R.lim;
            float add = 0.f;
            if (ok && p.mask) ok = mask_at(p, p.md[3] == 1 ? R.mrow : R.mrow + j, add);
            const float v = sacc[nt][e] * sc + (SOFTMAX ? add * 1.4426950408889634f : add);
            sacc[nt][e] = ok ? v : (SOFTMAX ? -INFINITY : 0.f);
            mx[e >> 1] = fmaxf(mx[e >> 1], sacc[nt][e]);
        }
    if (SOFTMAX) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
            const float m_new = fmaxf(m_r[r], mx[r]);
            const float mu = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = ex2(m_r[r] - mu);
            l_r[r] *= alpha;
#pragma unroll
            for (int n = 0; n < NT; ++n) { o[n][2 * r] *= alpha; o[n][2 * r + 1] *= alpha; }
            m_r[r] = m_new;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                sacc[nt][2 * r] = ex2(sacc[nt][2 * r] - mu);
                sacc[nt][2 * r + 1] = ex2(sacc[nt][2 * r + 1] - mu);
                l_r[r] += sacc[nt][2 * r] + sacc[nt][2 * r + 1];
            }
        }
    }
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
        uint32_t a[4];
        a[0] = pack2<BF16>(sacc[2 * kk][0], sacc[2 * kk][1]);
        a[1] = pack2<BF16>(sacc[2 * kk][2], sacc[2 * kk][3]);
        a[2] = pack2<BF16>(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
        a[3] = pack2<BF16>(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
#pragma unroll
        for (int n = 0; n < NT; n += 2) {
            uint32_t r0, r1, r2, r3;
            const int mi = lane >> 3;
            ldsm_x4_t(vb + swz(kk * 16 + (mi & 1) * 8 + (lane & 7), n + (mi >> 1), L::BLK),
                      r0, r1, r2, r3);
            mma16816<BF16>(o[n], a, r0, r1);
            mma16816<BF16>(o[n + 1], a, r2, r3);
        }
    }
}

// Y row of this lane's fragment rows, scaled by f (rows outside are skipped).
template <int D, bool BF16>
__device__ __forceinline__ void dec_store_y(const AttnParams &p, const DecRow (&rr)[2],
                                            const float (&o)[D / 8][4], const float (&f)[2]) {
    const int lane = threadIdx.x & 31;
    uint16_t *y = static_cast<uint16_t *>(p.y);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        if (!rr[r].valid) continue;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
            const int col = n * 8 + (lane & 3) * 2;
            *reinterpret_cast<uint32_t *>(y + rr[r].qoff + col) =
                pack2<BF16>(o[n][2 * r] * f[r], o[n][2 * r + 1] * f[r]);
        }
    }
}

template <int D, bool BF16, bool SOFTMAX>
__global__ void __launch_bounds__(DEC_THREADS, 1)
decode_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ TensorMaps tm) {
    using L = DecLayout<D>;
    constexpr int NT = D / 8;
    constexpr int KS = D / 16;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::BAR_OFF);
    volatile int *abort = reinterpret_cast<volatile int *>(sm + L::BAR_OFF + DEC_WARPS * DEC_STAGES * 8);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    int *boff = reinterpret_cast<int *>(sm + L::BOFF_OFF);    // first unit of each batch
    int *flags = reinterpret_cast<int *>(sm + L::BAR_OFF + DEC_WARPS * DEC_STAGES * 8 + 4);
    if (threadIdx.x == 0) {
        for (int i = 0; i < DEC_WARPS * DEC_STAGES; ++i) mbar_init(&bars[i], 1);
        *abort = 0;
        flags[0] = 0;   // bad lengths
        fence_mbar_init();
    }
    __syncthreads();
    // Every CTA validates the lengths and lists the units itself: unit u of
    // batch b is (split, KV head) = ((u - boff[b]) / Hkv, (u - boff[b]) % Hkv).
    for (int b = threadIdx.x; b < p.B; b += DEC_THREADS) {
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
        boff[b + 1] = (ok && s.q_len > 0) ? dec_splits(p, s) * p.Hkv : 0;
    }
    __syncthreads();
    if (flags[0]) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_status(p.status, 4);
        return;
    }
    if (threadIdx.x == 0) {   // prefix over batches (serial: B is at most DEC_MAX_B)
        boff[0] = 0;
        for (int b = 0; b < p.B; ++b) boff[b + 1] += boff[b];
    }
    __syncthreads();
    const int n_units = boff[p.B];
    pdl_wait();   // the tickets and the unit counter have been cleared
    int *tickets = reinterpret_cast<int *>(p.ws + dec_tickets_off(p));
    float *part = reinterpret_cast<float *>(p.ws + dec_part_off(p));
    float2 *pml = reinterpret_cast<float2 *>(p.ws + dec_ml_off(p));

    uint8_t *ring = sm + warp * L::WARP_RING;
    uint64_t *wbar = bars + warp * DEC_STAGES;
    const uint32_t ring_u32 = smem_u32(ring);
    uint32_t issued = 0, consumed = 0;

    int *next_unit = tickets + p.B * p.Hkv;    // cleared with the tickets
    for (;;) {
        int u = 0;
        if (lane == 0) u = atomicAdd(next_unit, 1);
        u = __shfl_sync(0xffffffffu, u, 0);
        if (u >= n_units || *abort) break;
        int lo = 0, hi = p.B;   // boff[lo] <= u < boff[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (boff[mid] <= u) lo = mid; else hi = mid;
        }
        const int b = lo;
        const int g = (u - boff[b]) % p.Hkv, split = (u - boff[b]) / p.Hkv;
        const int ns = (boff[b + 1] - boff[b]) / p.Hkv;
        const SeqInfo s = seq_info(p, b);
        const int rows = s.q_len * p.G;
        const int kv_hi = key_extent(p.causal, s.q_len - 1, s);
        const int k0 = split * DEC_SPLIT;
        const int k1 = (ns == 1) ? kv_hi : min(kv_hi, k0 + DEC_SPLIT);
        const int ntiles = k1 > k0 ? (k1 - k0 + DEC_KEYS - 1) / DEC_KEYS : 0;
        const int nrc = (rows + DEC_ROWS - 1) / DEC_ROWS;
        const size_t unit_idx = ((size_t)b * p.Hkv + g) * p.max_splits + split;
        bool unit_ok = true;

        for (int rc = 0; rc < nrc && unit_ok; ++rc) {
            DecRow rr[2];
            rr[0] = dec_row(p, s, b, g, rc * DEC_ROWS + (lane >> 2), rows, k1);
            rr[1] = dec_row(p, s, b, g, rc * DEC_ROWS + (lane >> 2) + 8, rows, k1);
            uint32_t qa[KS][4];
            const uint32_t *q32 = static_cast<const uint32_t *>(p.q);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int col = ks * 16 + (lane & 3) * 2;
                qa[ks][0] = rr[0].valid ? q32[(rr[0].qoff + col) >> 1] : 0u;
                qa[ks][1] = rr[1].valid ? q32[(rr[1].qoff + col) >> 1] : 0u;
                qa[ks][2] = rr[0].valid ? q32[(rr[0].qoff + col + 8) >> 1] : 0u;
                qa[ks][3] = rr[1].valid ? q32[(rr[1].qoff + col + 8) >> 1] : 0u;
            }
            float o[NT][4];
#pragma unroll
            for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
            float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};

            if (lane == 0)
                for (int it = 0; it < DEC_STAGES && it < ntiles; ++it) {
                    const uint32_t c = issued + it;
                    dec_tma(p, tm, s, b, g, k0 + it * DEC_KEYS, ring + (c % DEC_STAGES) * L::STAGE,
                            &wbar[c % DEC_STAGES], D);
                }
            issued += min(DEC_STAGES, ntiles);
            for (int it = 0; it < ntiles; ++it) {
                const uint32_t c = consumed;
                const int st = c % DEC_STAGES;
                if (!mbar_wait(&wbar[st], (c / DEC_STAGES) & 1, abort)) { unit_ok = false; break; }
                ++consumed;
                const int j0 = k0 + it * DEC_KEYS;
                const uint32_t kb = ring_u32 + st * L::STAGE, vb = kb + L::TILE;
                const int rem = s.kv_len - j0;
                if (rem < DEC_KEYS) {   // rows past the sequence end may hold NaN: zero them
                    uint8_t *vp = ring + st * L::STAGE + L::TILE;
                    for (int idx = lane; idx < DEC_KEYS * (D / 8); idx += 32) {
                        const int row = idx / (D / 8), ch = idx % (D / 8);
                        if (row >= rem)
                            *reinterpret_cast<uint4 *>(vp + swz(row, ch, L::BLK)) = make_uint4(0, 0, 0, 0);
                    }
                    __syncwarp();
                }
                dec_tile<D, BF16, SOFTMAX>(p, rr, qa, kb, vb, j0, o, m_r, l_r);
                __syncwarp();
                if (it + DEC_STAGES < ntiles) {   // refill the stage just used
                    if (lane == 0) {
                        fence_proxy_async_smem();
                        dec_tma(p, tm, s, b, g, k0 + (it + DEC_STAGES) * DEC_KEYS,
                                ring + (issued % DEC_STAGES) * L::STAGE, &wbar[issued % DEC_STAGES], D);
                    }
                    ++issued;
                }
            }
            if (!unit_ok) break;
            if (SOFTMAX)
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 1);
                    l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 2);
                }
            if (ns == 1) {
                float f[2];
#pragma unroll
                for (int r = 0; r < 2; ++r)
                    f[r] = SOFTMAX ? (l_r[r] > 0.f ? 1.f / l_r[r] : 0.f) : 1.f;
                dec_store_y<D, BF16>(p, rr, o, f);
            } else {
                // partial (O, m, l) of this split
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int row = (lane >> 2) + 8 * r;
                    float *po = part + (unit_idx * DEC_ROWS + row) * D;
#pragma unroll
                    for (int n = 0; n < NT; ++n)
                        *reinterpret_cast<float2 *>(po + n * 8 + (lane & 3) * 2) =
                            make_float2(o[n][2 * r], o[n][2 * r + 1]);
                    if ((lane & 3) == 0) pml[unit_idx * DEC_ROWS + row] = make_float2(m_r[r], l_r[r]);
                }
            }
        }
        if (!unit_ok) break;
        if (ns > 1) {
            // the last split of the pair to finish merges all of them
            __threadfence();
            __syncwarp();
            int t = 0;
            if (lane == 0) t = atomicAdd(&tickets[b * p.Hkv + g], 1);
            t = __shfl_sync(0xffffffffu, t, 0);
            if (t == ns - 1) {
                __threadfence();
                const size_t u0 = ((size_t)b * p.Hkv + g) * p.max_splits;
                const int row = lane >> 1, c0 = (lane & 1) * (D / 2);
                float M = -INFINITY;
                if (SOFTMAX)
                    for (int sp = 0; sp < ns; ++sp) M = fmaxf(M, __ldcg(&pml[(u0 + sp) * DEC_ROWS + row].x));
                float acc[D / 2];
#pragma unroll
                for (int c = 0; c < D / 2; ++c) acc[c] = 0.f;
                float Lsum = 0.f;
                for (int sp = 0; sp < ns; ++sp) {
                    float wt = 1.f;
                    if (SOFTMAX) {
                        const float2 v = __ldcg(&pml[(u0 + sp) * DEC_ROWS + row]);
                        wt = (v.x == -INFINITY) ? 0.f : ex2(v.x - M);
                        Lsum += v.y * wt;
                    }
                    const float4 *src = reinterpret_cast<const float4 *>(part + ((u0 + sp) * DEC_ROWS + row) * D + c0);
#pragma unroll
                    for (int c = 0; c < D / 8; ++c) {
                        const float4 x4 = __ldcg(src + c);
                        acc[4 * c] += x4.x * wt;
                        acc[4 * c + 1] += x4.y * wt;
                        acc[4 * c + 2] += x4.z * wt;
                        acc[4 * c + 3] += x4.w * wt;
                    }
                }
                const DecRow R = dec_row(p, s, b, g, row, rows, k1);
                if (R.valid) {
                    const float f = SOFTMAX ? (Lsum > 0.f ? 1.f / Lsum : 0.f) : 1.f;
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.y) + R.qoff + c0);
#pragma unroll
                    for (int c = 0; c < D / 16; ++c)
                        dst[c] = make_uint4(pack2<BF16>(acc[8 * c] * f, acc[8 * c + 1] * f),
                                            pack2<BF16>(acc[8 * c + 2] * f, acc[8 * c + 3] * f),
                                            pack2<BF16>(acc[8 * c + 4] * f, acc[8 * c + 5] * f),
                                            pack2<BF16>(acc[8 * c + 6] * f, acc[8 * c + 7] * f));
                }
                if (lane == 0) tickets[b * p.Hkv + g] = 0;
            }
        }
    }
    // copies still in flight (only after an abort) land before the CTA exits
    while (consumed < issued) {
        mbar_wait_drain(&wbar[consumed % DEC_STAGES], (consumed / DEC_STAGES) & 1);
        ++consumed;
    }
    __syncwarp();
    if (lane == 0 && *abort) set_status(p.status, 5);
}

// Clears the split tickets and the next-unit counter of a decode call; the
// decode kernel follows it as a programmatic dependent.
__global__ void decode_prep_kernel(int *tickets, int n) {
    pdl_launch_dependents();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        tickets[i] = 0;
}

template <int D, bool BF16, bool SOFTMAX>
static cudaError_t dec_launch(const AttnParams &p, const TensorMaps &m, cudaStream_t s) {
    using L = DecLayout<D>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, BF16, SOFTMAX>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int n = p.B * p.Hkv + 1;
    decode_prep_kernel<<<(n + 255) / 256 < 64 ? (n + 255) / 256 : 64, 256, 0, s>>>(
        reinterpret_cast<int *>(p.ws + dec_tickets_off(p)), n);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_dependent(decode_kernel<D, BF16, SOFTMAX>, p.grid, DEC_THREADS, L::ALLOC, s, p, m);
}

cudaError_t launch_decode(const AttnParams &p, const TensorMaps &m, int mode, cudaStream_t s,
                          int bf16) {
    const bool sm = (mode == MODE_SOFTMAX);
    if (p.D == 64) {
        if (bf16) return sm ? dec_launch<64, true, true>(p, m, s) : dec_launch<64, true, false>(p, m, s);
        return sm ? dec_launch<64, false, true>(p, m, s) : dec_launch<64, false, false>(p, m, s);
    }
    if (bf16) return sm ? dec_launch<128, true, true>(p, m, s) : dec_launch<128, true, false>(p, m, s);
    return sm ? dec_launch<128, false, true>(p, m, s) : dec_launch<128, false, false>(p, m, s);
}

}  // namespace rga
