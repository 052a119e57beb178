// decode.cu - split-KV attention for short query lengths (decode), the
// HBM-bound path of the AttentionPlugin ("TensorRT Plugins Guide":
// vanilla decoding attention) with the TRT_Attention semantics of
// "TensorRT Custom Operator Schemas".
//
// Work: pairs (batch b, KV head g, chunk of 16 query rows), each with the
// 32-key tiles of the batch's key extent.  The query rows of a pair are the
// (token, head) pairs of the G heads of g, 16 at a time (one MMA row block).
// All tiles of all pairs form one batch-major line that is cut into equal
// contiguous ranges, one per warp of the persistent grid, so that every
// warp streams the same number of tiles and none is left finishing a long
// unit alone at the end.  Each CTA validates the lengths and lays out the
// line itself (no scheduler launch).  A warp streams its range's K/V tiles
// with TMA through its own DEC_STAGES-deep, 128-byte-swizzled ring, straight
// across pair boundaries, computes S = Q K^T and O += P V with m16n8k16 MMAs
// (K and V are read once from HBM for all G query heads of the KV head) and
// keeps an online softmax in fp32 registers.  A pair inside one range is
// written to Y by its warp; a pair cut by range ends leaves a partial
// (O, m, l) per warp, and the last of its warps to finish (atomic ticket)
// merges them in warp order and writes Y.
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
    static constexpr int SCR_OFF = BAR_OFF + DEC_WARPS * DEC_STAGES * 8 + 64;   // prefix scratch
    static constexpr int TPRE_OFF = SCR_OFF + (DEC_THREADS + 1) * 4 + 12;
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

// One lane's view of the pair being computed or loaded: a pair is
// (batch b, KV head g, row chunk rc of DEC_ROWS query rows); its key tiles
// are the 32-key tiles of [0, key extent of the batch).
struct DecCur {
    int b, pib;          // batch, pair within the batch (g * nrc + rc)
    int tile;            // tile within the pair
    int nt, nrc;         // tiles per pair, row chunks of the batch
    SeqInfo s;
};

// Batch b's row chunks and key tiles per pair (0 chunks: no query rows).
__device__ __forceinline__ void dec_batch_shape(const AttnParams &p, const SeqInfo &s, int &nrc,
                                                int &nt) {
    const int rows = s.q_len * p.G;
    nrc = (rows + DEC_ROWS - 1) / DEC_ROWS;
    const int kv_hi = rows > 0 ? key_extent(p.causal, s.q_len - 1, s) : 0;
    nt = (kv_hi + DEC_KEYS - 1) / DEC_KEYS;
}

// Block-wide exclusive prefix of v[0..n) in place (n <= DEC_MAX_B), with
// v[n] set to the total; every thread of the block calls it.
__device__ __forceinline__ void dec_prefix(int *v, int n, int *scratch) {
    const int per = (n + DEC_THREADS - 1) / DEC_THREADS;
    const int lo = threadIdx.x * per, hi = min(n, lo + per);
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += v[i];
    scratch[threadIdx.x] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int t = 0; t < DEC_THREADS; ++t) {
            const int x = scratch[t];
            scratch[t] = run;
            run += x;
        }
        scratch[DEC_THREADS] = run;
    }
    __syncthreads();
    int run = scratch[threadIdx.x];
    for (int i = lo; i < hi; ++i) {
        const int x = v[i];
        v[i] = run;
        run += x;
    }
    if (threadIdx.x == 0) v[n] = scratch[DEC_THREADS];
    __syncthreads();
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
    int *flags = reinterpret_cast<int *>(sm + L::BAR_OFF + DEC_WARPS * DEC_STAGES * 8 + 4);
    int *scratch = reinterpret_cast<int *>(sm + L::SCR_OFF);
    int *tpre = reinterpret_cast<int *>(sm + L::TPRE_OFF);   // key tiles before batch b
    int *ppre = reinterpret_cast<int *>(sm + L::PPRE_OFF);   // pairs before batch b
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < DEC_WARPS * DEC_STAGES; ++i) mbar_init(&bars[i], 1);
        *abort = 0;
        flags[0] = 0;   // bad lengths
        fence_mbar_init();
    }
    __syncthreads();
    // Every CTA validates the lengths and lays out the work itself.
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
        int nrc = 0, nt = 0;
        if (ok) dec_batch_shape(p, s, nrc, nt);
        tpre[b] = p.Hkv * nrc * nt;
        ppre[b] = p.Hkv * nrc;
    }
    __syncthreads();
    if (flags[0]) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_status(p.status, 4);
        return;
    }
    dec_prefix(tpre, p.B, scratch);
    dec_prefix(ppre, p.B, scratch);
    pdl_wait();   // the tickets have been cleared

    // Stream-K split of the work: all key tiles of all pairs, batch-major,
    // in one line of T tiles, cut into equal contiguous ranges, one per warp
    // of the grid.  A pair inside one range is finished by its warp; a pair
    // cut by range ends is finished by the last of its warps to arrive
    // (atomic ticket), which merges the others' partials in warp order.
    const int T = tpre[p.B];
    const int wg = blockIdx.x * DEC_WARPS + warp;
    // at most one warp per tile, so that every range holds at least one
    // (the merge counts a pair's warps from the range ends); later warps idle
    const int Wn = max(1, min((int)gridDim.x * DEC_WARPS, T));
    auto range_start = [&](int w) { return (int)((long long)w * T / Wn); };
    auto warp_of = [&](int x) { return (int)(((long long)(x + 1) * Wn - 1) / T); };
    int *tickets = reinterpret_cast<int *>(p.ws + dec_tickets_off(p));
    float *part = reinterpret_cast<float *>(p.ws + dec_part_off(p));
    float2 *pml = reinterpret_cast<float2 *>(p.ws + dec_ml_off(p));

    // batches with query rows but no key tile: their rows are zero
    for (int b = wg; b < p.B; b += gridDim.x * DEC_WARPS) {
        const SeqInfo s = seq_info(p, b);
        int nrc, nt;
        dec_batch_shape(p, s, nrc, nt);
        if (nrc == 0 || nt > 0) continue;
        const int rows = s.q_len * p.G;
        for (int r = lane; r < p.Hkv * rows; r += 32) {
            const DecRow R = dec_row(p, s, b, r / rows, r % rows, rows, 0);
            uint4 *y = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.y) + R.qoff);
            for (int c = 0; c < D / 8; ++c) y[c] = make_uint4(0, 0, 0, 0);
        }
    }

    uint8_t *ring = sm + warp * L::WARP_RING;
    uint64_t *wbar = bars + warp * DEC_STAGES;
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
        dec_batch_shape(p, c.s, c.nrc, c.nt);
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
        dec_batch_shape(p, c.s, c.nrc, c.nt);
    };
    auto issue = [&](const DecCur &c) {
        if (lane == 0) {
            fence_proxy_async_smem();   // the stage's previous tile was read by ldmatrix
            dec_tma(p, tm, c.s, c.b, c.pib / c.nrc, c.tile * DEC_KEYS,
                    ring + (issued % DEC_STAGES) * L::STAGE, &wbar[issued % DEC_STAGES], D);
        }
        ++issued;
    };

    bool ok = true;
    if (t_begin < t_end) {
        DecCur lc, cc;
        locate(t_begin, lc);
        cc = lc;
        int next_issue = t_begin;
        for (; next_issue < t_end && next_issue < t_begin + DEC_STAGES; ++next_issue) {
            issue(lc);
            advance(lc);
        }
        DecRow rr[2];
        uint32_t qa[KS][4];
        float o[NT][4];
        float m_r[2], l_r[2];
        int seg0 = t_begin;    // first tile of the current pair in this range
        int kv_hi = 0, rows = 0;
        auto start_pair = [&]() {
            const int g = cc.pib / cc.nrc, rc = cc.pib % cc.nrc;
            rows = cc.s.q_len * p.G;
            kv_hi = key_extent(p.causal, cc.s.q_len - 1, cc.s);
            rr[0] = dec_row(p, cc.s, cc.b, g, rc * DEC_ROWS + (lane >> 2), rows, kv_hi);
            rr[1] = dec_row(p, cc.s, cc.b, g, rc * DEC_ROWS + (lane >> 2) + 8, rows, kv_hi);
            const uint32_t *q32 = static_cast<const uint32_t *>(p.q);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int col = ks * 16 + (lane & 3) * 2;
                qa[ks][0] = rr[0].valid ? q32[(rr[0].qoff + col) >> 1] : 0u;
                qa[ks][1] = rr[1].valid ? q32[(rr[1].qoff + col) >> 1] : 0u;
                qa[ks][2] = rr[0].valid ? q32[(rr[0].qoff + col + 8) >> 1] : 0u;
                qa[ks][3] = rr[1].valid ? q32[(rr[1].qoff + col + 8) >> 1] : 0u;
            }
#pragma unroll
            for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
            m_r[0] = m_r[1] = -INFINITY;
            l_r[0] = l_r[1] = 0.f;
        };
        start_pair();

        for (int t = t_begin; t < t_end; ++t) {
            const uint32_t c = consumed;
            const int st = c % DEC_STAGES;
            if (!mbar_wait(&wbar[st], (c / DEC_STAGES) & 1, abort)) { ok = false; break; }
            ++consumed;
            const int j0 = cc.tile * DEC_KEYS;
            const uint32_t kb = ring_u32 + st * L::STAGE, vb = kb + L::TILE;
            const int rem = cc.s.kv_len - j0;
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
            if (next_issue < t_end) {   // refill the stage just used
                issue(lc);
                advance(lc);
                ++next_issue;
            }
            const bool pair_end = cc.tile + 1 == cc.nt;
            if (pair_end || t + 1 == t_end) {
                // this range's share of the pair is done
                if (SOFTMAX)
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 1);
                        l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 2);
                    }
                const int b = cc.b, g = cc.pib / cc.nrc, rc = cc.pib % cc.nrc;
                const int ps = tpre[b] + cc.pib * cc.nt, pe = ps + cc.nt;
                if (seg0 == ps && t + 1 == pe) {   // the whole pair: write Y
                    float f[2];
#pragma unroll
                    for (int r = 0; r < 2; ++r)
                        f[r] = SOFTMAX ? (l_r[r] > 0.f ? 1.f / l_r[r] : 0.f) : 1.f;
                    dec_store_y<D, BF16>(p, rr, o, f);
                } else {
                    // partial (O, m, l): slot 0 for the first pair of the
                    // range, slot 1 for the last
                    const size_t slot = (size_t)wg * 2 + (seg0 == t_begin ? 0 : 1);
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int row = (lane >> 2) + 8 * r;
                        float *po = part + (slot * DEC_ROWS + row) * D;
#pragma unroll
                        for (int n = 0; n < NT; ++n)
                            *reinterpret_cast<float2 *>(po + n * 8 + (lane & 3) * 2) =
                                make_float2(o[n][2 * r], o[n][2 * r + 1]);
                        if ((lane & 3) == 0) pml[slot * DEC_ROWS + row] = make_float2(m_r[r], l_r[r]);
                    }
                    __threadfence();
                    __syncwarp();
                    const int w_lo = warp_of(ps), w_hi = warp_of(pe - 1);
                    const int pidx = ppre[b] + cc.pib;
                    int tk = 0;
                    if (lane == 0) tk = atomicAdd(&tickets[pidx], 1);
                    tk = __shfl_sync(0xffffffffu, tk, 0);
                    if (tk == w_hi - w_lo) {   // the last of the pair's warps: merge
                        __threadfence();
                        const int row = lane >> 1, c0 = (lane & 1) * (D / 2);
                        // the first warp's share is its slot 1 unless the pair
                        // starts its range; every later warp's share is its slot 0
                        auto slot_of = [&](int w) -> size_t {
                            return (size_t)w * 2 + ((w == w_lo && range_start(w) != ps) ? 1 : 0);
                        };
                        float M = -INFINITY;
                        if (SOFTMAX)
                            for (int w = w_lo; w <= w_hi; ++w)
                                M = fmaxf(M, __ldcg(&pml[slot_of(w) * DEC_ROWS + row].x));
                        float acc[D / 2];
#pragma unroll
                        for (int k = 0; k < D / 2; ++k) acc[k] = 0.f;
                        float Lsum = 0.f;
                        for (int w = w_lo; w <= w_hi; ++w) {
                            const size_t sl = slot_of(w);
                            float wt = 1.f;
                            if (SOFTMAX) {
                                const float2 v = __ldcg(&pml[sl * DEC_ROWS + row]);
                                wt = (v.x == -INFINITY) ? 0.f : ex2(v.x - M);
                                Lsum += v.y * wt;
                            }
                            const float4 *src = reinterpret_cast<const float4 *>(part + (sl * DEC_ROWS + row) * D + c0);
#pragma unroll
                            for (int k = 0; k < D / 8; ++k) {
                                const float4 x4 = __ldcg(src + k);
                                acc[4 * k] += x4.x * wt;
                                acc[4 * k + 1] += x4.y * wt;
                                acc[4 * k + 2] += x4.z * wt;
                                acc[4 * k + 3] += x4.w * wt;
                            }
                        }
                        const DecRow R = dec_row(p, cc.s, b, g, rc * DEC_ROWS + row, rows, kv_hi);
                        if (R.valid) {
                            const float f = SOFTMAX ? (Lsum > 0.f ? 1.f / Lsum : 0.f) : 1.f;
                            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.y) + R.qoff + c0);
#pragma unroll
                            for (int k = 0; k < D / 16; ++k)
                                dst[k] = make_uint4(pack2<BF16>(acc[8 * k] * f, acc[8 * k + 1] * f),
                                                    pack2<BF16>(acc[8 * k + 2] * f, acc[8 * k + 3] * f),
                                                    pack2<BF16>(acc[8 * k + 4] * f, acc[8 * k + 5] * f),
                                                    pack2<BF16>(acc[8 * k + 6] * f, acc[8 * k + 7] * f));
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
        mbar_wait_drain(&wbar[consumed % DEC_STAGES], (consumed / DEC_STAGES) & 1);
        ++consumed;
    }
    __syncwarp();
    if (lane == 0 && (!ok || *abort)) set_status(p.status, 5);
}

// Clears the merge tickets of a decode call; the decode kernel follows it as
// a programmatic dependent.
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
    const int n = p.max_pairs + 1;
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
