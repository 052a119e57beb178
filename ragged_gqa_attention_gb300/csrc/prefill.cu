// prefill.cu - fused attention forward for sm_103a on the 5th-generation
// tensor cores (tcgen05 + TMEM), with TMA-staged, 128-byte-swizzled Q/K/V
// tiles and warp-specialised roles.
//
// Computes, per work item (batch b, KV head g, query tile):
//   S = Q K^T (BMM1, fp32 in TMEM)  ->  scale, causal / length / mask
//   ->  softmax (online, fp32, exp2) or 'none'  ->  optional fp8/int8 Q/DQ
//   ->  O += P V (BMM2, fp32 in TMEM)  ->  O / l  ->  Y
// following "TensorRT Custom Operator Schemas" (TRT_Attention,
// TRT_QuantizedAttention) and the MHA/GQA AttentionPlugin of the "TensorRT
// Plugins Guide".
//
// GQA reuse: the 128 rows of a query tile are the G = Hq/Hkv query heads of
// one KV head times 128/G tokens, so every K/V tile is loaded once for the
// whole group.  Row r maps to (token t, head hh) as r = t*G + hh for packed
// Q ([T,H,D]: the G heads of a token are adjacent) and r = hh*TQ + t for
// padded Q ([B,H,N,D]).
//
// Roles (192 threads):
//   warps 0-3  softmax / correction / epilogue; thread = TMEM lane = row
//   warp 4     TMEM owner and single-thread MMA issuer
//   warp 5     TMA producer (Q once per item, K and V rings)
// TMEM columns: S0 [0,128), S1 [128,256), O [256, 256+D).  P (16-bit) is
// written over the S buffer it came from and fed to BMM2 from TMEM.
//
// The grid is persistent (one CTA per SM); CTA c takes items c, c+grid, ...
// of the work list, which the scheduler sorted longest first.
#include <cuda.h>
#include "device_common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace rga {

constexpr int PF_THREADS = 192;
constexpr int KST = 2;      // K ring stages
constexpr int VST = 2;      // V ring stages
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t S_COL0 = 0, O_COL = 256;
constexpr float RESCALE_THRESHOLD = 8.0f;   // log2 units: rescale O when the max grows by > 2^8

template <int D>
struct PfLayout {
    static constexpr int BLK = 128 * 128;                // one 64-column block of 128 rows
    static constexpr int NBLK = D / 64;
    static constexpr int TILE = NBLK * BLK;              // 128 rows x D x 2 bytes
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + TILE;
    static constexpr int V_OFF = K_OFF + KST * TILE;
    static constexpr int BAR_OFF = V_OFF + VST * TILE;
    // barriers: q_full, q_empty, k_full[KST], k_empty[KST], v_full[VST],
    // v_empty[VST], s_full[2], p_full[2], o_done
    static constexpr int NBAR = 2 + 2 * KST + 2 * VST + 2 + 2 + 1;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr int BYTES = MISC_OFF + 64;
    // room to align the base to 1024; at least 120 KB so that only one CTA
    // (and one 512-column TMEM allocation) is resident per SM
    static constexpr int ALLOC = (BYTES + 1024) > 120 * 1024 ? (BYTES + 1024) : 120 * 1024;
};

struct PfBars {
    uint64_t *q_full, *q_empty, *k_full, *k_empty, *v_full, *v_empty, *s_full, *p_full,
        *o_done;
};

__device__ __forceinline__ PfBars pf_bars(uint8_t *base) {
    uint64_t *b = reinterpret_cast<uint64_t *>(base);
    PfBars r;
    r.q_full = b;
    r.q_empty = b + 1;
    r.k_full = b + 2;
    r.k_empty = b + 2 + KST;
    r.v_full = b + 2 + 2 * KST;
    r.v_empty = b + 2 + 2 * KST + VST;
    r.s_full = b + 2 + 2 * KST + 2 * VST;
    r.p_full = r.s_full + 2;
    r.o_done = r.p_full + 2;
    return r;
}

// Per-item geometry, computed identically by every role.
struct Item {
    int b, qt, g;
    SeqInfo s;
    int i0;          // first query token of the tile (within the sequence)
    int ntok;        // valid tokens in the tile
    int nkt;         // key tiles visited
    int ntiles;      // BMM1 steps (2 * nkt for the two-pass quantized softmax)
};

template <int MODE>
__device__ __forceinline__ Item load_item(const AttnParams &p, int idx) {
    const int4 it = reinterpret_cast<const int4 *>(p.ws + WS_HEADER)[idx];
    Item m;
    m.b = it.x;
    m.qt = it.y;
    m.g = it.z;
    m.s = seq_info(p, m.b);
    m.i0 = m.qt * p.tq;
    m.ntok = min(p.tq, m.s.q_len - m.i0);
    int n = key_extent(p.causal, m.i0 + m.ntok - 1, m.s);
    m.nkt = (n + BN - 1) / BN;
    m.ntiles = (MODE == MODE_SOFTMAX_Q) ? 2 * m.nkt : m.nkt;
    return m;
}

// Whether BMM1 step t (of ntiles) is followed by a BMM2 (pass 1 of the
// two-pass quantized softmax only gathers row statistics).
template <int MODE>
__device__ __forceinline__ bool is_pv(const Item &m, int t) {
    return MODE != MODE_SOFTMAX_Q || t >= m.nkt;
}
template <int MODE>
__device__ __forceinline__ int key_tile(const Item &m, int t) {
    return (MODE == MODE_SOFTMAX_Q && t >= m.nkt) ? t - m.nkt : t;
}

// ------------------------------------------------------------------ producer
// Load a partial V tile (keys j0 .. j0+127 with only `rem` < 128 valid) with
// plain loads, zero the rows past the sequence end (they may hold NaN), and
// publish it to the tensor core through the async proxy.
template <int D>
__device__ void load_v_partial(const AttnParams &p, const Item &m, int j0, int rem,
                               uint8_t *dst, int lane) {
    constexpr int CH = D / 8;   // 16-byte chunks per row
    const uint16_t *v = static_cast<const uint16_t *>(p.v);
    for (int idx = lane; idx < 128 * CH; idx += 32) {
        const int r = idx / CH, c = idx % CH;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (r < rem) {
            const long long j = (long long)j0 + r;
            long long off = p.kv_packed
                ? ((m.s.kv_off + j) * p.Hkv + m.g) * (long long)D
                : (((long long)m.b * p.Hkv + m.g) * p.kv_seq + j) * (long long)D;
            val = *reinterpret_cast<const uint4 *>(v + off + c * 8);
        }
        const int blk = c / 8, cc = c % 8;
        uint8_t *row = dst + blk * PfLayout<D>::BLK + r * 128;
        *reinterpret_cast<uint4 *>(row + ((cc ^ (r & 7)) * 16)) = val;
    }
    fence_proxy_async_smem();
    __syncwarp();
}

// TMA box coordinates of the Q tile / a K or V tile (per 64-column block).
__device__ __forceinline__ void tma_q(const AttnParams &p, const CUtensorMap *map,
                                      const Item &m, void *dst, uint64_t *bar, int d0) {
    if (p.q_packed)   // dims (D, Hq, T): box (64, G, TQ)
        tma_load_3d(dst, map, bar, d0, m.g * p.G, m.s.q_off + m.i0);
    else              // dims (D, Nq, Hq, B): box (64, TQ, G, 1)
        tma_load_4d(dst, map, bar, d0, m.i0, m.g * p.G, m.b);
}
__device__ __forceinline__ void tma_kv(const AttnParams &p, const CUtensorMap *map,
                                       const Item &m, int j0, void *dst, uint64_t *bar,
                                       int d0) {
    if (p.kv_packed)  // dims (D, Hkv, T): box (64, 1, 128)
        tma_load_3d(dst, map, bar, d0, m.g, m.s.kv_off + j0);
    else              // dims (D, Nkv, Hkv, B): box (64, 128, 1, 1)
        tma_load_4d(dst, map, bar, d0, j0, m.g, m.b);
}

template <int D, int MODE>
__device__ void producer_role(const AttnParams &p, const TensorMaps &tm, uint8_t *sm,
                              const PfBars &bar, volatile int *abort, int n_items) {
    using L = PfLayout<D>;
    const int lane = threadIdx.x & 31;
    const uint32_t q_bytes = (uint32_t)(L::NBLK * p.G * p.tq * 128);
    const uint32_t kv_bytes = (uint32_t)L::TILE;
    uint32_t kc = 0, vc = 0, qc = 0;   // running ring counters
    for (int idx = blockIdx.x; idx < n_items && !*abort; idx += gridDim.x) {
        const Item m = load_item<MODE>(p, idx);
        if (m.nkt == 0) continue;
        // Q tile, once per item (wait until the previous item's BMM1s are done)
        if (qc > 0 && !mbar_wait(bar.q_empty, (qc - 1) & 1, abort)) break;
        if (lane == 0) {
            mbar_arrive_expect_tx(bar.q_full, q_bytes);
            for (int blk = 0; blk < L::NBLK; ++blk)
                tma_q(p, &tm.q, m, sm + L::Q_OFF + blk * L::BLK, bar.q_full, blk * 64);
        }
        ++qc;
        for (int t = 0; t < m.ntiles && !*abort; ++t) {
            const int j0 = key_tile<MODE>(m, t) * BN;
            const int ks = kc % KST;
            if (kc >= KST && !mbar_wait(&bar.k_empty[ks], ((kc / KST) - 1) & 1, abort)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(&bar.k_full[ks], kv_bytes);
                for (int blk = 0; blk < L::NBLK; ++blk)
                    tma_kv(p, &tm.k, m, j0, sm + L::K_OFF + ks * L::TILE + blk * L::BLK,
                           &bar.k_full[ks], blk * 64);
            }
            ++kc;
            if (!is_pv<MODE>(m, t)) continue;
            const int vs = vc % VST;
            if (vc >= VST && !mbar_wait(&bar.v_empty[vs], ((vc / VST) - 1) & 1, abort)) break;
            uint8_t *vdst = sm + L::V_OFF + vs * L::TILE;
            const int rem = m.s.kv_len - j0;
            if (rem >= BN) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bar.v_full[vs], kv_bytes);
                    for (int blk = 0; blk < L::NBLK; ++blk)
                        tma_kv(p, &tm.v, m, j0, vdst + blk * L::BLK, &bar.v_full[vs], blk * 64);
                }
            } else {
                load_v_partial<D>(p, m, j0, rem, vdst, lane);
                if (lane == 0) mbar_arrive(&bar.v_full[vs]);
            }
            ++vc;
        }
    }
    // Before the CTA exits, let every copy this warp started land.
    for (uint32_t c = kc > KST ? kc - KST : 0; c < kc; ++c)
        mbar_wait_drain(&bar.k_full[c % KST], (c / KST) & 1);
    for (uint32_t c = vc > VST ? vc - VST : 0; c < vc; ++c)
        mbar_wait_drain(&bar.v_full[c % VST], (c / VST) & 1);
    if (qc > 0) mbar_wait_drain(bar.q_full, (qc - 1) & 1);
}

// ------------------------------------------------------------------ MMA issuer
// One thread issues every tcgen05.mma.  BMM1 of step t+1 is queued before
// BMM2 of step t, so the tensor core computes the next scores while the
// softmax warps turn the current scores into probabilities.
template <int D, int MODE, bool BF16>
__device__ void mma_role(const AttnParams &p, uint8_t *sm, const PfBars &bar,
                         volatile int *abort, int n_items, uint32_t tmem) {
    using L = PfLayout<D>;
    constexpr uint32_t ID_S = idesc_f16(BF16 ? 1 : 0, 128, BN, 0, 0);   // Q K-major, K K-major
    constexpr uint32_t ID_O = idesc_f16(BF16 ? 1 : 0, 128, D, 0, 1);    // P from TMEM, V MN-major
    const uint32_t q_base = smem_u32(sm + L::Q_OFF);
    const uint32_t k_base = smem_u32(sm + L::K_OFF);
    const uint32_t v_base = smem_u32(sm + L::V_OFF);
    uint32_t kc = 0, vc = 0, qc = 0, tc = 0;
    bool ok = true;
    for (int idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x) {
        const Item m = load_item<MODE>(p, idx);
        if (m.nkt == 0) continue;
        if (!mbar_wait(bar.q_full, qc & 1, abort)) break;
        ++qc;
        int u = 0;   // BMM2 steps issued for this item
        // BMM2 for step t (its P must be ready)
        auto issue_pv = [&](int t, uint32_t tcount) -> bool {
            const uint32_t sb = tcount & 1;
            if (!mbar_wait(&bar.p_full[sb], (tcount >> 1) & 1, abort)) return false;
            tc_fence_after();
            if (!is_pv<MODE>(m, t)) return true;
            const int vs = vc % VST;
            if (!mbar_wait(&bar.v_full[vs], (vc / VST) & 1, abort)) return false;
            tc_fence_after();
            const uint32_t vb = v_base + vs * L::TILE;
            const uint32_t pa = tmem + S_COL0 + sb * 128;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
                mma_ts(tmem + O_COL, pa + kk * 8, sdesc(vb + kk * 2048, L::BLK, 1024), ID_O,
                       (u > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&bar.v_empty[vs]);
            mma_commit(bar.o_done);
            ++vc;
            ++u;
            return true;
        };
        for (int t = 0; t < m.ntiles; ++t) {
            const int ks = kc % KST;
            if (!mbar_wait(&bar.k_full[ks], (kc / KST) & 1, abort)) { ok = false; break; }
            tc_fence_after();
            const uint32_t kb = k_base + ks * L::TILE;
            const uint32_t sb = tc & 1;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * L::BLK + (kk & 3) * 32;
                mma_ss(tmem + S_COL0 + sb * 128, sdesc(q_base + off, 16, 1024),
                       sdesc(kb + off, 16, 1024), ID_S, kk > 0 ? 1u : 0u);
            }
            mma_commit(&bar.k_empty[ks]);
            mma_commit(&bar.s_full[sb]);
            if (t == m.ntiles - 1) mma_commit(bar.q_empty);
            ++kc;
            if (t > 0 && !issue_pv(t - 1, tc - 1)) { ok = false; break; }
            ++tc;
        }
        if (ok && !issue_pv(m.ntiles - 1, tc - 1)) ok = false;
    }
}

// ------------------------------------------------------------------ softmax
constexpr float LOG2E = 1.4426950408889634f;

// Load this thread's 128 scores (its TMEM lane, 128 columns).
__device__ __forceinline__ void load_scores(uint32_t taddr, float (&x)[BN]) {
    uint32_t r[32];
#pragma unroll
    for (int c = 0; c < BN / 32; ++c) {
        tmem_ld32(taddr + c * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k) x[c * 32 + k] = __uint_as_float(r[k]);
    }
}

// Per-element scale and masking of a partial tile.  Writes log2-domain
// scores (softmax) or natural-unit scores ('none') and -inf / excluded
// marks; returns the row max of the result.
template <bool LOG2>
__device__ __forceinline__ float mask_scores(const AttnParams &p, float (&x)[BN], int j0,
                                             int lim, long long mrow, bool use_mask) {
    const float sc = LOG2 ? p.scale_log2 : p.scale;
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < BN; ++c) {
        const int j = j0 + c;
        bool ok = j <= lim;
        float add = 0.f;
        if (use_mask && ok) ok = mask_at(p, p.md[3] == 1 ? mrow : mrow + j, add);
        float v = x[c] * sc + (LOG2 ? add * LOG2E : add);
        x[c] = ok ? v : -INFINITY;
        mx = fmaxf(mx, x[c]);
    }
    return mx;
}

template <int D, bool BF16>
__device__ __forceinline__ void store_row(const AttnParams &p, const Item &m, int i, int h,
                                          uint32_t o_taddr, float f, bool zero, bool write) {
    // every lane takes part in the (warp-collective) TMEM loads; only rows
    // that belong to the sequence are written
    uint16_t *y = static_cast<uint16_t *>(p.y);
    const long long off = p.q_packed
        ? ((long long)(m.s.q_off + i) * p.Hq + h) * D
        : (((long long)m.b * p.Hq + h) * p.q_seq + i) * D;
    uint4 *dst = reinterpret_cast<uint4 *>(y + off);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        if (!zero) {
            tmem_ld32(o_taddr + c * 32, r);
            tmem_wait_ld();
        }
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
            w[k] = zero ? 0u
                        : pack2<BF16>(__uint_as_float(r[2 * k]) * f,
                                      __uint_as_float(r[2 * k + 1]) * f);
        if (write) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                dst[c * 4 + k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
        }
    }
}

template <int D, int MODE, bool BF16>
__device__ void softmax_role(const AttnParams &p, const PfBars &bar, volatile int *abort,
                             int n_items, uint32_t tmem) {
    constexpr bool SOFTMAX = (MODE == MODE_SOFTMAX || MODE == MODE_SOFTMAX_Q);
    constexpr bool QUANT = (MODE == MODE_SOFTMAX_Q || MODE == MODE_NONE_Q);
    const int r = threadIdx.x;                 // row = TMEM lane
    const uint32_t lane_base = (uint32_t)((r & ~31) << 16);
    const int G = p.G, TQ = p.tq;
    const int t_row = p.q_packed ? r / G : r % TQ;
    const int hh = p.q_packed ? r % G : r / TQ;
    const bool in_tile = r < G * TQ;
    const float qs = QUANT ? load_qscale(p) : 1.f;
    const float inv_qs = 1.f / qs;
    uint32_t tc = 0, pvw = 0;                  // S-buffer uses, BMM2 completions waited
    bool ok = true;

    for (int idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x) {
        const Item m = load_item<MODE>(p, idx);
        const int i = m.i0 + t_row;
        const int h = m.g * G + hh;
        const bool row_ok = in_tile && t_row < m.ntok;
        if (m.nkt == 0) {                      // no attendable key: the rows are zero
            store_row<D, BF16>(p, m, i, h, 0, 0.f, true, row_ok);
            continue;
        }
        const int lim = row_ok ? min(causal_limit(p.causal, i, m.s), m.s.kv_len - 1) : -1;
        const int lim_first = min(causal_limit(p.causal, m.i0, m.s), m.s.kv_len - 1);
        const bool use_mask = p.mask != nullptr;
        const long long mrow = (use_mask && row_ok) ? mask_row(p, m.b, h, i) : 0;
        float m_ref = -INFINITY, l = 0.f;
        float lse2 = 0.f;                      // pass 2 of the quantized softmax
        int u = 0;
        for (int t = 0; t < m.ntiles; ++t) {
            const uint32_t sb = tc & 1;
            if (!mbar_wait(&bar.s_full[sb], (tc >> 1) & 1, abort)) { ok = false; break; }
            tc_fence_after();
            const int j0 = key_tile<MODE>(m, t) * BN;
            const uint32_t s_addr = tmem + lane_base + S_COL0 + sb * 128;
            float x[BN];
            load_scores(s_addr, x);
            const bool full = !use_mask && j0 + BN - 1 <= lim_first;
            // scaled scores: log2 domain for softmax, natural units for 'none'
            float mx;
            if (full) {
                const float sc = SOFTMAX ? p.scale_log2 : p.scale;
                mx = -INFINITY;
#pragma unroll
                for (int c = 0; c < BN; ++c) { x[c] *= sc; mx = fmaxf(mx, x[c]); }
                if (!row_ok) mx = -INFINITY;
            } else {
                mx = mask_scores<SOFTMAX>(p, x, j0, lim, mrow, use_mask && row_ok);
            }

            if (MODE == MODE_SOFTMAX_Q && t < m.nkt) {
                // pass 1: exact row max and sum only
                const float m_new = fmaxf(m_ref, mx);
                if (m_new != -INFINITY) {
                    float sum = 0.f;
#pragma unroll
                    for (int c = 0; c < BN; ++c) sum += ex2(x[c] - m_new);
                    l = l * ex2(m_ref - m_new) + sum;
                    m_ref = m_new;
                }
                if (t == m.nkt - 1)
                    lse2 = (l > 0.f) ? m_ref + log2f(l) + log2f(qs) : INFINITY;
                tc_fence_before();
                mbar_arrive(&bar.p_full[sb]);
                ++tc;
                continue;
            }

            float alpha = 1.f;
            bool need = false;
            float mu = 0.f;
            if (MODE == MODE_SOFTMAX) {
                const float m_new = fmaxf(m_ref, mx);
                if (m_new > m_ref + RESCALE_THRESHOLD) {
                    alpha = ex2(m_ref - m_new);
                    l *= alpha;
                    m_ref = m_new;
                    need = true;
                }
                mu = (m_ref == -INFINITY) ? 0.f : m_ref;
            }
            // P for this tile, 16-bit pairs over the S columns it came from
            float psum = 0.f;
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t w[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    float a = x[c * 32 + 2 * k], b = x[c * 32 + 2 * k + 1];
                    if (MODE == MODE_SOFTMAX) {
                        a = ex2(a - mu);
                        b = ex2(b - mu);
                        psum += a + b;
                    } else if (MODE == MODE_NONE) {
                        a = (a == -INFINITY) ? 0.f : a;
                        b = (b == -INFINITY) ? 0.f : b;
                    } else {
                        if (MODE == MODE_SOFTMAX_Q) {   // p / s_q, exactly normalised
                            a = ex2(a - lse2);
                            b = ex2(b - lse2);
                        } else {                        // 'none': s / s_q
                            a = (a == -INFINITY) ? 0.f : a * inv_qs;
                            b = (b == -INFINITY) ? 0.f : b * inv_qs;
                        }
                        if (p.quant == 0) {
                            float2 e = e4m3_round2(a, b);
                            a = e.x;
                            b = e.y;
                        } else {
                            a = int8_round(a);
                            b = int8_round(b);
                        }
                    }
                    w[k] = pack2<BF16>(a, b);
                }
                tmem_st16(s_addr + c * 16, w);
            }
            l += psum;
            if (u > 0) {   // BMM2 of the previous step must be done before O is touched
                if (!mbar_wait(bar.o_done, pvw & 1, abort)) { ok = false; break; }
                ++pvw;
                if (MODE == MODE_SOFTMAX && __any_sync(0xffffffffu, need)) {
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tmem + lane_base + O_COL + c * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                        tmem_st32(tmem + lane_base + O_COL + c * 32, o);
                    }
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bar.p_full[sb]);
            ++u;
            ++tc;
        }
        if (!ok) break;
        // epilogue: the last BMM2 of the item
        if (!mbar_wait(bar.o_done, pvw & 1, abort)) { ok = false; break; }
        ++pvw;
        tc_fence_after();
        float f;
        if (MODE == MODE_SOFTMAX) f = (l > 0.f) ? 1.f / l : 0.f;
        else f = qs;    // 'none': 1; quantized: the Q/DQ scale
        store_row<D, BF16>(p, m, i, h, tmem + lane_base + O_COL, f, false, row_ok);
        tc_fence_before();
    }
}

// ------------------------------------------------------------------ kernel
template <int D, int MODE, bool BF16>
__global__ void __launch_bounds__(PF_THREADS, 1)
prefill_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ TensorMaps tm) {
    using L = PfLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const PfBars bar = pf_bars(sm + L::BAR_OFF);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::MISC_OFF);
    volatile int *abort = reinterpret_cast<volatile int *>(sm + L::MISC_OFF + 8);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_items = *reinterpret_cast<volatile const int *>(p.ws);

    if (threadIdx.x == 0) {
        mbar_init(bar.q_full, 1);
        mbar_init(bar.q_empty, 1);
        for (int s = 0; s < KST; ++s) { mbar_init(&bar.k_full[s], 1); mbar_init(&bar.k_empty[s], 1); }
        for (int s = 0; s < VST; ++s) { mbar_init(&bar.v_full[s], 1); mbar_init(&bar.v_empty[s], 1); }
        for (int s = 0; s < 2; ++s) { mbar_init(&bar.s_full[s], 1); mbar_init(&bar.p_full[s], 128); }
        mbar_init(bar.o_done, 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 4) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 5 && lane == 0) {
        prefetch_tmap(&tm.q);
        prefetch_tmap(&tm.k);
        prefetch_tmap(&tm.v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {
        softmax_role<D, MODE, BF16>(p, bar, abort, n_items, tmem);
    } else if (warp == 4) {
        if (lane == 0) mma_role<D, MODE, BF16>(p, sm, bar, abort, n_items, tmem);
        __syncwarp();
    } else {
        producer_role<D, MODE>(p, tm, sm, bar, abort, n_items);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 4) tmem_dealloc(tmem, TMEM_COLS);
    if (threadIdx.x == 0 && *abort) set_status(p.status, 5);
}

template <int D, int MODE, bool BF16>
static cudaError_t launch_one(const AttnParams &p, const TensorMaps &m, int grid,
                              cudaStream_t s) {
    using L = PfLayout<D>;
    static bool attr_set = false;   // per process; the attribute is per function
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D, MODE, BF16>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             L::ALLOC);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    prefill_kernel<D, MODE, BF16><<<grid, PF_THREADS, L::ALLOC, s>>>(p, m);
    return cudaGetLastError();
}

template <int D, bool BF16>
static cudaError_t launch_mode(const AttnParams &p, const TensorMaps &m, int mode, int grid,
                               cudaStream_t s) {
    switch (mode) {
    case MODE_SOFTMAX: return launch_one<D, MODE_SOFTMAX, BF16>(p, m, grid, s);
    case MODE_NONE: return launch_one<D, MODE_NONE, BF16>(p, m, grid, s);
    case MODE_SOFTMAX_Q: return launch_one<D, MODE_SOFTMAX_Q, BF16>(p, m, grid, s);
    default: return launch_one<D, MODE_NONE_Q, BF16>(p, m, grid, s);
    }
}

cudaError_t launch_prefill(const AttnParams &p, const TensorMaps &m, int mode, int grid,
                           cudaStream_t s, int bf16) {
    if (p.D == 64)
        return bf16 ? launch_mode<64, true>(p, m, mode, grid, s)
                    : launch_mode<64, false>(p, m, mode, grid, s);
    return bf16 ? launch_mode<128, true>(p, m, mode, grid, s)
                : launch_mode<128, false>(p, m, mode, grid, s);
}

}  // namespace rga
