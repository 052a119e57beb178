// decode.cu - split-KV attention for short query lengths (decode), the
// HBM-bound path of the AttentionPlugin ("TensorRT Plugins Guide":
// vanilla decoding attention) with the TRT_Attention semantics of
// "TensorRT Custom Operator Schemas".
//
// Work unit: (batch b, KV head g, split of DEC_SPLIT keys).  The query rows
// of the unit are the (token, head) pairs of the G query heads of KV head g,
// taken 16 at a time (one MMA row block).  Each of the 4 warps streams its
// share of 32-key K/V tiles with TMA into its own double-buffered,
// 128-byte-swizzled ring, computes S = Q K^T and O += P V with m16n8k16
// MMAs (K and V are read once from HBM for all G heads), and keeps an
// online softmax in fp32 registers.  The warps' partial (m, l, O) are merged
// in shared memory; splits are merged through the workspace by the last CTA
// of the (b, g) pair to arrive (atomic ticket).
//
// A pair with more than 16 query rows (more than 16/G tokens) is handled by
// a single split that loops over the row blocks.
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
    static constexpr int COMB = DEC_WARPS * DEC_ROWS * D * 4;   // fp32 partial O per warp
    static constexpr int DATA = RING > COMB ? RING : COMB;
    static constexpr int BAR_OFF = DATA;
    static constexpr int ML_OFF = BAR_OFF + DEC_WARPS * DEC_STAGES * 8;
    static constexpr int MISC_OFF = ML_OFF + DEC_WARPS * DEC_ROWS * 8;
    static constexpr int BYTES = MISC_OFF + 64;
    static constexpr int ALLOC = BYTES + 1024;
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

template <int D, bool BF16, bool SOFTMAX>
__global__ void __launch_bounds__(DEC_THREADS)
decode_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ TensorMaps tm) {
    using L = DecLayout<D>;
    constexpr int NT = D / 8;     // 8-column output tiles
    constexpr int KS = D / 16;    // 16-deep k-steps over the head dimension
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::BAR_OFF);
    float2 *mlw = reinterpret_cast<float2 *>(sm + L::ML_OFF);
    volatile int *abort = reinterpret_cast<volatile int *>(sm + L::MISC_OFF);
    int *ticket_s = reinterpret_cast<int *>(sm + L::MISC_OFF + 4);
    float *comb = reinterpret_cast<float *>(sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (reinterpret_cast<const volatile int *>(p.ws)[0] == 0) return;   // lengths rejected
    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const SeqInfo s = seq_info(p, b);
    const int rows = s.q_len * p.G;
    if (rows <= 0) return;
    const int kv_hi = key_extent(p.causal, s.q_len - 1, s);
    const int nrc = (rows + DEC_ROWS - 1) / DEC_ROWS;
    int nsplit = (kv_hi + DEC_SPLIT - 1) / DEC_SPLIT;
    if (nsplit < 1 || nrc > 1) nsplit = 1;
    if (split >= nsplit) return;
    const int k0 = split * DEC_SPLIT;
    const int k1 = (nsplit == 1) ? kv_hi : min(kv_hi, k0 + DEC_SPLIT);

    if (threadIdx.x == 0) {
        for (int i = 0; i < DEC_WARPS * DEC_STAGES; ++i) mbar_init(&bars[i], 1);
        *abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    uint8_t *ring = sm + warp * L::WARP_RING;
    uint64_t *wbar = bars + warp * DEC_STAGES;
    const int ntiles = (k1 - k0 + DEC_KEYS - 1) / DEC_KEYS;
    const int my_n = ntiles > warp ? (ntiles - warp + DEC_WARPS - 1) / DEC_WARPS : 0;
    const uint32_t ring_u32 = smem_u32(ring);
    uint32_t issued = 0, consumed = 0;
    const float sc = SOFTMAX ? p.scale_log2 : p.scale;
    const float LOG2E_ = 1.4426950408889634f;

    for (int rc = 0; rc < nrc; ++rc) {
        // ---- this lane's two rows (lane/4 and lane/4 + 8) and Q fragments
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

        // ---- prefetch
        if (lane == 0)
            for (int it = 0; it < DEC_STAGES && it < my_n; ++it) {
                const uint32_t u = issued + it;
                dec_tma(p, tm, s, b, g, k0 + (warp + it * DEC_WARPS) * DEC_KEYS,
                        ring + (u % DEC_STAGES) * L::STAGE, &wbar[u % DEC_STAGES], D);
            }
        issued += min(DEC_STAGES, my_n);

        // ---- stream this warp's key tiles
        for (int it = 0; it < my_n && !*abort; ++it) {
            const uint32_t u = consumed;
            const int st = u % DEC_STAGES;
            if (!mbar_wait(&wbar[st], (u / DEC_STAGES) & 1, abort)) break;
            ++consumed;
            const int j0 = k0 + (warp + it * DEC_WARPS) * DEC_KEYS;
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
            // S = Q K^T  (16 rows x 32 keys)
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
            // scale, mask, online softmax
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
                    const float v = sacc[nt][e] * sc + (SOFTMAX ? add * LOG2E_ : add);
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
            // O += P V
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
            __syncwarp();
            // refill this stage
            const int nxt = it + DEC_STAGES;
            if (nxt < my_n) {
                if (lane == 0) {
                    fence_proxy_async_smem();
                    dec_tma(p, tm, s, b, g, k0 + (warp + nxt * DEC_WARPS) * DEC_KEYS,
                            ring + (issued % DEC_STAGES) * L::STAGE, &wbar[issued % DEC_STAGES], D);
                }
                ++issued;
            }
        }
        // copies still in flight (only after an abort) land before reuse
        while (consumed < issued) {
            mbar_wait_drain(&wbar[consumed % DEC_STAGES], (consumed / DEC_STAGES) & 1);
            ++consumed;
        }

        // ---- merge the 4 warps' partials in shared memory (reuses the ring)
        if (SOFTMAX)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 1);
                l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 2);
            }
        __syncthreads();
        {
            float *cw = comb + warp * DEC_ROWS * D;
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int row = (lane >> 2) + (e >> 1) * 8;
                    const int col = n * 8 + (lane & 3) * 2 + (e & 1);
                    cw[row * D + col] = o[n][e];
                }
            if ((lane & 3) == 0) {
                mlw[warp * DEC_ROWS + (lane >> 2)] = make_float2(m_r[0], l_r[0]);
                mlw[warp * DEC_ROWS + (lane >> 2) + 8] = make_float2(m_r[1], l_r[1]);
            }
        }
        __syncthreads();
        {
            constexpr int CPT = D / 8;                 // columns per thread (8 threads per row)
            const int row = threadIdx.x >> 3, c0 = (threadIdx.x & 7) * CPT;
            float wts[DEC_WARPS];
            float M = -INFINITY, Lsum = 0.f;
            if (SOFTMAX) {
#pragma unroll
                for (int w = 0; w < DEC_WARPS; ++w) M = fmaxf(M, mlw[w * DEC_ROWS + row].x);
#pragma unroll
                for (int w = 0; w < DEC_WARPS; ++w) {
                    const float2 v = mlw[w * DEC_ROWS + row];
                    wts[w] = (v.x == -INFINITY) ? 0.f : ex2(v.x - M);
                    Lsum += v.y * wts[w];
                }
            } else {
#pragma unroll
                for (int w = 0; w < DEC_WARPS; ++w) wts[w] = 1.f;
            }
            float acc[CPT];
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                float a = 0.f;
#pragma unroll
                for (int w = 0; w < DEC_WARPS; ++w) a += comb[(w * DEC_ROWS + row) * D + c0 + c] * wts[w];
                acc[c] = a;
            }
            const DecRow R = dec_row(p, s, b, g, rc * DEC_ROWS + row, rows, k1);
            if (nsplit == 1) {
                if (R.valid && !*abort) {
                    const float f = SOFTMAX ? (Lsum > 0.f ? 1.f / Lsum : 0.f) : 1.f;
                    uint32_t w[CPT / 2];
#pragma unroll
                    for (int c = 0; c < CPT / 2; ++c) w[c] = pack2<BF16>(acc[2 * c] * f, acc[2 * c + 1] * f);
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.y) + R.qoff + c0);
#pragma unroll
                    for (int c = 0; c < CPT / 8; ++c)
                        dst[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
                }
            } else {
                const size_t unit = ((size_t)b * p.Hkv + g) * p.max_splits + split;
                float *po = reinterpret_cast<float *>(p.ws + dec_part_off(p)) + (unit * DEC_ROWS + row) * D;
#pragma unroll
                for (int c = 0; c < CPT; ++c) po[c0 + c] = acc[c];
                if ((threadIdx.x & 7) == 0) {
                    float2 *pml = reinterpret_cast<float2 *>(p.ws + dec_ml_off(p));
                    pml[unit * DEC_ROWS + row] = make_float2(M, Lsum);
                }
            }
        }
        __syncthreads();
    }

    // ---- merge the splits of this (batch, KV head): the last CTA to finish does it
    if (nsplit > 1) {
        __threadfence();
        __syncthreads();
        int *tickets = reinterpret_cast<int *>(p.ws + WS_HEADER);
        if (threadIdx.x == 0) *ticket_s = atomicAdd(&tickets[b * p.Hkv + g], 1);
        __syncthreads();
        if (*ticket_s != nsplit - 1) return;
        __threadfence();
        constexpr int CPT = D / 8;
        const int row = threadIdx.x >> 3, c0 = (threadIdx.x & 7) * CPT;
        const size_t unit0 = ((size_t)b * p.Hkv + g) * p.max_splits;
        const float *po = reinterpret_cast<const float *>(p.ws + dec_part_off(p));
        const float2 *pml = reinterpret_cast<const float2 *>(p.ws + dec_ml_off(p));
        float M = -INFINITY;
        if (SOFTMAX)
            for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, __ldcg(&pml[(unit0 + sp) * DEC_ROWS + row].x));
        float acc[CPT];
#pragma unroll
        for (int c = 0; c < CPT; ++c) acc[c] = 0.f;
        float Lsum = 0.f;
        for (int sp = 0; sp < nsplit; ++sp) {
            float wt = 1.f;
            if (SOFTMAX) {
                const float2 v = __ldcg(&pml[(unit0 + sp) * DEC_ROWS + row]);
                wt = (v.x == -INFINITY) ? 0.f : ex2(v.x - M);
                Lsum += v.y * wt;
            }
            const float *src = po + ((unit0 + sp) * DEC_ROWS + row) * D + c0;
#pragma unroll
            for (int c = 0; c < CPT; ++c) acc[c] += __ldcg(src + c) * wt;
        }
        const DecRow R = dec_row(p, s, b, g, row, rows, k1);
        if (R.valid && !*abort) {
            const float f = SOFTMAX ? (Lsum > 0.f ? 1.f / Lsum : 0.f) : 1.f;
            uint32_t w[CPT / 2];
#pragma unroll
            for (int c = 0; c < CPT / 2; ++c) w[c] = pack2<BF16>(acc[2 * c] * f, acc[2 * c + 1] * f);
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.y) + R.qoff + c0);
#pragma unroll
            for (int c = 0; c < CPT / 8; ++c)
                dst[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        }
        if (threadIdx.x == 0) tickets[b * p.Hkv + g] = 0;
    }
    if (threadIdx.x == 0 && *abort) set_status(p.status, 5);
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
    dim3 grid(p.max_splits, p.Hkv, p.B);
    decode_kernel<D, BF16, SOFTMAX><<<grid, DEC_THREADS, L::ALLOC, s>>>(p, m);
    return cudaGetLastError();
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
