// rope.cu - rotary position embedding ("TensorRT Plugins Guide",
// AttentionPlugin: rotary positional encoding; RopeCosSin rows aligned with
// the physical token rows, position -1 marking padding rows), in place on
// Q/K rows, and fused with the KV cache update of the new keys
// ("TensorRT Custom Operator Schemas", TRT_KVCacheUpdate, packed form).
//
// Row t, head h, pair i < R/2 (R = rotary_dim) with c, s from row t of the
// cos/sin table:  x'[i] = x[i] c - x[i + R/2] s,  x'[i + R/2] = x[i + R/2] c
// + x[i] s.  HBM-bound elementwise work: one unit is eight consecutive
// pairs of one (row, head) (16-byte loads of each half and of the cosines
// and sines), or four (8-byte loads) where the rotary dims, the head dim or
// a base address do not allow 16-byte vectors; in the fused form a unit of
// the new keys writes its
// rotated (or, past the rotary dims, copied) elements straight into the
// cache row the update lands in.  The fused form checks every window first,
// in every CTA, so that a bad call changes nothing (status 4).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>
#include "rga.h"
#include "device_common.cuh"
#include "kernels.h"

namespace rga {

constexpr int ROPE_THREADS = 256;
constexpr int ROPE_MAX_B = 8192;

struct RopeParams {
    uint16_t *q, *k;            // rotated in place (k: the standalone form only)
    int T, Hq, Hk, D, R;
    const float *cs;            // [T, R]
    const int32_t *pos;         // [T] or null
    // fused form: update rows [T, Hk, D] into cache [B, Hk, N, D] in place
    const uint16_t *upd;
    uint16_t *cache;
    int B, N;
    const int32_t *wi, *cu;
    int32_t *status;
};

// P consecutive 16-bit elements (P = 4: 8 bytes, P = 8: 16 bytes) as one
// vector, unpacked to and packed from fp32.
template <int P> struct Vec;
template <> struct Vec<4> { using T = uint2; };
template <> struct Vec<8> { using T = uint4; };

template <bool BF16, int P>
__device__ __forceinline__ void unpack(const typename Vec<P>::T &w, float (&x)[P]) {
    const uint32_t *u = reinterpret_cast<const uint32_t *>(&w);
#pragma unroll
    for (int i = 0; i < P / 2; ++i) {
        if constexpr (BF16) {
            x[2 * i] = __uint_as_float(u[i] << 16);
            x[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
        } else {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&u[i]));
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        }
    }
}

template <bool BF16, int P>
__device__ __forceinline__ typename Vec<P>::T pack(const float (&x)[P]) {
    typename Vec<P>::T w;
    uint32_t *u = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
    for (int i = 0; i < P / 2; ++i) {
        if constexpr (BF16) {
            __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
            u[i] = *reinterpret_cast<uint32_t *>(&h);
        } else {
            __half2 h = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
            u[i] = *reinterpret_cast<uint32_t *>(&h);
        }
    }
    return w;
}

// Pairs P u .. P u + P - 1 of one row: src -> dst (may alias), rotated with
// the table row cs, or copied unchanged when !rotate.
template <bool BF16, int P>
__device__ __forceinline__ void rope_group(const uint16_t *src, uint16_t *dst, const float *cs,
                                           int R, int u, bool rotate) {
    using V = typename Vec<P>::T;
    const int h = R / 2;
    const V a = *reinterpret_cast<const V *>(src + P * u);
    const V b = *reinterpret_cast<const V *>(src + P * u + h);
    if (!rotate) {
        *reinterpret_cast<V *>(dst + P * u) = a;
        *reinterpret_cast<V *>(dst + P * u + h) = b;
        return;
    }
    float c[P], sn[P];
#pragma unroll
    for (int q = 0; q < P / 4; ++q) {
        const float4 c4 = *reinterpret_cast<const float4 *>(cs + P * u + 4 * q);
        const float4 s4 = *reinterpret_cast<const float4 *>(cs + h + P * u + 4 * q);
        c[4 * q] = c4.x; c[4 * q + 1] = c4.y; c[4 * q + 2] = c4.z; c[4 * q + 3] = c4.w;
        sn[4 * q] = s4.x; sn[4 * q + 1] = s4.y; sn[4 * q + 2] = s4.z; sn[4 * q + 3] = s4.w;
    }
    float x[P], y[P], xo[P], yo[P];
    unpack<BF16, P>(a, x);
    unpack<BF16, P>(b, y);
#pragma unroll
    for (int e = 0; e < P; ++e) {
        xo[e] = fmaf(x[e], c[e], -(y[e] * sn[e]));
        yo[e] = fmaf(y[e], c[e], x[e] * sn[e]);
    }
    *reinterpret_cast<V *>(dst + P * u) = pack<BF16, P>(xo);
    *reinterpret_cast<V *>(dst + P * u + h) = pack<BF16, P>(yo);
}

// I: the index type of the unit loop (32-bit whenever every unit index and
// row offset fits: the divisions that map a unit to its row are then cheap).
// P: pairs per unit (8 when the rotary dims, the head dim and every base
// address allow 16-byte vectors, else 4).
template <bool BF16, bool FUSED, typename I, int P>
__global__ void __launch_bounds__(ROPE_THREADS) rope_kernel(const __grid_constant__ RopeParams p) {
    extern __shared__ int rope_smem[];
    int *s_cu = rope_smem;            // fused: [B + 1] cumulative update rows
    int *s_w = rope_smem + p.B + 1;   // fused: [B] write positions
    if constexpr (FUSED) {
        __shared__ int bad;
        if (threadIdx.x == 0) bad = 0;
        __syncthreads();
        for (int b = threadIdx.x; b <= p.B; b += ROPE_THREADS) {
            s_cu[b] = p.cu[b];
            if (b < p.B) s_w[b] = p.wi ? p.wi[b] : 0;
        }
        __syncthreads();
        for (int b = threadIdx.x; b < p.B; b += ROPE_THREADS) {
            const int len = s_cu[b + 1] - s_cu[b];
            bool ok = len >= 0 && s_w[b] >= 0 && (long long)s_w[b] + len <= p.N &&
                      s_cu[b + 1] <= p.T;
            if (b == 0) ok = ok && s_cu[0] == 0;
            if (!ok) atomicOr(&bad, 1);
        }
        __syncthreads();
        if (bad) {
            if (blockIdx.x == 0 && threadIdx.x == 0) set_status(p.status, 4);
            return;
        }
    }
    const int G4 = p.R / (2 * P);                 // rotated P-pair groups per row
    const int CG = FUSED ? (p.D - p.R) / P : 0;   // copied P-element groups (fused keys)
    const I nq = p.q ? (I)p.T * p.Hq * G4 : 0;
    const I nk = (!FUSED && p.k) ? (I)p.T * p.Hk * G4 : 0;
    const I nu = FUSED ? (I)s_cu[p.B] * p.Hk * (G4 + CG) : 0;
    const I total = nq + nk + nu;
    for (I i = (I)blockIdx.x * ROPE_THREADS + threadIdx.x; i < total;
         i += (I)gridDim.x * ROPE_THREADS) {
        if (i < nq + nk) {   // in place on Q (then K)
            const bool isq = i < nq;
            const I j = isq ? i : i - nq;
            const int H = isq ? p.Hq : p.Hk;
            const int u = (int)(j % (I)G4);
            const I r = j / (I)G4;                 // (t, h) row
            const int t = (int)(r / (I)H);
            if (p.pos && p.pos[t] < 0) continue;   // padding row: left as it is
            if (!dbg_ok(t < p.T && 2 * P * (u + 1) <= p.R, p.status)) continue;
            uint16_t *row = (isq ? p.q : p.k) + (long long)r * p.D;
            rope_group<BF16, P>(row, row, p.cs + (long long)t * p.R, p.R, u, true);
        } else {             // fused: the new keys into their cache rows
            const I j = i - nq;
            const int per = G4 + CG;
            const int u = (int)(j % (I)per);
            const I r = j / (I)per;                // (update row, head)
            const int tg = (int)(r / (I)p.Hk), h = (int)(r % (I)p.Hk);
            int lo = 0, hi = p.B;                  // s_cu[lo] <= tg < s_cu[lo + 1]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (s_cu[mid] <= tg) lo = mid; else hi = mid;
            }
            const int n = s_w[lo] + (tg - s_cu[lo]);
            if (!dbg_ok(tg < p.T && n >= 0 && n < p.N, p.status)) continue;
            const uint16_t *src = p.upd + (long long)r * p.D;
            uint16_t *dst = p.cache + (((long long)lo * p.Hk + h) * p.N + n) * p.D;
            if (u < G4) {
                const bool rot = !(p.pos && p.pos[tg] < 0);
                rope_group<BF16, P>(src, dst, p.cs + (long long)tg * p.R, p.R, u, rot);
            } else {
                using V = typename Vec<P>::T;
                const int d0 = p.R + P * (u - G4);
                *reinterpret_cast<V *>(dst + d0) = *reinterpret_cast<const V *>(src + d0);
            }
        }
    }
}

static bool aligned(const void *ptr, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0;
}

static rga_status check_rope(const rga_rope_args *r, bool need_qk) {
    if (!r) return RGA_ERR_INVALID_ARG;
    if (r->dtype != RGA_F16 && r->dtype != RGA_BF16) return RGA_ERR_INVALID_ARG;
    if (r->tokens < 0 || r->head_dim <= 0 || r->head_dim % 4 != 0) return RGA_ERR_INVALID_ARG;
    if (r->rotary_dim <= 0 || r->rotary_dim % 8 != 0 || r->rotary_dim > r->head_dim)
        return RGA_ERR_INVALID_ARG;
    if (!r->cos_sin || !aligned(r->cos_sin, 16)) return RGA_ERR_INVALID_ARG;
    if (need_qk && !r->q && !r->k) return RGA_ERR_INVALID_ARG;
    if (r->q && (r->q_heads <= 0 || !aligned(r->q, 8))) return RGA_ERR_INVALID_ARG;
    if (r->k && (r->kv_heads <= 0 || !aligned(r->k, 8))) return RGA_ERR_INVALID_ARG;
    return RGA_OK;
}

template <bool FUSED>
static rga_status rope_launch(const RopeParams &p, bool bf16, bool wide, long long units4,
                              cudaStream_t s) {
    if (units4 <= 0 && !FUSED) return RGA_OK;
    const int sms = sm_count();
    if (sms <= 0) return RGA_ERR_CUDA;
    // P = 8 pairs per unit (16-byte vectors) halves the units of P = 4
    const long long units = wide ? (units4 + 1) / 2 : units4;
    long long grid = (units + ROPE_THREADS - 1) / ROPE_THREADS;
    if (grid > 4LL * sms) grid = 4LL * sms;
    if (grid < 1) grid = 1;
    const size_t smem = FUSED ? (2 * (size_t)p.B + 1) * sizeof(int) : 0;
    // 32-bit unit indices when every unit (plus one grid stride) fits
    const bool narrow = units4 + grid * ROPE_THREADS < INT32_MAX;
    const int which = (bf16 ? 4 : 0) + (narrow ? 2 : 0) + (wide ? 1 : 0);
    using K = void (*)(RopeParams);
    static const K kernels[8] = {
        rope_kernel<false, FUSED, long long, 4>, rope_kernel<false, FUSED, long long, 8>,
        rope_kernel<false, FUSED, int, 4>,       rope_kernel<false, FUSED, int, 8>,
        rope_kernel<true, FUSED, long long, 4>,  rope_kernel<true, FUSED, long long, 8>,
        rope_kernel<true, FUSED, int, 4>,        rope_kernel<true, FUSED, int, 8>};
    if (FUSED) {
        static std::atomic<unsigned long long> configured[8] = {};
        const cudaError_t e = once_per_device(configured[which], [which] {
            return cudaFuncSetAttribute(kernels[which], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (2 * ROPE_MAX_B + 1) * (int)sizeof(int));
        });
        if (e != cudaSuccess) return RGA_ERR_CUDA;
    }
    kernels[which]<<<(int)grid, ROPE_THREADS, smem, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? RGA_OK : RGA_ERR_CUDA;
}

}  // namespace rga

extern "C" rga_status rga_rope_apply(const rga_rope_args *r, cudaStream_t stream) {
    using namespace rga;
    const rga_status st = check_rope(r, true);
    if (st != RGA_OK) return st;
    RopeParams p = {};
    p.q = static_cast<uint16_t *>(r->q);
    p.k = static_cast<uint16_t *>(r->k);
    p.T = r->tokens;
    p.Hq = r->q_heads;
    p.Hk = r->kv_heads;
    p.D = r->head_dim;
    p.R = r->rotary_dim;
    p.cs = r->cos_sin;
    p.pos = r->positions;
    const long long units = (long long)p.T * ((p.q ? p.Hq : 0) + (p.k ? p.Hk : 0)) * (p.R / 8);
    const bool wide = p.R % 16 == 0 && p.D % 8 == 0 && (!p.q || aligned(p.q, 16)) &&
                      (!p.k || aligned(p.k, 16));
    return rope_launch<false>(p, r->dtype == RGA_BF16, wide, units, stream);
}

extern "C" rga_status trt_kv_cache_update_rope(const rga_kv_update_args *kv,
                                                const rga_rope_args *r, cudaStream_t stream) {
    using namespace rga;
    const rga_status st = check_rope(r, false);
    if (st != RGA_OK) return st;
    if (!kv || !kv->past_cache || !kv->update || !kv->y || !kv->device_status)
        return RGA_ERR_INVALID_ARG;
    if (kv->dtype != r->dtype || kv->update_form != RGA_FORM_PACKED_NHD || !kv->update_lengths ||
        kv->y != kv->past_cache)
        return RGA_ERR_INVALID_ARG;
    if (kv->batch < 0 || kv->heads <= 0 || kv->cache_seq < 0 || kv->heads != r->kv_heads ||
        kv->head_dim != r->head_dim || kv->update_seq != r->tokens)
        return RGA_ERR_INVALID_ARG;
    if (!aligned(kv->past_cache, 8) || !aligned(kv->update, 8)) return RGA_ERR_INVALID_ARG;
    if (kv->batch > ROPE_MAX_B) return RGA_ERR_UNSUPPORTED;
    if (kv->batch == 0) {   // no key to write: only Q, if any
        if (!r->q) return RGA_OK;
        rga_rope_args q_only = *r;
        q_only.k = nullptr;
        return rga_rope_apply(&q_only, stream);
    }
    RopeParams p = {};
    p.q = static_cast<uint16_t *>(r->q);
    p.T = r->tokens;
    p.Hq = r->q_heads;
    p.Hk = kv->heads;
    p.D = r->head_dim;
    p.R = r->rotary_dim;
    p.cs = r->cos_sin;
    p.pos = r->positions;
    p.upd = static_cast<const uint16_t *>(kv->update);
    p.cache = static_cast<uint16_t *>(kv->y);
    p.B = kv->batch;
    p.N = kv->cache_seq;
    p.wi = kv->write_indices;
    p.cu = kv->update_lengths;
    p.status = kv->device_status;
    const long long units = (long long)p.T * ((p.q ? p.Hq : 0) * (p.R / 8) +
                                             p.Hk * (p.R / 8 + (p.D - p.R) / 4));
    const bool wide = p.R % 16 == 0 && p.D % 8 == 0 && (!p.q || aligned(p.q, 16)) &&
                      aligned(p.upd, 16) && aligned(p.cache, 16);
    return rope_launch<true>(p, r->dtype == RGA_BF16, wide, units, stream);
}
