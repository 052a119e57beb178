// rope.cu - rotary position embedding ("TensorRT Plugins Guide",
// AttentionPlugin: rotary positional encoding; RopeCosSin rows aligned with
// the physical token rows, position -1 marking padding rows), in place on
// Q/K rows, and fused with the KV cache update of the new keys
// ("TensorRT Custom Operator Schemas", TRT_KVCacheUpdate, packed form).
//
// Row t, head h, pair i < R/2 (R = rotary_dim) with c, s from row t of the
// cos/sin table:  x'[i] = x[i] c - x[i + R/2] s,  x'[i + R/2] = x[i + R/2] c
// + x[i] s.  HBM-bound elementwise work: one unit is four consecutive pairs
// of one (row, head) (8-byte loads of each half, 16-byte loads of the
// cosines and sines); in the fused form a unit of the new keys writes its
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

template <bool BF16>
__device__ __forceinline__ void unpack4(uint2 w, float (&x)[4]) {
    const uint32_t u[2] = {w.x, w.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
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

template <bool BF16>
__device__ __forceinline__ uint2 pack4(const float (&x)[4]) {
    uint32_t u[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        if constexpr (BF16) {
            __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
            u[i] = *reinterpret_cast<uint32_t *>(&h);
        } else {
            __half2 h = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
            u[i] = *reinterpret_cast<uint32_t *>(&h);
        }
    }
    return make_uint2(u[0], u[1]);
}

// Pairs 4u .. 4u + 3 of one row: src -> dst (may alias), rotated with the
// table row cs, or copied unchanged when !rotate.
template <bool BF16>
__device__ __forceinline__ void rope_group(const uint16_t *src, uint16_t *dst, const float *cs,
                                           int R, int u, bool rotate) {
    const int h = R / 2;
    const uint2 a = *reinterpret_cast<const uint2 *>(src + 4 * u);
    const uint2 b = *reinterpret_cast<const uint2 *>(src + 4 * u + h);
    if (!rotate) {
        *reinterpret_cast<uint2 *>(dst + 4 * u) = a;
        *reinterpret_cast<uint2 *>(dst + 4 * u + h) = b;
        return;
    }
    const float4 c4 = *reinterpret_cast<const float4 *>(cs + 4 * u);
    const float4 s4 = *reinterpret_cast<const float4 *>(cs + h + 4 * u);
    const float c[4] = {c4.x, c4.y, c4.z, c4.w}, s[4] = {s4.x, s4.y, s4.z, s4.w};
    float x[4], y[4], xo[4], yo[4];
    unpack4<BF16>(a, x);
    unpack4<BF16>(b, y);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        xo[e] = fmaf(x[e], c[e], -(y[e] * s[e]));
        yo[e] = fmaf(y[e], c[e], x[e] * s[e]);
    }
    *reinterpret_cast<uint2 *>(dst + 4 * u) = pack4<BF16>(xo);
    *reinterpret_cast<uint2 *>(dst + 4 * u + h) = pack4<BF16>(yo);
}

// I: the index type of the unit loop (32-bit whenever every unit index and
// row offset fits: the divisions that map a unit to its row are then cheap).
template <bool BF16, bool FUSED, typename I>
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
    const int G4 = p.R / 8;                       // rotated 4-pair groups per row
    const int CG = FUSED ? (p.D - p.R) / 4 : 0;   // copied 4-element groups (fused keys)
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
            if (!dbg_ok(t < p.T && 8 * u + 8 <= p.R, p.status)) continue;
            uint16_t *row = (isq ? p.q : p.k) + (long long)r * p.D;
            rope_group<BF16>(row, row, p.cs + (long long)t * p.R, p.R, u, true);
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
                rope_group<BF16>(src, dst, p.cs + (long long)tg * p.R, p.R, u, rot);
            } else {
                const int d0 = p.R + 4 * (u - G4);
                *reinterpret_cast<uint2 *>(dst + d0) = *reinterpret_cast<const uint2 *>(src + d0);
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
static rga_status rope_launch(const RopeParams &p, bool bf16, long long units, cudaStream_t s) {
    if (units <= 0 && !FUSED) return RGA_OK;
    const int sms = sm_count();
    if (sms <= 0) return RGA_ERR_CUDA;
    long long grid = (units + ROPE_THREADS - 1) / ROPE_THREADS;
    if (grid > 4LL * sms) grid = 4LL * sms;
    if (grid < 1) grid = 1;
    const size_t smem = FUSED ? (2 * (size_t)p.B + 1) * sizeof(int) : 0;
    // 32-bit unit indices when every unit (plus one grid stride) fits
    const bool narrow = units + grid * ROPE_THREADS < INT32_MAX;
    if (FUSED) {
        static std::atomic<unsigned long long> configured[4] = {{0}, {0}, {0}, {0}};
        const cudaError_t e = once_per_device(configured[2 * bf16 + narrow], [bf16, narrow] {
            auto k = bf16 ? (narrow ? rope_kernel<true, true, int> : rope_kernel<true, true, long long>)
                          : (narrow ? rope_kernel<false, true, int> : rope_kernel<false, true, long long>);
            return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (2 * ROPE_MAX_B + 1) * (int)sizeof(int));
        });
        if (e != cudaSuccess) return RGA_ERR_CUDA;
    }
    if (bf16) {
        if (narrow) rope_kernel<true, FUSED, int><<<(int)grid, ROPE_THREADS, smem, s>>>(p);
        else rope_kernel<true, FUSED, long long><<<(int)grid, ROPE_THREADS, smem, s>>>(p);
    } else {
        if (narrow) rope_kernel<false, FUSED, int><<<(int)grid, ROPE_THREADS, smem, s>>>(p);
        else rope_kernel<false, FUSED, long long><<<(int)grid, ROPE_THREADS, smem, s>>>(p);
    }
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
    return rope_launch<false>(p, r->dtype == RGA_BF16, units, stream);
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
    return rope_launch<true>(p, r->dtype == RGA_BF16, units, stream);
}
