// kv_update.cu - TRT_KVCacheUpdate ("TensorRT Custom Operator Schemas",
// TRT_KVCacheUpdate): the TensorScatter update of a KV cache [B, H, N, D] in
// "linear" mode along axis -2.  Batch b's first len_b update tokens land at
// sequence positions w_b, w_b + 1, ... of every head; everything else of Y
// is past_cache.
//
// HBM-bound copy kernel.  Every CTA first reads the lengths and write
// positions into shared memory and checks all of them, so that a bad call
// writes nothing (status RGA_ERR_DEVICE_LENGTHS); then the grid strides over
// the vectors of the rows it must write:
//   - in place (y == past_cache): the update rows only;
//   - otherwise: every cache row, taken from the update inside the window
//     and from past_cache outside it (one pass, no separate copy).
// Rows move in 16-byte vectors when the row size and every base address
// allow it, else in 4-, 2- or (fp8 codes) 1-byte units.
#include <cuda_runtime.h>
#include <algorithm>
#include <cstdint>
#include "rga.h"
#include "device_common.cuh"
#include "kernels.h"

namespace rga {

constexpr int KVU_THREADS = 256;
constexpr int KVU_UNROLL = 4;   // vectors a lane reads before it writes (packed, in place)
constexpr int KVU_MAX_B = 8192;

struct KvuParams {
    const uint8_t *cache, *update;
    uint8_t *y;
    int B, H, N, D, esize, nu, packed;
    const int32_t *wi, *cu;
    int32_t *status;
    int in_place;
};

// I: the index type of the vector loops (32-bit whenever every index fits,
// which keeps the divisions that map a vector to its row cheap).
template <int V, typename I>
__global__ void __launch_bounds__(KVU_THREADS)
kv_update_kernel(const __grid_constant__ KvuParams p) {
    extern __shared__ int kvu_smem[];
    int *s_cu = kvu_smem;                 // [B + 1] first update token of each batch (cumulative)
    int *s_w = kvu_smem + p.B + 1;        // [B] write position of each batch
    __shared__ int bad;
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    for (int b = threadIdx.x; b <= p.B; b += KVU_THREADS) {
        int c;
        if (p.cu) c = p.cu[b];
        else c = b * p.nu;                          // padded without lengths: all N_u tokens
        s_cu[b] = c;
        if (b < p.B) s_w[b] = p.wi ? p.wi[b] : 0;
    }
    __syncthreads();
    for (int b = threadIdx.x; b < p.B; b += KVU_THREADS) {
        const int len = s_cu[b + 1] - s_cu[b];
        bool ok = len >= 0 && s_w[b] >= 0 && (long long)s_w[b] + len <= p.N;
        if (p.packed) ok = ok && s_cu[b + 1] <= p.nu;
        else ok = ok && len <= p.nu;
        if (b == 0) ok = ok && s_cu[0] == 0;
        if (!ok) atomicOr(&bad, 1);
    }
    __syncthreads();
    if (bad) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_status(p.status, 4);
        return;
    }

    const int64_t row = (int64_t)p.D * p.esize;       // bytes per row
    const I vpr = (I)(row / V);                        // vectors per row
    const I stride = (I)gridDim.x * KVU_THREADS;
    const int64_t cache_bytes = (int64_t)p.B * p.H * p.N * row;
    const int64_t upd_bytes = p.packed ? (int64_t)s_cu[p.B] * p.H * row
                                       : (int64_t)p.B * p.H * p.nu * row;
    auto copy = [&](const uint8_t *src, uint8_t *dst) {
        // debug-checks builds: the destination lies in the cache, the source
        // in the update tensor or the cache
        const int64_t di = dst - p.y;
        const bool src_ok = (src >= p.update && src - p.update + V <= upd_bytes) ||
                            (p.cache && src >= p.cache && src - p.cache + V <= cache_bytes);
        if (!dbg_ok(di >= 0 && di + V <= cache_bytes && src_ok, p.status)) return;
        if constexpr (V == 16) *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
        else if constexpr (V == 4) *reinterpret_cast<uint32_t *>(dst) = *reinterpret_cast<const uint32_t *>(src);
        else if constexpr (V == 2) *reinterpret_cast<uint16_t *>(dst) = *reinterpret_cast<const uint16_t *>(src);
        else *dst = *src;
    };
    // byte offset of update token t of batch b, head h
    auto upd_row = [&](int b, int h, int t) -> int64_t {
        return p.packed ? ((int64_t)(s_cu[b] + t) * p.H + h) * row
                        : (((int64_t)b * p.H + h) * p.nu + t) * row;
    };
    auto cache_row = [&](int b, int h, int n) -> int64_t {
        return (((int64_t)b * p.H + h) * p.N + n) * row;
    };

    if (p.in_place) {
        if (p.packed) {
            // one warp per update token: its H rows are one contiguous block
            // of the update tensor; the token's batch is found once, and the
            // lane's vectors are read before any is written (KVU_UNROLL at a
            // time), so their loads overlap
            const int lane = threadIdx.x & 31;
            const int wpb = KVU_THREADS / 32;
            const int per = p.H * (int)vpr;   // vectors of one token
            for (int tg = (int)blockIdx.x * wpb + (threadIdx.x >> 5); tg < s_cu[p.B];
                 tg += (int)gridDim.x * wpb) {
                int lo = 0, hi = p.B;   // s_cu[lo] <= tg < s_cu[lo + 1]
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if (s_cu[mid] <= tg) lo = mid; else hi = mid;
                }
                const int n = s_w[lo] + (tg - s_cu[lo]);
                const uint8_t *src = p.update + (int64_t)tg * p.H * row;
                for (int v0 = lane; v0 < per; v0 += 32 * KVU_UNROLL) {
                    uint4 buf[KVU_UNROLL];
                    const uint8_t *sp[KVU_UNROLL];
                    uint8_t *dp[KVU_UNROLL];
#pragma unroll
                    for (int k = 0; k < KVU_UNROLL; ++k) {
                        const int v = v0 + 32 * k;
                        const int h = v / (int)vpr, c = v - h * (int)vpr;
                        sp[k] = v < per ? src + (int64_t)v * V : nullptr;
                        dp[k] = v < per ? p.y + cache_row(lo, h, n) + (int64_t)c * V : nullptr;
                        if constexpr (V == 16)
                            if (sp[k]) buf[k] = *reinterpret_cast<const uint4 *>(sp[k]);
                    }
#pragma unroll
                    for (int k = 0; k < KVU_UNROLL; ++k) {
                        if (!sp[k]) continue;
                        if constexpr (V == 16) {
                            const int64_t di = dp[k] - p.y;
                            if (dbg_ok(di >= 0 && di + V <= cache_bytes &&
                                       sp[k] - p.update + V <= upd_bytes, p.status))
                                *reinterpret_cast<uint4 *>(dp[k]) = buf[k];
                        } else {
                            copy(sp[k], dp[k]);
                        }
                    }
                }
            }
        } else {
            const I total = (I)p.B * p.H * p.nu * vpr;
            for (I v = (I)blockIdx.x * KVU_THREADS + threadIdx.x; v < total; v += stride) {
                const I r = v / vpr, c = v % vpr;
                const int t = (int)(r % p.nu), h = (int)((r / p.nu) % p.H), b = (int)(r / ((I)p.nu * p.H));
                if (t >= s_cu[b + 1] - s_cu[b]) continue;
                copy(p.update + upd_row(b, h, t) + (int64_t)c * V,
                     p.y + cache_row(b, h, s_w[b] + t) + (int64_t)c * V);
            }
        }
    } else {
        const I total = (I)p.B * p.H * p.N * vpr;
        for (I v = (I)blockIdx.x * KVU_THREADS + threadIdx.x; v < total; v += stride) {
            const I r = v / vpr, c = v % vpr;
            const int n = (int)(r % p.N), h = (int)((r / p.N) % p.H), b = (int)(r / ((I)p.N * p.H));
            const int t = n - s_w[b];
            const bool from_update = t >= 0 && t < s_cu[b + 1] - s_cu[b];
            const uint8_t *src = from_update ? p.update + upd_row(b, h, t) : p.cache + cache_row(b, h, n);
            copy(src + (int64_t)c * V, p.y + cache_row(b, h, n) + (int64_t)c * V);
        }
    }
}


template <int V, typename I>
static cudaError_t kvu_launch_i(const KvuParams &p, int grid, cudaStream_t s) {
    const size_t smem = (2 * (size_t)p.B + 1) * sizeof(int);
    static std::atomic<unsigned long long> configured{0};
    cudaError_t e = once_per_device(configured, [] {
        return cudaFuncSetAttribute(kv_update_kernel<V, I>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (2 * KVU_MAX_B + 1) * (int)sizeof(int));
    });
    if (e != cudaSuccess) return e;
    kv_update_kernel<V, I><<<grid, KVU_THREADS, smem, s>>>(p);
    return cudaGetLastError();
}

// 32-bit indices when the largest vector loop (plus one grid stride) fits.
template <int V>
static cudaError_t kvu_launch(const KvuParams &p, int grid, cudaStream_t s) {
    const int64_t vpr = (int64_t)p.D * p.esize / V;
    const int64_t rows = std::max<int64_t>(
        (int64_t)p.B * p.H * (p.in_place ? (int64_t)p.nu : (int64_t)p.N), (int64_t)p.nu * p.H);
    const int64_t span = rows * vpr + (int64_t)grid * KVU_THREADS;
    if (span < INT32_MAX) return kvu_launch_i<V, uint32_t>(p, grid, s);
    return kvu_launch_i<V, int64_t>(p, grid, s);
}

}  // namespace rga

extern "C" rga_status trt_kv_cache_update(const rga_kv_update_args *a, cudaStream_t stream) {
    using namespace rga;
    if (!a || !a->past_cache || !a->update || !a->y || !a->device_status) return RGA_ERR_INVALID_ARG;
    int esize;
    switch (a->dtype) {
    case RGA_F16: case RGA_BF16: esize = 2; break;
    case RGA_F32: esize = 4; break;
    case RGA_FP8_E4M3: esize = 1; break;
    default: return RGA_ERR_INVALID_ARG;
    }
    if (a->update_form != RGA_FORM_PADDED_BHND && a->update_form != RGA_FORM_PACKED_NHD)
        return RGA_ERR_INVALID_ARG;
    if (a->batch < 0 || a->heads <= 0 || a->cache_seq < 0 || a->head_dim <= 0 || a->update_seq < 0)
        return RGA_ERR_INVALID_ARG;
    const bool packed = a->update_form == RGA_FORM_PACKED_NHD;
    if (packed && !a->update_lengths) return RGA_ERR_INVALID_ARG;
    if (a->batch > KVU_MAX_B) return RGA_ERR_UNSUPPORTED;
    // implicit cumulative offsets (padded without lengths) must fit in 32 bits
    if (!packed && !a->update_lengths && (int64_t)a->batch * a->update_seq > INT32_MAX)
        return RGA_ERR_UNSUPPORTED;
    const bool in_place = a->y == a->past_cache;
    if (a->batch == 0 || (in_place && a->update_seq == 0)) return RGA_OK;   // nothing to move

    KvuParams p;
    p.cache = static_cast<const uint8_t *>(a->past_cache);
    p.update = static_cast<const uint8_t *>(a->update);
    p.y = static_cast<uint8_t *>(a->y);
    p.B = a->batch;
    p.H = a->heads;
    p.N = a->cache_seq;
    p.D = a->head_dim;
    p.esize = esize;
    p.nu = a->update_seq;
    p.packed = packed;
    p.wi = a->write_indices;
    p.cu = a->update_lengths;
    p.status = a->device_status;
    p.in_place = in_place;

    const int64_t row = (int64_t)p.D * esize;
    auto aligned = [&](int v) {
        return row % v == 0 && reinterpret_cast<uintptr_t>(p.cache) % v == 0 &&
               reinterpret_cast<uintptr_t>(p.update) % v == 0 &&
               reinterpret_cast<uintptr_t>(p.y) % v == 0;
    };
    const int sms = sm_count();
    if (sms <= 0) return RGA_ERR_CUDA;
    const int grid = 4 * sms;
    cudaError_t e;
    if (aligned(16)) e = kvu_launch<16>(p, grid, stream);
    else if (aligned(4)) e = kvu_launch<4>(p, grid, stream);
    else if (aligned(2)) e = kvu_launch<2>(p, grid, stream);
    else if (esize == 1) e = kvu_launch<1>(p, grid, stream);
    else return RGA_ERR_INVALID_ARG;   // 16-bit element storage not 2-byte aligned
    return e == cudaSuccess ? RGA_OK : RGA_ERR_CUDA;
}
