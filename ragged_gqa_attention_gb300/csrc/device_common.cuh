// device_common.cuh - per-sequence offsets/lengths, causal limits and mask
// reads, shared by the scheduler, prefill and decode kernels.
#pragma once
#include <climits>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include "kernels.h"

namespace rga {

struct SeqInfo {
    int q_off, q_len, kv_off, kv_len;
};

// Offsets and lengths of batch b from the two length inputs
// ("TensorRT Custom Operator Schemas", TRT_Attention inputs query_lengths
// and kv_lengths): cumulative [B+1] for packed forms, per-batch [B] (or
// absent) for padded KV, optional cumulative for padded Q.
__device__ __forceinline__ SeqInfo seq_info(const AttnParams &p, int b) {
    SeqInfo s;
    const int32_t *ql = p.query_lengths, *kl = p.kv_lengths;
    if (p.q_packed) {
        s.q_off = ql[b];
        s.q_len = ql[b + 1] - ql[b];
    } else {
        s.q_off = 0;
        s.q_len = ql ? ql[b + 1] - ql[b] : p.q_seq;
    }
    if (p.kv_packed) {
        s.kv_off = kl[b];
        s.kv_len = kl[b + 1] - kl[b];
    } else {
        s.kv_off = 0;
        s.kv_len = kl ? kl[b] : p.kv_seq;
    }
    return s;
}

// Largest key index query i may attend under the causal kind (before the
// kv_len bound): upper_left j <= i; lower_right j <= i + kv_len - q_len.
__device__ __forceinline__ int causal_limit(int causal, int i, const SeqInfo &s) {
    if (causal == 1) return i;
    if (causal == 2) return i + s.kv_len - s.q_len;
    return INT_MAX - 1;
}

// Number of keys [0, n) that any query in tokens [i0, i1) may attend.
__device__ __forceinline__ int key_extent(int causal, int i_last, const SeqInfo &s) {
    long long lim = (long long)causal_limit(causal, i_last, s) + 1;
    if (lim > s.kv_len) lim = s.kv_len;
    if (lim < 0) lim = 0;
    return (int)lim;
}

// Record an error code in the status word unless one is already there.
__device__ __forceinline__ void set_status(int32_t *status, int code) {
    atomicCAS(status, 0, code);
}

// Debug-checks builds (RGA_DEBUG_CHECKS): dbg_ok(ok, status) is false when
// an access failed its bounds check, after recording status 7 (the caller
// then skips the access).  Ordinary builds carry no checks: it is true and
// the condition is not evaluated.
#ifdef RGA_DEBUG_CHECKS
constexpr bool RGA_DEBUG = true;
#else
constexpr bool RGA_DEBUG = false;
#endif
constexpr int RGA_STATUS_BOUNDS = 7;
#define dbg_ok(cond, status)                                                   \
    (!::rga::RGA_DEBUG || (cond) ||                                            \
     (::rga::set_status((status), ::rga::RGA_STATUS_BOUNDS), false))

// Elements of the tensors a call reads and writes (for the checks).
__device__ __forceinline__ long long q_elems(const AttnParams &p) {
    return (long long)(p.q_packed ? p.q_seq : (long long)p.B * p.q_seq) * p.Hq * p.D;
}
__device__ __forceinline__ long long mask_elems(const AttnParams &p) {
    return p.md[0] * p.md[1] * p.md[2] * p.md[3];
}

// Flat offset of mask row (b, h, i) under right-aligned broadcast.
__device__ __forceinline__ long long mask_row(const AttnParams &p, int b, int h, int i) {
    long long ib = p.md[0] == 1 ? 0 : b;
    long long ih = p.md[1] == 1 ? 0 : h;
    long long iq = p.md[2] == 1 ? 0 : i;
    return ((ib * p.md[1] + ih) * p.md[2] + iq) * p.md[3];
}

// Read mask element at flat index e: returns whether the pair may attend
// and the additive term (natural units).
__device__ __forceinline__ bool mask_at(const AttnParams &p, long long e, float &add) {
    if (!dbg_ok(e >= 0 && e < mask_elems(p), p.status)) {
        add = 0.f;
        return false;
    }
    switch (p.mask_dtype) {
    case 3:  // bool
        add = 0.f;
        return static_cast<const uint8_t *>(p.mask)[e] != 0;
    case 0:
        add = __half2float(static_cast<const __half *>(p.mask)[e]);
        return true;
    case 1:
        add = __bfloat162float(static_cast<const __nv_bfloat16 *>(p.mask)[e]);
        return true;
    default:
        add = static_cast<const float *>(p.mask)[e];
        return true;
    }
}


// mask_at for a mask type known at compile time (MK: the rga_dtype of the
// mask, 3 bool), for loops that would otherwise carry every type's load.
template <int MK>
__device__ __forceinline__ bool mask_at_t(const AttnParams &p, long long e, float &add) {
    if (!dbg_ok(e >= 0 && e < mask_elems(p), p.status)) {
        add = 0.f;
        return false;
    }
    if constexpr (MK == 3) {
        add = 0.f;
        return static_cast<const uint8_t *>(p.mask)[e] != 0;
    } else if constexpr (MK == 0) {
        add = __half2float(static_cast<const __half *>(p.mask)[e]);
    } else if constexpr (MK == 1) {
        add = __bfloat162float(static_cast<const __nv_bfloat16 *>(p.mask)[e]);
    } else {
        add = static_cast<const float *>(p.mask)[e];
    }
    return true;
}

__device__ __forceinline__ float load_qscale(const AttnParams &p) {
    if (p.qscale_dtype == 0) return __half2float(*static_cast<const __half *>(p.qscale));
    if (p.qscale_dtype == 1)
        return __bfloat162float(*static_cast<const __nv_bfloat16 *>(p.qscale));
    return *static_cast<const float *>(p.qscale);
}

}  // namespace rga
