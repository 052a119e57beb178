// api.cu - the C ABI (include/rga.h): argument validation, workspace sizing,
// TMA descriptor set-up and dispatch to the scheduler, prefill and decode
// kernels.  No allocation, no synchronisation: everything is enqueued on
// the caller's stream.
#include <cmath>
#include <cstring>
#include <cudaTypedefs.h>
#include "rga.h"
#include "kernels.h"

using namespace rga;

namespace rga {
// SMs of the current device (0 when it cannot be read).
int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}
}  // namespace rga

namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Tiled TMA descriptor over a row-major tensor whose innermost dim is D:
// 16-bit elements with a 64-element inner box by default, or bytes (esize
// 1, fp8 codes) with a D-byte inner box; `swizzle` as the box's row size
// allows (128-byte rows: 128B, 64-byte rows: 64B).
bool encode(CUtensorMap *m, const void *base, int rank, const uint64_t *dims,
            const uint32_t *box, int esize = 2,
            CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    auto fn = get_encode();
    if (!fn) return false;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bd[5], es[5];
    uint64_t stride = (uint64_t)esize;
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i] < 1 ? 1 : dims[i];
        bd[i] = box[i];
        es[i] = 1;
        if (i > 0) gs[i - 1] = stride;
        stride *= gd[i];
    }
    return fn(m, esize == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16,
              rank, const_cast<void *>(base), gd, gs, bd, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q (and Y, same shape): one query tile is G heads x TQ tokens per box.
bool encode_q(CUtensorMap *m, const void *base, const AttnParams &p) {
    if (p.q_packed) {
        const uint64_t d[3] = {(uint64_t)p.D, (uint64_t)p.Hq, (uint64_t)p.q_seq};
        const uint32_t b[3] = {64, (uint32_t)p.G, (uint32_t)p.tq};
        return encode(m, base, 3, d, b);
    }
    const uint64_t d[4] = {(uint64_t)p.D, (uint64_t)p.q_seq, (uint64_t)p.Hq, (uint64_t)p.B};
    const uint32_t b[4] = {64, (uint32_t)p.tq, (uint32_t)p.G, 1};
    return encode(m, base, 4, d, b);
}

bool encode_kv(CUtensorMap *m, const void *base, const AttnParams &p, uint32_t rows) {
    if (p.kv_packed) {
        const uint64_t d[3] = {(uint64_t)p.D, (uint64_t)p.Hkv, (uint64_t)p.kv_seq};
        const uint32_t b[3] = {64, 1, rows};
        return encode(m, base, 3, d, b);
    }
    const uint64_t d[4] = {(uint64_t)p.D, (uint64_t)p.kv_seq, (uint64_t)p.Hkv, (uint64_t)p.B};
    const uint32_t b[4] = {64, rows, 1, 1};
    return encode(m, base, 4, d, b);
}

// fp8 K or V (one byte per element): a box is `rows` whole D-byte rows,
// swizzled as the decode kernel reads them, or unswizzled (`plain`) for the
// prefill kernel's converter warps.
bool encode_kv8(CUtensorMap *m, const void *base, const AttnParams &p, uint32_t rows,
                bool plain = false) {
    const CUtensorMapSwizzle sw = plain ? CU_TENSOR_MAP_SWIZZLE_NONE
                                  : p.D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                               : CU_TENSOR_MAP_SWIZZLE_64B;
    if (p.kv_packed) {
        const uint64_t d[3] = {(uint64_t)p.D, (uint64_t)p.Hkv, (uint64_t)p.kv_seq};
        const uint32_t b[3] = {(uint32_t)p.D, 1, rows};
        return encode(m, base, 3, d, b, 1, sw);
    }
    const uint64_t d[4] = {(uint64_t)p.D, (uint64_t)p.kv_seq, (uint64_t)p.Hkv, (uint64_t)p.B};
    const uint32_t b[4] = {(uint32_t)p.D, rows, 1, 1};
    return encode(m, base, 4, d, b, 1, sw);
}

// Bound on the decode work pairs (batch, KV head, chunk of `rows` query
// rows): ceil(q_seq*G/rows) chunks per batch for padded Q, and at most
// B + q_seq*G/rows chunks over all batches for packed Q.
static int64_t dec_max_pairs(int64_t B, int64_t Hkv, int64_t G, int64_t q_seq, bool packed,
                             int64_t rows) {
    const int64_t per = (q_seq * G + rows - 1) / rows;
    const int64_t chunks = packed ? B + per : B * per;
    return Hkv * chunks;
}

// Decode (split-KV) path: short query rows per (batch, KV head) -- one
// token each in vanilla decoding, a few draft tokens in tree decoding (at
// most 8 per sequence on average for packed Q; the decode kernel streams the
// keys once per chunk of 16 query rows, or of 8 for an fp8 cache and where a
// KV head has at most 8) -- no Q/DQ, and
// every key tile of the work countable in 32 bits.  (Tree decoding with 64
// rows per (batch, KV head) measured slower on the prefill kernel: it has no
// split over the keys, so the longest cache sets its time.)
bool use_decode(const rga_attention_args *a, bool quant, bool kv8 = false) {
    (void)kv8;   // both caches take the same shapes
    if (quant || a->batch > DEC_MAX_B) return false;
    const int G = a->q_heads / a->kv_heads;
    if (G > DEC_MAX_ROWS) return false;
    const bool packed = a->q_form == RGA_FORM_PACKED_NHD;
    if (packed ? a->q_seq > 8 * (int64_t)a->batch : (int64_t)a->q_seq * G > DEC_MAX_ROWS)
        return false;
    const int64_t tiles = dec_max_pairs(a->batch, a->kv_heads, G, a->q_seq, packed, DEC_ROWS_KV8) *
                          (((int64_t)a->kv_seq + DEC_KEYS - 1) / DEC_KEYS);
    return tiles < (int64_t(1) << 31);
}

// paged: K/V from page pools, whose kv_seq is a capacity rather than the
// extent of a padded cache: a mask's key dimension is then checked against
// every sequence's length on the device, as for packed KV.
rga_status validate(const rga_attention_args *a, bool quant, bool paged = false) {
    if (!a) return RGA_ERR_INVALID_ARG;
    if (a->dtype != RGA_F16 && a->dtype != RGA_BF16) {
        return a->dtype == RGA_F32 ? RGA_ERR_UNSUPPORTED : RGA_ERR_INVALID_ARG;
    }
    if ((a->q_form != RGA_FORM_PADDED_BHND && a->q_form != RGA_FORM_PACKED_NHD) ||
        (a->kv_form != RGA_FORM_PADDED_BHND && a->kv_form != RGA_FORM_PACKED_NHD))
        return RGA_ERR_INVALID_ARG;
    if (a->batch < 0 || a->q_heads <= 0 || a->kv_heads <= 0 || a->head_dim <= 0 ||
        a->q_seq < 0 || a->kv_seq < 0)
        return RGA_ERR_INVALID_ARG;
    if (a->q_heads % a->kv_heads != 0) return RGA_ERR_INVALID_ARG;
    if (a->causal < RGA_CAUSAL_NONE || a->causal > RGA_CAUSAL_LOWER_RIGHT) return RGA_ERR_INVALID_ARG;
    if (a->norm != RGA_NORM_SOFTMAX && a->norm != RGA_NORM_NONE) return RGA_ERR_INVALID_ARG;
    if (a->nb_rank != 1) return a->nb_rank < 1 ? RGA_ERR_INVALID_ARG : RGA_ERR_UNSUPPORTED;
    if (a->head_dim != 64 && a->head_dim != 128) return RGA_ERR_UNSUPPORTED;
    if (a->q_heads / a->kv_heads > 128) return RGA_ERR_UNSUPPORTED;
    if (a->q_form == RGA_FORM_PACKED_NHD && !a->query_lengths) return RGA_ERR_INVALID_ARG;
    if (a->kv_form == RGA_FORM_PACKED_NHD && !a->kv_lengths) return RGA_ERR_INVALID_ARG;
    if (!a->device_status) return RGA_ERR_INVALID_ARG;
    if (!std::isfinite(a->scale)) return RGA_ERR_INVALID_ARG;
    const bool any_q = a->batch > 0 && a->q_seq > 0;
    if (any_q && (!a->q || !a->y)) return RGA_ERR_INVALID_ARG;
    if (any_q && a->kv_seq > 0 && (!a->k || !a->v)) return RGA_ERR_INVALID_ARG;
    if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->y))
        return RGA_ERR_INVALID_ARG;
    if (a->mask) {
        if (!quant && a->causal != RGA_CAUSAL_NONE) return RGA_ERR_INVALID_ARG;
        if (a->mask_dtype != RGA_BOOL && a->mask_dtype != RGA_F16 && a->mask_dtype != RGA_BF16 &&
            a->mask_dtype != RGA_F32)
            return RGA_ERR_INVALID_ARG;
        if (a->mask_rank < 0 || a->mask_rank > 4) return RGA_ERR_INVALID_ARG;
        int64_t md[4] = {1, 1, 1, 1};
        for (int i = 0; i < a->mask_rank; ++i) {
            if (a->mask_dims[i] < 1) return RGA_ERR_INVALID_ARG;
            md[4 - a->mask_rank + i] = a->mask_dims[i];
        }
        if (md[0] != 1 && md[0] != a->batch) return RGA_ERR_INVALID_ARG;
        if (md[1] != 1 && md[1] != a->q_heads) return RGA_ERR_INVALID_ARG;
        if (a->q_form == RGA_FORM_PADDED_BHND && md[2] != 1 && md[2] != a->q_seq)
            return RGA_ERR_INVALID_ARG;
        if (a->kv_form == RGA_FORM_PADDED_BHND && !paged && md[3] != 1 && md[3] != a->kv_seq)
            return RGA_ERR_INVALID_ARG;
    }
    return RGA_OK;
}

// kv8: the fp8 KV cache decode layout (DEC_ROWS_KV8 rows per pair).
AttnParams make_params(const rga_attention_args *a, bool quant, bool kv8 = false) {
    AttnParams p;
    std::memset(&p, 0, sizeof(p));
    p.q = a->q; p.k = a->k; p.v = a->v; p.y = a->y;
    p.q_packed = a->q_form == RGA_FORM_PACKED_NHD;
    p.kv_packed = a->kv_form == RGA_FORM_PACKED_NHD;
    p.B = a->batch; p.Hq = a->q_heads; p.Hkv = a->kv_heads; p.D = a->head_dim;
    p.G = a->q_heads / a->kv_heads;
    p.q_seq = a->q_seq; p.kv_seq = a->kv_seq;
    p.query_lengths = a->query_lengths;
    p.kv_lengths = a->kv_form == RGA_FORM_PACKED_NHD || a->kv_lengths ? a->kv_lengths : nullptr;
    p.mask = a->mask;
    p.mask_dtype = a->mask_dtype;
    for (int i = 0; i < 4; ++i) p.md[i] = 1;
    if (a->mask)
        for (int i = 0; i < a->mask_rank; ++i) p.md[4 - a->mask_rank + i] = a->mask_dims[i];
    p.scale = a->scale;
    p.scale_log2 = (float)((double)a->scale * 1.4426950408889634);
    p.causal = a->causal;
    p.quant = -1;
    p.tq = BM / p.G;
    p.item_tokens = 2 * p.tq;
    const int it = p.item_tokens;
    if (p.q_packed)
        p.max_items = p.Hkv * ((p.q_seq + it - 1) / it + p.B);
    else
        p.max_items = p.Hkv * p.B * ((p.q_seq + it - 1) / it);
    // rows per decode pair: 8 for the fp8 tile; the 16-bit tile takes 16 (two
    // N-blocks sharing every K/V fragment) where a (batch, KV head) holds
    // more than 8 query rows on average (q_seq is per batch for padded Q,
    // the total for packed Q)
    const int64_t qrows = (int64_t)p.q_seq * p.G;
    const bool wide = p.q_packed ? qrows > 8LL * p.B : qrows > 8;
    p.dec_rows = kv8 ? DEC_ROWS_KV8 : (wide ? DEC_ROWS_WIDE : DEC_ROWS);
    p.max_pairs = (int)dec_max_pairs(p.B, p.Hkv, p.G, p.q_seq, p.q_packed != 0, p.dec_rows);
    p.dec_slots = 2 * DEC_WARPS_MAX * (sm_count() > 0 ? sm_count() : 1);
    p.status = a->device_status;
    p.ws = static_cast<uint8_t *>(a->workspace);
    (void)quant;
    return p;
}

// (covers both decode layouts: 16-bit and fp8 KV caches)
size_t workspace_bytes(const rga_attention_args *a, bool quant) {
    AttnParams p = make_params(a, quant);
    size_t n = align256(pf_ws_bytes(p));
    for (int kv8 = 0; kv8 < 2; ++kv8) {
        if (!use_decode(a, quant, kv8 != 0)) continue;
        const size_t d = align256(dec_ws_bytes(make_params(a, quant, kv8 != 0)));
        if (d > n) n = d;
    }
    return n;
}

// kv8: K and V are E4M3 codes dequantised with *k_scale / *v_scale (the
// fp8 KV cache; decode shapes only).
// paged: K and V come from page pools (a->k / a->v point at the pools).
rga_status run(const rga_attention_args *a, bool quant, rga_quant qtype, const void *qscale,
               rga_dtype qscale_dtype, cudaStream_t stream, bool kv8 = false,
               const float *k_scale = nullptr, const float *v_scale = nullptr,
               const rga_paged_kv *paged = nullptr) {
    rga_status st = validate(a, quant, paged != nullptr);
    if (st != RGA_OK) return st;
    if (kv8 && (!k_scale || !v_scale)) return RGA_ERR_INVALID_ARG;
    // (an FP8 or paged cache serves the unquantized op: decode shapes on the
    // split-KV kernel, any other shape on the prefill kernel)
    if ((kv8 || paged) && quant) return RGA_ERR_UNSUPPORTED;
    if (quant) {
        if (qtype != RGA_QUANT_FP8_E4M3 && qtype != RGA_QUANT_INT8) return RGA_ERR_INVALID_ARG;
        if (!qscale) return RGA_ERR_INVALID_ARG;
        if (qscale_dtype != RGA_F32 && qscale_dtype != RGA_F16 && qscale_dtype != RGA_BF16)
            return RGA_ERR_INVALID_ARG;
    }
    if (a->batch == 0 || a->q_seq == 0) return RGA_OK;   // no query rows: nothing to write
    const size_t need = workspace_bytes(a, false) > workspace_bytes(a, quant)
                            ? workspace_bytes(a, false) : workspace_bytes(a, quant);
    if (!a->workspace || a->workspace_bytes < need ||
        (reinterpret_cast<uintptr_t>(a->workspace) & 255))
        return RGA_ERR_WORKSPACE;

    AttnParams p = make_params(a, quant, kv8);
    if (quant) {
        p.quant = qtype == RGA_QUANT_FP8_E4M3 ? 0 : 1;
        p.qscale = qscale;
        p.qscale_dtype = qscale_dtype;
    }
    p.kv8 = kv8;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    if (paged) {
        p.paged = 1;
        p.page_table = paged->page_table;
        p.page_size = paged->page_size;
        p.max_pages = paged->max_pages_per_seq;
        p.num_pages = paged->num_pages;
    }
    const int bf16 = a->dtype == RGA_BF16;
    // Zero-extent K/V (no keys anywhere): the descriptors are never read,
    // so they point at Y, which is a valid address.
    const void *kp = a->kv_seq > 0 ? a->k : a->y;
    const void *vp = a->kv_seq > 0 ? a->v : a->y;
    const bool dec = use_decode(a, quant, kv8);
    TensorMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    if (!encode_q(&maps.q, p.q, p) || !encode_q(&maps.y, p.y, p))
        return RGA_ERR_CUDA;
    // a paged pool has the padded layout with pages for batches and a page's
    // keys for the sequence: [num_pages, Hkv, page_size, D]
    AttnParams pm = p;
    if (paged) {
        pm.kv_packed = 0;
        pm.B = paged->num_pages;
        pm.kv_seq = paged->page_size;
    }
    // key rows per box: decode tiles of DEC_KEYS; prefill tiles of BN, as
    // boxes of pf_page_rows() rows (each inside one page) for a paged cache
    const uint32_t rows = dec ? DEC_KEYS : paged ? pf_page_rows(paged->page_size) : BN;
    if (kv8 ? !encode_kv8(&maps.k, kp, pm, rows, !dec) || !encode_kv8(&maps.v, vp, pm, rows, !dec)
            : !encode_kv(&maps.k, kp, pm, rows) || !encode_kv(&maps.v, vp, pm, rows))
        return RGA_ERR_CUDA;
    int mode;
    if (a->norm == RGA_NORM_SOFTMAX) mode = quant ? MODE_SOFTMAX_Q : MODE_SOFTMAX;
    else mode = quant ? MODE_NONE_Q : MODE_NONE;

    cudaError_t e;
    if (!dec && launch_sched(p, 0, stream) != cudaSuccess) return RGA_ERR_CUDA;
    if (dec) {
        const int sms = sm_count();
        if (sms <= 0) return RGA_ERR_CUDA;
        p.grid = sms;
        e = launch_decode(p, maps, mode, stream, bf16, kv8);
    } else {
        int grid = sm_count();
        if (grid <= 0) return RGA_ERR_CUDA;
        if (grid > p.max_items) grid = p.max_items;
        if (grid < 1) grid = 1;
        e = launch_prefill(p, maps, mode, grid, stream, bf16, kv8);
    }
    return e == cudaSuccess ? RGA_OK : RGA_ERR_CUDA;
}

}  // namespace

namespace rga {
cudaError_t launch_prefill(const AttnParams &p, const TensorMaps &m, int mode, int grid,
                           cudaStream_t s, int bf16, int kv8) {
    if (kv8)
        return bf16 ? launch_prefill_kv8_typed<true>(p, m, mode, grid, s)
                    : launch_prefill_kv8_typed<false>(p, m, mode, grid, s);
    return bf16 ? launch_prefill_typed<true>(p, m, mode, grid, s)
                : launch_prefill_typed<false>(p, m, mode, grid, s);
}
}  // namespace rga

extern "C" {

size_t rga_attention_workspace_size(const rga_attention_args *args) {
    // (valid for any entry point: the size does not depend on the mask's
    // key extent, which a paged call checks on the device)
    if (validate(args, true) != RGA_OK && validate(args, false) != RGA_OK &&
        validate(args, false, true) != RGA_OK)
        return 0;
    const size_t a = workspace_bytes(args, false), b = workspace_bytes(args, true);
    return a > b ? a : b;
}

rga_status trt_attention(const rga_attention_args *args, cudaStream_t stream) {
    return run(args, false, RGA_QUANT_FP8_E4M3, nullptr, RGA_F32, stream);
}

rga_status trt_quantized_attention(const rga_attention_args *args, rga_quant qtype,
                                   const void *quant_scale, rga_dtype quant_scale_dtype,
                                   cudaStream_t stream) {
    return run(args, true, qtype, quant_scale, quant_scale_dtype, stream);
}

rga_status trt_attention_fp8_kv(const rga_attention_args *args, const float *k_scale,
                                const float *v_scale, cudaStream_t stream) {
    return run(args, false, RGA_QUANT_FP8_E4M3, nullptr, RGA_F32, stream, true, k_scale, v_scale);
}

rga_status trt_attention_paged_kv(const rga_attention_args *args, const rga_paged_kv *kv,
                                  cudaStream_t stream) {
    if (!args || !kv) return RGA_ERR_INVALID_ARG;
    if (!kv->k_pool || !kv->v_pool || !kv->page_table) return RGA_ERR_INVALID_ARG;
    if (kv->num_pages <= 0 || kv->max_pages_per_seq <= 0 || kv->page_size <= 0 ||
        kv->page_size % DEC_KEYS != 0)
        return RGA_ERR_INVALID_ARG;
    if ((int64_t)kv->max_pages_per_seq * kv->page_size > INT32_MAX) return RGA_ERR_UNSUPPORTED;
    if (args->kv_form != RGA_FORM_PADDED_BHND || !args->kv_lengths) return RGA_ERR_INVALID_ARG;
    const bool kv8 = kv->kv_dtype == RGA_FP8_E4M3;
    if (!kv8 && kv->kv_dtype != args->dtype) return RGA_ERR_INVALID_ARG;
    rga_attention_args a = *args;
    a.k = kv->k_pool;
    a.v = kv->v_pool;
    a.kv_seq = kv->max_pages_per_seq * kv->page_size;
    return run(&a, false, RGA_QUANT_FP8_E4M3, nullptr, RGA_F32, stream, kv8,
               kv8 ? kv->k_scale : nullptr, kv8 ? kv->v_scale : nullptr, kv);
}

rga_status rga_get_device_status(const int32_t *device_status, cudaStream_t stream,
                                 int32_t *out) {
    if (!device_status || !out) return RGA_ERR_INVALID_ARG;
    if (cudaMemcpyAsync(out, device_status, sizeof(int32_t), cudaMemcpyDeviceToHost, stream) !=
        cudaSuccess)
        return RGA_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return RGA_ERR_CUDA;
    return RGA_OK;
}

const char *rga_status_string(rga_status s) {
    switch (s) {
    case RGA_OK: return "RGA_OK";
    case RGA_ERR_INVALID_ARG: return "RGA_ERR_INVALID_ARG";
    case RGA_ERR_UNSUPPORTED: return "RGA_ERR_UNSUPPORTED";
    case RGA_ERR_CUDA: return "RGA_ERR_CUDA";
    case RGA_ERR_DEVICE_LENGTHS: return "RGA_ERR_DEVICE_LENGTHS";
    case RGA_ERR_TIMEOUT: return "RGA_ERR_TIMEOUT";
    case RGA_ERR_WORKSPACE: return "RGA_ERR_WORKSPACE";
    case RGA_ERR_DEBUG_BOUNDS: return "RGA_ERR_DEBUG_BOUNDS";
    }
    return "RGA_ERR_UNKNOWN";
}

int32_t rga_abi_version(void) { return RGA_ABI_VERSION; }

}  // extern "C"
