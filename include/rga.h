/*
 * rga.h - C ABI of the ragged GQA fused attention library (GB300, sm_103a).
 *
 * The operation is the fused attention forward of the TRT_Attention and
 * TRT_QuantizedAttention custom operators ("TensorRT Custom Operator
 * Schemas"), covering the MHA/GQA attention of the AttentionPlugin
 * ("TensorRT Plugins Guide", AttentionPlugin):
 *
 *     Y = softmax(scale * Q K^T + mask) V        (TRT_normalization_op "softmax")
 *     Y = (scale * Q K^T + mask) V  on allowed pairs   ("none")
 *
 * and, for the quantized operator, a quantize/dequantize of the normalised
 * probabilities to fp8 E4M3 or int8 with a given scale before the second
 * batched matmul (BMM2).
 *
 * Conventions shared by every entry point:
 *  - Every tensor pointer is a DEVICE pointer owned by the caller.  The
 *    library never allocates, frees or synchronises; all work is enqueued on
 *    the caller's stream.
 *  - Synchronous argument errors are returned as an rga_status and nothing
 *    is launched.  Errors that depend on device data (the length inputs) are
 *    detected on the device: the affected call writes a non-zero code to
 *    *device_status, enqueues no attention work and leaves Y untouched.
 *    rga_get_device_status reads that word back.
 *  - Padded query rows at or beyond a sequence's query length, and packed
 *    rows beyond the last sequence, are never written.
 */
#ifndef RGA_H
#define RGA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RGA_ABI_VERSION 1

typedef enum {
    RGA_OK = 0,
    RGA_ERR_INVALID_ARG = 1,     /* bad pointer, shape, enum or combination */
    RGA_ERR_UNSUPPORTED = 2,     /* valid per the schema, not implemented here */
    RGA_ERR_CUDA = 3,            /* a CUDA runtime/driver call failed */
    RGA_ERR_DEVICE_LENGTHS = 4,  /* device-side: inconsistent length inputs */
    RGA_ERR_TIMEOUT = 5,         /* device-side: a bounded wait ran out */
    RGA_ERR_WORKSPACE = 6,       /* workspace missing or too small */
    RGA_ERR_DEBUG_BOUNDS = 7     /* device-side, debug-checks builds only: an access
                                    outside its tensor was caught and skipped */
} rga_status;

/* IO forms (TRT_Attention attributes query_form / kv_form):
 *   PADDED_BHND: 4-D [B, H, N, D], row-major;
 *   PACKED_NHD:  3-D [T, H, D], row-major, sequences concatenated along T. */
typedef enum { RGA_FORM_PADDED_BHND = 0, RGA_FORM_PACKED_NHD = 1 } rga_form;

/* causal_kind (TRT_Attention).  For a sequence with q_len query rows and
 * kv_len keys, query i may attend key j when:
 *   NONE:        always;
 *   UPPER_LEFT:  j <= i  (the is_causal of TRT_QuantizedAttention);
 *   LOWER_RIGHT: j <= i + kv_len - q_len. */
typedef enum {
    RGA_CAUSAL_NONE = 0,
    RGA_CAUSAL_UPPER_LEFT = 1,
    RGA_CAUSAL_LOWER_RIGHT = 2
} rga_causal;

/* TRT_normalization_op. */
typedef enum { RGA_NORM_SOFTMAX = 0, RGA_NORM_NONE = 1 } rga_norm;

/* Element types.  Q, K, V and Y share one of F16 / BF16 (K and V are
 * E4M3 codes for trt_attention_fp8_kv).  A mask is BOOL (one byte per
 * element, non-zero = may attend) or additive F16/BF16/F32.  FP8_E4M3: OCP
 * E4M3FN codes, one byte each (an fp8 KV cache). */
typedef enum {
    RGA_F16 = 0, RGA_BF16 = 1, RGA_F32 = 2, RGA_BOOL = 3, RGA_FP8_E4M3 = 4
} rga_dtype;

/* normalization_quantize_to_type (TRT_QuantizedAttention). */
typedef enum { RGA_QUANT_FP8_E4M3 = 0, RGA_QUANT_INT8 = 1 } rga_quant;

/*
 * Arguments of one attention call ("TensorRT Custom Operator Schemas",
 * TRT_Attention: attributes, inputs 0-5 and output Y).
 *
 * q:  padded [B, Hq, q_seq, D] or packed [q_seq, Hq, D]       (input Q)
 * k, v: padded [B, Hkv, kv_seq, D] or packed [kv_seq, Hkv, D] (inputs K, V)
 * y:  same shape, form and dtype as q                          (output Y)
 *
 * query_lengths: int32 [B+1] cumulative, starting at 0.  Required when q is
 *   packed.  Optional when q is padded: then query_lengths[b+1] -
 *   query_lengths[b] (<= q_seq) is the number of valid rows of batch b and
 *   the remaining rows are left untouched; NULL means all q_seq rows.
 * kv_lengths: packed KV: int32 [B+1] cumulative, required.  Padded KV:
 *   int32 [B] per-batch lengths (<= kv_seq), optional (NULL = kv_seq).
 * Rows of K/V at or beyond a sequence's length may hold any bits,
 *   including NaN/Inf; they never reach Y.
 *
 * mask: optional (NULL = none), row-major, rank mask_rank <= 4 with sizes
 *   mask_dims[0..mask_rank-1]; it is right-aligned against the logical
 *   [B, Hq, Nq, Nkv] and each size is 1 (broadcast) or full (B, Hq, or at
 *   least the longest query / key length of the batch).  It is indexed with
 *   within-sequence positions (i, j).  BOOL: true = may attend.  F16, BF16,
 *   F32: added to scale * QK^T.  TRT_Attention rejects a mask together with
 *   a causal kind other than NONE; TRT_QuantizedAttention accepts both (a
 *   pair must then pass both).
 * scale: multiplies QK^T before the additive mask.  TRT_Attention itself
 *   applies no scale (use 1.0); TRT_QuantizedAttention's default is
 *   1/sqrt(D).
 * nb_rank: must be 1 (single-device execution).
 * workspace: device scratch of at least rga_attention_workspace_size(args)
 *   bytes, 256-byte aligned, owned by the caller; its contents on entry do
 *   not matter.  Calls that overlap on the device must not share it.
 * device_status: one int32 on the device, owned by the caller.  A call sets
 *   it to a non-zero rga_status when the device finds bad lengths or a wait
 *   times out; it is never cleared by the library (clear it yourself).
 */
typedef struct {
    const void *q, *k, *v;
    void *y;
    rga_dtype dtype;               /* of q, k, v, y: RGA_F16 or RGA_BF16 */
    rga_form q_form, kv_form;      /* independent of each other */
    int32_t batch, q_heads, kv_heads, head_dim;   /* q_heads % kv_heads == 0 */
    int32_t q_seq;                 /* padded: N_q; packed: rows T_q of q */
    int32_t kv_seq;                /* padded: N_kv; packed: rows T_kv of k, v */
    const int32_t *query_lengths;
    const int32_t *kv_lengths;
    const void *mask;
    rga_dtype mask_dtype;
    int32_t mask_rank;
    int64_t mask_dims[4];
    float scale;
    rga_causal causal;
    rga_norm norm;
    int32_t nb_rank;
    void *workspace;
    size_t workspace_bytes;
    int32_t *device_status;
} rga_attention_args;

/* Bytes of workspace that trt_attention / trt_quantized_attention need for
 * these arguments (a bound computed from the shapes alone; the length
 * inputs are not read).  Returns 0 when the arguments are invalid. */
size_t rga_attention_workspace_size(const rga_attention_args *args);

/* TRT_Attention ("TensorRT Custom Operator Schemas", TRT_Attention).
 * Supported: head_dim 64 or 128; q_heads / kv_heads <= 128.
 * Returns RGA_OK after enqueueing the work on `stream`. */
rga_status trt_attention(const rga_attention_args *args, cudaStream_t stream);

/* TRT_QuantizedAttention ("TensorRT Custom Operator Schemas",
 * TRT_QuantizedAttention).  Same as trt_attention, plus a Q/DQ of the
 * probabilities between normalisation and BMM2: x = p / s, q = saturate(
 * round-half-even(x)) in E4M3FN (max 448) or int8 [-128, 127], p' = q * s.
 * With softmax, p is the fully normalised probability.  quant_scale is a
 * device pointer to one scalar of type quant_scale_dtype (F32, F16 or
 * BF16), required and > 0. */
rga_status trt_quantized_attention(const rga_attention_args *args,
                                   rga_quant qtype, const void *quant_scale,
                                   rga_dtype quant_scale_dtype,
                                   cudaStream_t stream);

/* Attention over an FP8 KV cache ("TensorRT Plugins Guide",
 * AttentionPlugin: kv_cache_type FP8; prefill, chunked prefill, vanilla and
 * tree decoding).  Same as
 * trt_attention, except that args->k and args->v hold OCP E4M3FN codes (one
 * byte per element, same shapes and forms as there) and the keys and values
 * attended are
 *     K[..] = e4m3(code) * (*k_scale),   V[..] = e4m3(code) * (*v_scale)
 * (per-tensor dequantisation; k_scale, v_scale: device pointers to one
 * float each, required).  args->dtype is the type of q and y (F16 or BF16);
 * k and v must be 16-byte aligned.  The codes past a sequence's kv length
 * may hold any bits, NaN codes included.
 * Every shape and option of trt_attention: decode shapes (q_heads /
 * kv_heads <= 16 and either padded q with q_seq * (q_heads / kv_heads) <=
 * 16 or packed q with q_seq <= 8 * batch) run on the split-KV decode
 * kernel, every other shape on the prefill kernel, which expands each tile
 * of codes to 16-bit values in shared memory.  Workspace:
 * rga_attention_workspace_size(args) bytes. */
rga_status trt_attention_fp8_kv(const rga_attention_args *args, const float *k_scale,
                                const float *v_scale, cudaStream_t stream);

/* Paged KV cache ("TensorRT Plugins Guide", AttentionPlugin: the decoder
 * tensor contract's kv_page_table [N, 2, max_pages_per_sequence], a
 * current-entry page-table view into resident paged KV pools).
 *
 * k_pool, v_pool: device pools of num_pages pages, each page
 *   [kv_heads, page_size, head_dim] row-major, so a pool is
 *   [num_pages, kv_heads, page_size, head_dim]; 16-byte aligned.
 * kv_dtype: the pools' element type: args->dtype (F16 / BF16), or
 *   FP8_E4M3 with k_scale / v_scale (device fp32 scalars, required then;
 *   ignored otherwise) as in trt_attention_fp8_kv.
 * page_table: device int32 [batch, 2, max_pages_per_seq]: row 0 of batch b
 *   lists the K pages of its keys in order (key n is row n % page_size of
 *   page page_table[b][0][n / page_size]), row 1 the V pages.  Entries
 *   past a sequence's last page are never read.
 * page_size: keys per page, a positive multiple of 32.
 */
typedef struct {
    const void *k_pool, *v_pool;
    rga_dtype kv_dtype;
    const float *k_scale, *v_scale;
    const int32_t *page_table;
    int32_t num_pages, page_size, max_pages_per_seq;
} rga_paged_kv;

/* Attention over a paged KV cache.  Same as trt_attention (or
 * trt_attention_fp8_kv for an FP8_E4M3 pool), except that the keys and
 * values come from the pools through the page table: args->k and args->v
 * are ignored, args->kv_form must be RGA_FORM_PADDED_BHND, args->kv_lengths
 * (device int32 [batch]) is required, and args->kv_seq is ignored (a
 * sequence may hold up to max_pages_per_seq * page_size keys; a mask's key
 * dimension is 1 or at least every sequence's length, checked on the
 * device).  Every shape, as for trt_attention_fp8_kv (the prefill kernel
 * loads a 128-key tile as boxes of 128, 64 or 32 rows, the largest that
 * divides page_size, each inside one page).  A page index outside
 * [0, num_pages) among a
 * sequence's pages sets *device_status to RGA_ERR_DEVICE_LENGTHS and leaves
 * Y untouched, as bad lengths do.  Workspace: rga_attention_workspace_size
 * of the same args with kv_seq = max_pages_per_seq * page_size. */
rga_status trt_attention_paged_kv(const rga_attention_args *args, const rga_paged_kv *kv,
                                  cudaStream_t stream);

/* Size of the library-owned device scratch used by
 * trt_attention_static_scratch (40 MiB). */
#define RGA_STATIC_SCRATCH_BYTES (40ull << 20)

/* trt_attention without caller-provided scratch, for callers that cannot
 * allocate device memory themselves (a host application that owns every
 * allocation and hands the library only its tensors, or a caller with no
 * allocator at hand).  The pages describe no such call: this entry point
 * has no counterpart there.
 *
 * Same arguments and results as trt_attention, except that args->workspace
 * and args->workspace_bytes are ignored: the scratch is a 40 MiB device
 * array inside the library, held on a GPU from the first call made on it
 * (from context creation when CUDA loads modules eagerly) until the process
 * exits.  Inputs, Y and device_status are still the caller's.  Allocates
 * nothing (no cudaMalloc, no allocating library routine).
 *
 * Returns RGA_ERR_WORKSPACE when rga_attention_workspace_size(args) exceeds
 * RGA_STATIC_SCRATCH_BYTES.  Every call looks up the array's device address
 * in the current context (cudaGetSymbolAddress, with the caller's device
 * current); the first call on a device also loads the array there.  Every
 * call shares the one array: calls that overlap on the device race and give wrong results,
 * so serialise them (one stream, or events).  Each call rewrites all the
 * scratch it reads, so what a previous call left there does not matter. */
rga_status trt_attention_static_scratch(const rga_attention_args *args, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * TRT_KVCacheUpdate ("TensorRT Custom Operator Schemas", TRT_KVCacheUpdate):
 * the TensorScatter update of a KV cache in "linear" mode along axis -2, the
 * step in front of decode attention.  For every batch b, every head h and
 * every update token t < len_b:
 *     Y[b, h, w_b + t, :] = update token t of batch b, head h
 * and every other element of Y equals past_cache.
 *   w_b   = write_indices[b] (device int32 [B]); 0 for every batch when NULL.
 *   len_b = update_lengths[b+1] - update_lengths[b] (device int32 [B+1],
 *           cumulative from 0); required for the packed form, where batch
 *           b's tokens are rows update_lengths[b] .. update_lengths[b+1]-1
 *           of the update; for the padded form, NULL means update_seq
 *           tokens for every batch.
 * past_cache, y: [B, H, N, D] (row-major, N = cache_seq); update: padded
 * [B, H, update_seq, D] or packed [update_seq, H, D].  All device pointers,
 * owned by the caller.  y == past_cache updates the cache in place (only the
 * written rows move); otherwise the whole cache is copied to y with the
 * update applied, and y must not overlap past_cache or update otherwise.
 * The op moves element bits without arithmetic: dtype only sets the element
 * size (RGA_F16, RGA_BF16, RGA_F32, or RGA_FP8_E4M3 for an fp8 cache whose
 * update arrives already encoded).
 * Errors: RGA_ERR_INVALID_ARG for bad pointers, shapes or enums (nothing is
 * enqueued); batch > 8192 gives RGA_ERR_UNSUPPORTED.  On the device, a
 * window [w_b, w_b + len_b) outside [0, N), negative or non-cumulative
 * lengths, or lengths past the update tensor set *device_status to
 * RGA_ERR_DEVICE_LENGTHS and nothing is written.
 * ------------------------------------------------------------------------- */
typedef struct {
    const void *past_cache;
    const void *update;
    void *y;
    rga_dtype dtype;               /* element size only: F16, BF16, F32 or FP8_E4M3 */
    rga_form update_form;
    int32_t batch, heads, cache_seq, head_dim;
    int32_t update_seq;            /* padded: N_u of the update; packed: rows T */
    const int32_t *write_indices;  /* [B] or NULL */
    const int32_t *update_lengths; /* [B+1] cumulative, or NULL (padded only) */
    int32_t *device_status;
} rga_kv_update_args;

/* Enqueue TRT_KVCacheUpdate on `stream`; returns RGA_OK once enqueued. */
rga_status trt_kv_cache_update(const rga_kv_update_args *args, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Rotary position embedding ("TensorRT Plugins Guide", AttentionPlugin:
 * the plugin handles rotary positional encoding; its decoder contract
 * passes RopeCosSin token-aligned with the physical rows, and positions
 * with -1 marking padding rows).  For every row t of the T physical rows
 * whose position is >= 0 (every row when positions is NULL), every head h
 * and every i < R/2 (R = rotary_dim):
 *     c = cos_sin[t * R + i],  s = cos_sin[t * R + R/2 + i]
 *     x'[i]       = x[i] * c - x[i + R/2] * s
 *     x'[i + R/2] = x[i + R/2] * c + x[i] * s
 * (the rotate-half pairing); dims R .. D-1 are unchanged.  Computed in
 * fp32, rounded to the element type (nearest even).  Rows with a negative
 * position are left exactly as they are.
 * ------------------------------------------------------------------------- */
typedef struct {
    void *q;                   /* [T, q_heads, D] rotated in place, or NULL */
    void *k;                   /* [T, kv_heads, D] rotated in place, or NULL */
    rga_dtype dtype;           /* F16 or BF16 */
    int32_t tokens, q_heads, kv_heads, head_dim;
    int32_t rotary_dim;        /* even multiple of 8, <= head_dim */
    const float *cos_sin;      /* [T, rotary_dim]: the R/2 cosines, then the R/2 sines */
    const int32_t *positions;  /* [T] or NULL */
} rga_rope_args;

/* Rotate q and/or k in place (device pointers, 8-byte aligned). */
rga_status rga_rope_apply(const rga_rope_args *rope, cudaStream_t stream);

/* RoPE fused with the KV cache update of the new keys: in one pass, rotate
 * rope->q in place and write the update rows of kv (the new keys, packed
 * form: kv->update is [T, heads, D] with T = rope->tokens) into the cache
 * rotated, exactly as trt_attention would then read them; the update tensor
 * itself is not modified.  kv must be an in-place update (y == past_cache)
 * of the packed form with update_lengths; rope->k is ignored and
 * rope->kv_heads must equal kv->heads.  Row t of the update is rotated with
 * cos_sin row t (and skipped, i.e. written unrotated, when its position is
 * negative).  Errors as for trt_kv_cache_update and rga_rope_apply. */
rga_status trt_kv_cache_update_rope(const rga_kv_update_args *kv, const rga_rope_args *rope,
                                    cudaStream_t stream);

/* Copy *device_status to *out after the work already enqueued on `stream`
 * has finished.  This call synchronises the stream: use it in tests and
 * debugging, not on a hot path. */
rga_status rga_get_device_status(const int32_t *device_status,
                                 cudaStream_t stream, int32_t *out);

/* Failure-path self-test: enqueue one CTA whose single wait (on an mbarrier
 * that nothing arrives on) gives up after `wait_cycles` SM clock cycles
 * (1 .. 2^32) and sets *device_status to RGA_ERR_TIMEOUT, exactly as a
 * timed-out wait in the attention kernels does.  Nothing faults or hangs and
 * the context stays usable; the attention kernels bound every wait at about
 * 2 s of clock cycles the same way.  device_status: one device int32 owned
 * by the caller.  Returns RGA_ERR_INVALID_ARG for a null pointer or a limit
 * out of range. */
rga_status rga_selftest_wait_timeout(int32_t *device_status, int64_t wait_cycles,
                                     cudaStream_t stream);

/* Conversion self-test of the fp8 KV cache path: enqueue one CTA that
 * decodes all 256 E4M3 codes with the in-register conversion of the decode
 * kernel and writes the f16 bits of code c to out_f16[c] and the bf16 bits
 * to out_bf16[c] (device arrays of 256 uint16 each, owned by the caller).
 * Returns RGA_ERR_INVALID_ARG for a null pointer. */
rga_status rga_selftest_e4m3_decode(uint16_t *out_f16, uint16_t *out_bf16, cudaStream_t stream);

/* Self-test of the debug-checks build (librga_debug.so, built with
 * RGA_DEBUG_CHECKS).  Its kernels check every TMA start coordinate against
 * its tensor's extent and every direct global read or write against its
 * buffer; an access outside is skipped and RGA_ERR_DEBUG_BOUNDS written to
 * the device status word (a skipped TMA load still completes its
 * mbarrier's transaction count, so no wait hangs).  This call asks one
 * thread for a store to element `index` of the device int32 buffer `buf` of
 * `n` elements through the same check: with index >= n the store is
 * skipped and *device_status becomes RGA_ERR_DEBUG_BOUNDS; otherwise buf
 * [index] = 1.  Returns RGA_ERR_UNSUPPORTED in the ordinary build, whose
 * kernels carry no checks.  Stream-ordered, no synchronisation. */
rga_status rga_selftest_bounds_check(int32_t *buf, int64_t n, int64_t index,
                                     int32_t *device_status, cudaStream_t stream);

/* Human-readable name of a status code (static storage). */
const char *rga_status_string(rga_status status);

/* ABI version of the loaded library (RGA_ABI_VERSION). */
int32_t rga_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RGA_H */
