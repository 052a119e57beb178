// kernels.h - internal launch parameters shared by the host dispatcher
// (api.cu) and the device kernels.  Not part of the public ABI.
#pragma once
#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime_api.h>

namespace rga {

// Prefill tile geometry: 128 query rows (tokens x heads of one KV group)
// against 128 keys per step.
constexpr int BM = 128;
constexpr int BN = 128;

// Decode geometry: pairs of 8 query rows (the MMA's N of the transposed
// products), or 16 as two N-blocks where a (batch, KV head) holds more than
// 8 rows on average (16-bit cache only), 32 keys per tile, independent
// warps (6 per CTA with 2-stage TMA rings for a 16-bit KV cache, 8 with
// 3-stage rings for an fp8 one, whose tiles take half the bytes); the key
// tiles of all work are split into equal contiguous ranges, one per warp.
constexpr int DEC_MAX_ROWS = 16;    // decode shapes: at most 16 rows per (batch, KV head) on average
constexpr int DEC_ROWS = 8;
constexpr int DEC_ROWS_WIDE = 16;
constexpr int DEC_ROWS_KV8 = 8;
constexpr int DEC_KEYS = 32;
constexpr int DEC_WARPS = 6;
constexpr int DEC_WARPS_KV8 = 8;
constexpr int DEC_WARPS_MAX = 8;
constexpr int DEC_STAGES = 2;
constexpr int DEC_STAGES_KV8 = 3;

enum Mode { MODE_SOFTMAX = 0, MODE_NONE = 1, MODE_SOFTMAX_Q = 2, MODE_NONE_Q = 3 };

struct AttnParams {
    const void *q, *k, *v;
    void *y;
    int q_packed, kv_packed;
    int B, Hq, Hkv, D, G;
    int q_seq, kv_seq;
    const int32_t *query_lengths;   // may be null for padded q
    const int32_t *kv_lengths;      // may be null for padded kv
    const void *mask;               // null = none
    int mask_dtype;                 // rga_dtype
    int64_t md[4];                  // mask dims right-aligned to rank 4
    float scale;                    // natural units
    float scale_log2;               // scale * log2(e)
    int causal;                     // rga_causal
    int quant;                      // -1 off, 0 fp8, 1 int8
    const void *qscale;             // device scalar
    int qscale_dtype;
    int tq;                         // query tokens per prefill tile (BM / G)
    int item_tokens;                // query tokens per prefill work item (2 tiles)
    int max_items;                  // capacity of the work list
    int max_pairs;                  // decode: bound on (batch, KV head, row chunk) pairs
    int dec_slots;                  // decode: partial slots (2 per warp of the grid)
    int dec_rows;                   // decode: query rows per pair (DEC_ROWS, DEC_ROWS_WIDE or DEC_ROWS_KV8)
    int kv8;                        // K, V hold E4M3 codes (fp8 KV cache)
    const float *k_scale, *v_scale; // fp8 KV cache: dequantisation scales (device scalars)
    int paged;                      // K, V come from page pools
    const int32_t *page_table;      // paged: [B, 2, max_pages] K pages, V pages
    int page_size, max_pages, num_pages;
    int grid;                       // decode: persistent grid size
    int32_t *status;                // device status word
    uint8_t *ws;                    // workspace base
};

// Workspace layout (byte offsets from ws).
constexpr size_t WS_HEADER = 256;             // int counters
// Paged decode: each block of the decode prep kernel checks a slice of the
// page table and writes whether it found a page index outside the pools to
// its own header word WS_PAGE_FLAGS + block (no word has two writers).
constexpr int WS_PAGE_FLAGS = 8;
constexpr int DEC_PREP_MAX = 48;              // prep blocks (WS_PAGE_FLAGS + 48 <= 64 words)
// prefill: int4 items[max_items] after the header
// decode: after the prefill region: int tickets[max_pairs] (256-aligned),
// then float partial_o[dec_slots][dec_rows][D], float2 ml[dec_slots][dec_rows]

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// prefill workspace: header + work list
__host__ __device__ inline size_t pf_ws_bytes(const AttnParams &p) {
    return WS_HEADER + (size_t)p.max_items * 16;
}
// decode workspace, after the prefill region: merge tickets (cleared before
// each decode launch), partial O, partial (m, l)
__host__ __device__ inline size_t dec_tickets_off(const AttnParams &p) {
    return align256(pf_ws_bytes(p));
}
__host__ __device__ inline size_t dec_part_off(const AttnParams &p) {
    return align256(dec_tickets_off(p) + ((size_t)p.max_pairs + 1) * 4);
}
__host__ __device__ inline size_t dec_ml_off(const AttnParams &p) {
    return dec_part_off(p) + align256((size_t)p.dec_slots * p.dec_rows * p.D * 4);
}
__host__ __device__ inline size_t dec_ws_bytes(const AttnParams &p) {
    return dec_ml_off(p) + (size_t)p.dec_slots * p.dec_rows * 8;
}
// Blocks of the decode prep kernel (computed the same way by the launcher
// and by the decode kernel, which reads that many page flags).
__host__ __device__ inline int dec_prep_blocks(const AttnParams &p) {
    long long blocks = ((long long)p.max_pairs + 1 + 255) / 256;
    if (p.paged) {
        const long long v = ((long long)p.B * p.max_pages + 2047) / 2048;
        if (v > blocks) blocks = v;
    }
    if (blocks < 1) blocks = 1;
    return (int)(blocks < DEC_PREP_MAX ? blocks : DEC_PREP_MAX);
}

// Rows of one TMA box of a paged cache in the prefill kernel: the largest of
// 128, 64, 32 that divides the page size (a multiple of 32), so that each
// box lies inside one page and a 128-key tile is a whole number of boxes.
__host__ __device__ inline int pf_page_rows(int page_size) {
    return (page_size & 127) == 0 ? 128 : (page_size & 63) == 0 ? 64 : 32;
}

// Largest batch the decode kernel lists in shared memory.
constexpr int DEC_MAX_B = 4096;

struct TensorMaps {
    CUtensorMap q, k, v, y;   // y: same geometry and box as q
};

// Launch a kernel that follows the scheduler on the same stream as a
// programmatic dependent: it may start (and run its prologue) while the
// scheduler finishes, and waits for it with griddepcontrol.wait.
template <typename Kernel>
inline cudaError_t launch_dependent(Kernel kernel, int grid, int block, int smem,
                                    cudaStream_t s, const AttnParams &p, const TensorMaps &m) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p, m);
}

// SMs of the current device (0 when it cannot be read); api.cu.
int sm_count();

// Runs `set` (returning cudaError_t) once per device for the caller's flags
// word: kernel attributes such as the dynamic shared memory limit are set
// per device, so a process that drives several GPUs configures each of
// them.  Idempotent, so two threads racing on the first call is harmless.
template <typename F>
inline cudaError_t once_per_device(std::atomic<unsigned long long> &done, F set) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    const cudaError_t e = set();
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// Launchers (return cudaError_t of the launch).
cudaError_t launch_sched(const AttnParams &p, int decode, cudaStream_t s);
template <bool BF16>
cudaError_t launch_prefill_typed(const AttnParams &p, const TensorMaps &m, int mode, int grid,
                                 cudaStream_t s);
template <bool BF16>
cudaError_t launch_prefill_kv8_typed(const AttnParams &p, const TensorMaps &m, int mode, int grid,
                                     cudaStream_t s);
cudaError_t launch_prefill(const AttnParams &p, const TensorMaps &m, int mode, int grid,
                           cudaStream_t s, int bf16, int kv8);
// Decode over a 16-bit cache with several 16-row chunks per (batch, KV
// head) (tree decoding): warps in groups of four sharing each K/V tile.
cudaError_t launch_decode_group(const AttnParams &p, const TensorMaps &m, int mode,
                                cudaStream_t s, int bf16);
cudaError_t launch_decode(const AttnParams &p, const TensorMaps &m, int mode,
                          cudaStream_t s, int bf16, int kv8);

}  // namespace rga
