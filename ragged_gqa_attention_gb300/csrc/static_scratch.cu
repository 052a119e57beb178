// static_scratch.cu - trt_attention for callers that cannot allocate device
// memory (for example code that runs inside a host that owns every
// allocation, or a plugin that is handed tensors but no allocator).
//
// The scratch that trt_attention normally takes from the caller (the
// scheduler's work list, and for decode the split partials and tickets)
// comes here from one file-scope device array owned by the library.  A GPU
// holds that array from the first call made on it (when CUDA loads modules
// lazily, its default; from context creation when it loads them eagerly)
// until the process exits.
//
// Host code cannot use `g_rga_scratch` as an address: on the host the name
// stands for a host-side shadow, and a kernel given it would fault or, where
// the GPU can reach host memory, quietly use the wrong memory.  Every call
// looks up the device address with cudaGetSymbolAddress, with the caller's
// device current, so the address always belongs to the current context (a
// context re-created after cudaDeviceReset may place the array elsewhere).
// The first call on a device also loads the array's module there.
#include "rga.h"

namespace {

constexpr size_t kScratchBytes = RGA_STATIC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_rga_scratch[kScratchBytes];

// Device address of the scratch array in the current context.
rga_status scratch_address(void **out) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_rga_scratch) != cudaSuccess || !p) return RGA_ERR_CUDA;
    *out = p;
    return RGA_OK;
}

}  // namespace

extern "C" rga_status trt_attention_static_scratch(const rga_attention_args *args,
                                                   cudaStream_t stream) {
    if (!args) return RGA_ERR_INVALID_ARG;
    rga_attention_args a = *args;
    a.workspace = nullptr;
    a.workspace_bytes = 0;
    const size_t need = rga_attention_workspace_size(&a);
    if (need == 0) return trt_attention(&a, stream);   // reports the argument error
    if (need > kScratchBytes) return RGA_ERR_WORKSPACE;
    void *p = nullptr;
    rga_status st = scratch_address(&p);
    if (st != RGA_OK) return st;
    a.workspace = p;
    a.workspace_bytes = kScratchBytes;
    return trt_attention(&a, stream);
}
