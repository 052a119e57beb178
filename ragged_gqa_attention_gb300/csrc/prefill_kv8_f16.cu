// prefill_kv8_f16.cu - the f16 instantiations of the prefill kernel over an
// FP8 (E4M3) KV cache (one translation unit per element type, compiled in
// parallel).
#include "prefill.cuh"

namespace rga {
template cudaError_t launch_prefill_kv8_typed<false>(const AttnParams &, const TensorMaps &,
                                                     int, int, cudaStream_t);
}  // namespace rga
