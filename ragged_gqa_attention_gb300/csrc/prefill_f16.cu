// prefill_f16.cu - the fp16 instantiations of the prefill kernel
// (split from the fp16/bf16 pair so that the two compile in parallel).
#include "prefill.cuh"

namespace rga {
template cudaError_t launch_prefill_typed<false>(const AttnParams &, const TensorMaps &,
                                                       int, int, cudaStream_t);
}  // namespace rga
