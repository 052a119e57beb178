// decode_kv8.cu - the decode kernels over an FP8 (E4M3) KV cache, linear or
// paged (decode.cuh).
#include "decode.cuh"

namespace rga {

template cudaError_t launch_decode_kv<true, 1>(const AttnParams &, const TensorMaps &, int,
                                               cudaStream_t, int);

}  // namespace rga
