// decode_kv16w.cu - the decode kernels over a 16-bit (f16 / bf16) KV cache
// with two N-blocks (16 query rows) per pair, linear or paged (decode.cuh).
#include "decode.cuh"

namespace rga {

template cudaError_t launch_decode_kv<false, 2>(const AttnParams &, const TensorMaps &, int,
                                                cudaStream_t, int);

}  // namespace rga
