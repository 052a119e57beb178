// decode_kv16.cu - the decode kernels over a 16-bit (f16 / bf16) KV cache,
// linear or paged (decode.cuh), and the decode entry of the launchers.
#include "decode.cuh"

namespace rga {

// the fp8 kernels are instantiated in decode_kv8.cu
extern template cudaError_t launch_decode_kv<true>(const AttnParams &, const TensorMaps &, int,
                                                   cudaStream_t, int);
template cudaError_t launch_decode_kv<false>(const AttnParams &, const TensorMaps &, int,
                                            cudaStream_t, int);

cudaError_t launch_decode(const AttnParams &p, const TensorMaps &m, int mode, cudaStream_t s,
                          int bf16, int kv8) {
    return kv8 ? launch_decode_kv<true>(p, m, mode, s, bf16)
               : launch_decode_kv<false>(p, m, mode, s, bf16);
}

}  // namespace rga
