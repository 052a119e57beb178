// decode_kv16.cu - the decode kernels over a 16-bit (f16 / bf16) KV cache
// with one N-block of 8 query rows per pair, linear or paged (decode.cuh),
// and the decode entry of the launchers.
#include "decode.cuh"

namespace rga {

// instantiated in decode_kv16w.cu (two N-blocks) and decode_kv8.cu (fp8)
extern template cudaError_t launch_decode_kv<false, 2>(const AttnParams &, const TensorMaps &,
                                                       int, cudaStream_t, int);
extern template cudaError_t launch_decode_kv<true, 1>(const AttnParams &, const TensorMaps &,
                                                      int, cudaStream_t, int);
template cudaError_t launch_decode_kv<false, 1>(const AttnParams &, const TensorMaps &, int,
                                                cudaStream_t, int);

cudaError_t launch_decode(const AttnParams &p, const TensorMaps &m, int mode, cudaStream_t s,
                          int bf16, int kv8) {
    if (kv8) return launch_decode_kv<true, 1>(p, m, mode, s, bf16);
    // more than two 16-row chunks per (batch, KV head) on average (tree
    // decoding): the grouped kernel reads each K/V tile once for them all
    const long long qrows = p.q_packed ? (long long)p.q_seq * p.G / (p.B > 0 ? p.B : 1)
                                       : (long long)p.q_seq * p.G;
    if (p.dec_rows == DEC_ROWS_WIDE && qrows > 2 * DEC_ROWS_WIDE)
        return launch_decode_group(p, m, mode, s, bf16);
    return p.dec_rows == DEC_ROWS_WIDE ? launch_decode_kv<false, 2>(p, m, mode, s, bf16)
                                       : launch_decode_kv<false, 1>(p, m, mode, s, bf16);
}

}  // namespace rga
