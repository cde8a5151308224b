// Decode path of the W4A16 linear layer: the bf16-activation instantiations
// of the kernels in decode_impl.cuh (a translation unit of their own, so that
// the two activation types compile in parallel).
#include "decode_impl.cuh"

namespace w4a16 {

cudaError_t decode_dispatch_resident_bf16(const DecodeArgs& args, int mt, int nw, int apg_t, int ctas,
                                          int bytes, cudaStream_t stream) {
  return dispatch_resident<true>(args, mt, nw, apg_t, ctas, bytes, stream);
}

cudaError_t decode_dispatch_streamk_bf16(const DecodeArgs& args, int mt, int apg_t, int ctas,
                                         cudaStream_t stream) {
  return dispatch_streamk<true>(args, mt, apg_t, ctas, stream);
}

}  // namespace w4a16
