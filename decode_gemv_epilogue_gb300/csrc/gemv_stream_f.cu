// TMA-streamed GEMV instantiations for the F32 and F16 formats: the plain GEMV.
#include "gemv_stream_impl.cuh"

namespace gf {

int launch_stream_float_plain(int wtype, int ncols, const Plan& p, cudaStream_t st, bool pdl) {
  return wtype == WT_F32 ? dispatch_cols<WT_F32, FEAT_PLAIN>(ncols, p, st, pdl) : dispatch_cols<WT_F16, FEAT_PLAIN>(ncols, p, st, pdl);
}

}  // namespace gf
