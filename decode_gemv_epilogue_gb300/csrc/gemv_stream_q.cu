// TMA-streamed GEMV instantiations for the Q8_0 and Q4_0 formats: the plain GEMV.
#include "gemv_stream_impl.cuh"

namespace gf {

int launch_stream_block_plain(int wtype, int ncols, const Plan& p, cudaStream_t st, bool pdl) {
  return wtype == WT_Q8_0 ? dispatch_cols<WT_Q8_0, FEAT_PLAIN>(ncols, p, st, pdl) : dispatch_cols<WT_Q4_0, FEAT_PLAIN>(ncols, p, st, pdl);
}

}  // namespace gf
