// TMA-streamed GEMV instantiations for the Q8_0 and Q4_0 formats: the gated dual GEMV / RMS-normalisation prologue.
#include "gemv_stream_impl.cuh"

namespace gf {

int launch_stream_block_ext(int wtype, int ncols, const Plan& p, cudaStream_t st, bool pdl) {
  return wtype == WT_Q8_0 ? dispatch_cols<WT_Q8_0, FEAT_EXT>(ncols, p, st, pdl) : dispatch_cols<WT_Q4_0, FEAT_EXT>(ncols, p, st, pdl);
}

}  // namespace gf
