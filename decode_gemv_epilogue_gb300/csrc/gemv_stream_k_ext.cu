// TMA-streamed GEMV instantiations for the Q4_K format: the gated dual GEMV / RMS-normalisation prologue.
#include "gemv_stream_impl.cuh"

namespace gf {

int launch_stream_q4k_ext(int ncols, const Plan& p, cudaStream_t st, bool pdl) {
  return dispatch_cols<WT_Q4_K, FEAT_EXT>(ncols, p, st, pdl);
}

}  // namespace gf
