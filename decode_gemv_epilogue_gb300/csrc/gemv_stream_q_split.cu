// TMA-streamed GEMV instantiations for the Q8_0 and Q4_0 formats: split K over thread-block clusters.
#include "gemv_stream_impl.cuh"

namespace gf {

int launch_stream_block_split(int wtype, int ncols, const Plan& p, cudaStream_t st, bool pdl) {
  return wtype == WT_Q8_0 ? dispatch_cols<WT_Q8_0, FEAT_SPLIT>(ncols, p, st, pdl) : dispatch_cols<WT_Q4_0, FEAT_SPLIT>(ncols, p, st, pdl);
}

int stream_split_max_clusters_block(int wtype, int ncols, const Plan& p) {
  return wtype == WT_Q8_0 ? occupancy_cols<WT_Q8_0>(ncols, p) : occupancy_cols<WT_Q4_0>(ncols, p);
}

}  // namespace gf
