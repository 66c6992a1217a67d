// TMA-streamed GEMV instantiations for the Q4_K format: split K over thread-block clusters.
#include "gemv_stream_impl.cuh"

namespace gf {

int launch_stream_q4k_split(int ncols, const Plan& p, cudaStream_t st, bool pdl) {
  return dispatch_cols<WT_Q4_K, FEAT_SPLIT>(ncols, p, st, pdl);
}

int stream_split_max_clusters_q4k(int ncols, const Plan& p) { return occupancy_cols<WT_Q4_K>(ncols, p); }

}  // namespace gf
