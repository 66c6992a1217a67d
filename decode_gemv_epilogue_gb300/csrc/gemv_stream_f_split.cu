// TMA-streamed GEMV instantiations for the F32 and F16 formats: split K over thread-block clusters.
#include "gemv_stream_impl.cuh"

namespace gf {

int launch_stream_float_split(int wtype, int ncols, const Plan& p, cudaStream_t st, bool pdl) {
  return wtype == WT_F32 ? dispatch_cols<WT_F32, FEAT_SPLIT>(ncols, p, st, pdl) : dispatch_cols<WT_F16, FEAT_SPLIT>(ncols, p, st, pdl);
}

int stream_split_max_clusters_float(int wtype, int ncols, const Plan& p) {
  return wtype == WT_F32 ? occupancy_cols<WT_F32>(ncols, p) : occupancy_cols<WT_F16>(ncols, p);
}

}  // namespace gf
