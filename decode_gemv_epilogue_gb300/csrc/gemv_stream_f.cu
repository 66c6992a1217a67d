// TMA-streamed GEMV instantiations for the F32 and F16 weight formats.
#include "gemv_stream_impl.cuh"

namespace gf {

template <int WT>
static int dispatch_cols(int ncols, const Plan& p, cudaStream_t st, bool pdl) {
  switch (ncols) {
    case 1: return launch_stream_t<WT, 1>(p, st, pdl);
    case 2: return launch_stream_t<WT, 2>(p, st, pdl);
    case 3: return launch_stream_t<WT, 3>(p, st, pdl);
    case 4: return launch_stream_t<WT, 4>(p, st, pdl);
    case 5: return launch_stream_t<WT, 5>(p, st, pdl);
    case 6: return launch_stream_t<WT, 6>(p, st, pdl);
    case 7: return launch_stream_t<WT, 7>(p, st, pdl);
    case 8: return launch_stream_t<WT, 8>(p, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

int launch_stream_float(int wtype, int ncols, const Plan& p, cudaStream_t st, bool pdl) {
  return wtype == WT_F32 ? dispatch_cols<WT_F32>(ncols, p, st, pdl)
                         : dispatch_cols<WT_F16>(ncols, p, st, pdl);
}

}  // namespace gf
