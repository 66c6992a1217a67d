// TMA-streamed GEMV instantiations for the Q8_0 and Q4_0 block formats.
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

int launch_stream_block(int wtype, int ncols, const Plan& p, cudaStream_t st, bool pdl) {
  return wtype == WT_Q8_0 ? dispatch_cols<WT_Q8_0>(ncols, p, st, pdl)
                         : dispatch_cols<WT_Q4_0>(ncols, p, st, pdl);
}

}  // namespace gf
