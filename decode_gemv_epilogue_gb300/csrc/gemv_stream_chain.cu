// TMA-streamed GEMV instantiations for persistent chains of one-column calls, every format.
#include "gemv_stream_impl.cuh"

namespace gf {

int launch_stream_chain(int wtype, int grid, int threads, int smem, const ChainArgs& a, cudaStream_t st,
                        bool pdl) {
  switch (wtype) {
    case WT_F32: return launch_chain_t<WT_F32>(grid, threads, smem, a, st, pdl);
    case WT_F16: return launch_chain_t<WT_F16>(grid, threads, smem, a, st, pdl);
    case WT_Q8_0: return launch_chain_t<WT_Q8_0>(grid, threads, smem, a, st, pdl);
    case WT_Q4_0: return launch_chain_t<WT_Q4_0>(grid, threads, smem, a, st, pdl);
    case WT_Q4_K: return launch_chain_t<WT_Q4_K>(grid, threads, smem, a, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

int stream_chain_ctas_per_sm(int wtype, int threads, int smem) {
  switch (wtype) {
    case WT_F32: return chain_ctas_per_sm_t<WT_F32>(threads, smem);
    case WT_F16: return chain_ctas_per_sm_t<WT_F16>(threads, smem);
    case WT_Q8_0: return chain_ctas_per_sm_t<WT_Q8_0>(threads, smem);
    case WT_Q4_0: return chain_ctas_per_sm_t<WT_Q4_0>(threads, smem);
    case WT_Q4_K: return chain_ctas_per_sm_t<WT_Q4_K>(threads, smem);
    default: return 0;
  }
}

}  // namespace gf
