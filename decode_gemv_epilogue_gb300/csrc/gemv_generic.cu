// Generic GEMV with fused prologue/epilogue for the shapes and alignments the
// TMA-streamed kernel does not take (ragged K, unaligned pointers or row strides).
// x (all columns) is staged in shared memory, optionally transformed by the signed
// FWHT there or multiplied by the RMS-normalisation weight (the per-column 1/rms is
// computed from the staged x first); each warp owns whole rows (of both matrices for
// the gated dual GEMV), decodes weights element by element from global memory,
// reduces with shuffles and applies the tail in lane 0.
#include "gf_device.cuh"
#include "gf_internal.h"

namespace gf {

constexpr int kGenericThreads = 32 * kGenericWarps;

template <int WT, int NC>
__global__ void __launch_bounds__(kGenericThreads) gemv_generic_kernel(const GenericArgs a) {
  extern __shared__ __align__(16) float xs[];  // [NC][K]
  pdl_wait();
  pdl_trigger();
  const int K = a.K;
  float* invs = xs + NC * K;
  float* part = invs + NC;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < NC * K; i += blockDim.x) xs[i] = a.x[i];
  __syncthreads();
  if (a.fwht_B > 0)
    fwht_smem(xs, NC * K, a.fwht_B, K, 0, a.signs, a.nsigns, a.fwht_scale, threadIdx.x, blockDim.x,
              []() { __syncthreads(); });
  if (a.gamma) {
    // per-column sum of squares in a fixed order, then x *= gamma in place
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      float ss = 0.0f;
      for (int k = threadIdx.x; k < K; k += blockDim.x) ss = fmaf(xs[c * K + k], xs[c * K + k], ss);
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      if (lane == 0) part[wid * NC + c] = ss;
    }
    __syncthreads();
    if (threadIdx.x < NC) {
      float t = 0.0f;
      for (int w = 0; w < kGenericWarps; ++w) t += part[w * NC + threadIdx.x];
      invs[threadIdx.x] = 1.0f / sqrtf(t / static_cast<float>(K) + a.norm_eps);
    }
    for (int i = threadIdx.x; i < NC * K; i += blockDim.x) xs[i] *= a.gamma[i % K];
    __syncthreads();
  }
  const bool dual = a.W2 != nullptr;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + wid; row < a.M; row += warps) {
    const uint8_t* wrow = a.W + row * a.row_bytes;
    const uint8_t* urow = dual ? a.W2 + row * a.row_bytes : nullptr;
    float acc[NC], accu[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) acc[c] = accu[c] = 0.0f;
    for (int k = lane; k < K; k += 32) {
      const float w = decode_elem<WT>(wrow, k);
#pragma unroll
      for (int c = 0; c < NC; ++c) acc[c] = fmaf(w, xs[c * K + k], acc[c]);
      if (dual) {
        const float wu = decode_elem<WT>(urow, k);
#pragma unroll
        for (int c = 0; c < NC; ++c) accu[c] = fmaf(wu, xs[c * K + k], accu[c]);
      }
    }
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      float s = acc[c], su = accu[c];
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        s += __shfl_xor_sync(0xffffffffu, s, off);
        su += __shfl_xor_sync(0xffffffffu, su, off);
      }
      if (lane == 0) {
        const int64_t o = static_cast<int64_t>(c) * a.M + row;
        if (a.gamma) {
          s *= invs[c];
          su *= invs[c];
        }
        if (dual) {
          a.dst[o] = tail_silu(s) * su;
        } else {
          const float av = (a.epi == EPI_SILU_MUL || a.epi == EPI_ADD) ? a.aux[o] : 0.0f;
          a.dst[o] = apply_tail(a.epi, s, av);
        }
      }
    }
  }
}

template <int WT, int NC>
static int launch_generic_t(const GenericArgs& a, int grid, int smem, cudaStream_t st, bool pdl) {
  auto kern = gemv_generic_kernel<WT, NC>;
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (smem > 48 * 1024 && dev < 64 && configured[dev] < smem) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[dev] = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGenericThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int WT>
static int generic_cols(int ncols, const GenericArgs& a, int grid, int smem, cudaStream_t st, bool pdl) {
  switch (ncols) {
    case 1: return launch_generic_t<WT, 1>(a, grid, smem, st, pdl);
    case 2: return launch_generic_t<WT, 2>(a, grid, smem, st, pdl);
    case 3: return launch_generic_t<WT, 3>(a, grid, smem, st, pdl);
    case 4: return launch_generic_t<WT, 4>(a, grid, smem, st, pdl);
    case 5: return launch_generic_t<WT, 5>(a, grid, smem, st, pdl);
    case 6: return launch_generic_t<WT, 6>(a, grid, smem, st, pdl);
    case 7: return launch_generic_t<WT, 7>(a, grid, smem, st, pdl);
    case 8: return launch_generic_t<WT, 8>(a, grid, smem, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

int launch_generic(int wtype, int ncols, const GenericArgs& a, int grid, int smem, cudaStream_t st,
                   bool pdl) {
  switch (wtype) {
    case WT_F32: return generic_cols<WT_F32>(ncols, a, grid, smem, st, pdl);
    case WT_F16: return generic_cols<WT_F16>(ncols, a, grid, smem, st, pdl);
    case WT_Q8_0: return generic_cols<WT_Q8_0>(ncols, a, grid, smem, st, pdl);
    case WT_Q4_0: return generic_cols<WT_Q4_0>(ncols, a, grid, smem, st, pdl);
    case WT_Q4_K: return generic_cols<WT_Q4_K>(ncols, a, grid, smem, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gf
