// Stand-alone kernels: the host staging copy, the signed FWHT, the unfused element-wise
// control ops and the dequantize test hook.
#include <algorithm>

#include "gf_device.cuh"
#include "gf_internal.h"

namespace gf {

// ------------------------------------------------------------------ host staging copy
// dst[i] = src[i] for n16 16-byte words; either side may be host memory the device
// addresses (pinned, registered, or pageable where the device reads it).  Waits for the
// preceding grid first (src may be its output) and lets the next one start early.
__global__ void __launch_bounds__(256) copy16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                     int64_t n16) {
  pdl_wait();
  pdl_trigger();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride)
    dst[i] = src[i];
}

int launch_copy(void* dst, const void* src, int64_t bytes, cudaStream_t st, bool pdl) {
  const int64_t n16 = bytes / 16;
  if (n16 <= 0) return cudaSuccess;
  // one word per thread up to 1024 CTAs (latency-bound sizes), then a grid-stride loop
  const int64_t grid = std::min<int64_t>((n16 + 255) / 256, 1024);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, copy16_kernel, static_cast<const uint4*>(src), static_cast<uint4*>(dst), n16);
}

// ------------------------------------------------------------------ signed FWHT
// Each CTA transforms E consecutive elements (a whole number of blocks) in shared
// memory: load (coalesced), sign-multiply on the first pass, radix-4/radix-2 passes,
// scale on the last pass, store.  dst may equal x: a CTA reads its whole segment
// before the first barrier and writes only after the last one.
constexpr int kFwhtThreads = 256;

__global__ void __launch_bounds__(kFwhtThreads) fwht_signed_kernel(const float* x, const float* signs,
                                                                   float* dst, int64_t n, int B, int nsigns,
                                                                   float scale, int E) {
  extern __shared__ __align__(16) float buf[];
  pdl_wait();
  pdl_trigger();
  const int64_t base = static_cast<int64_t>(blockIdx.x) * E;
  const int len = static_cast<int>(min(static_cast<int64_t>(E), n - base));
  for (int i = threadIdx.x; i < len; i += blockDim.x) buf[i] = x[base + i];
  __syncthreads();
  fwht_smem(buf, len, B, len, base, signs, nsigns, scale, threadIdx.x, blockDim.x,
            []() { __syncthreads(); });
  for (int i = threadIdx.x; i < len; i += blockDim.x) dst[base + i] = buf[i];
}

int launch_fwht(const float* x, const float* signs, float* dst, int64_t n, int B, int nsigns,
                cudaStream_t st) {
  // one block per CTA for large blocks; several small blocks (up to 4096 elements) per CTA
  int64_t E = B >= 1024 ? B : (4096 / B) * B;
  if (E > n) E = n;
  const int64_t grid = (n + E - 1) / E;
  const int smem = static_cast<int>(E * 4);
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (smem > 48 * 1024 && dev < 64 && configured[dev] < smem) {
    cudaError_t e = cudaFuncSetAttribute(fwht_signed_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[dev] = smem;
  }
  const float scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(B)));
  fwht_signed_kernel<<<static_cast<unsigned>(grid), kFwhtThreads, smem, st>>>(x, signs, dst, n, B, nsigns,
                                                                            scale, static_cast<int>(E));
  return cudaGetLastError();
}

// ------------------------------------------------------------------ element-wise control
__global__ void elementwise_kernel(int op, const float* a, const float* b, int64_t nb, float* dst,
                                   int64_t n) {
  pdl_wait();
  pdl_trigger();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float av = a[i];
    float r;
    switch (op) {
      case 1: r = tail_sigmoid(av); break;                 // GF_EW_SIGMOID
      case 2: r = tail_silu(av); break;                    // GF_EW_SILU
      case 3: r = av * b[nb == n ? i : i % nb]; break;     // GF_EW_MUL
      default: r = av + b[nb == n ? i : i % nb]; break;    // GF_EW_ADD
    }
    dst[i] = r;
  }
}

int launch_elementwise(int op, const float* a, const float* b, int64_t nb, float* dst, int64_t n,
                       cudaStream_t st) {
  int64_t grid = (n + 255) / 256;
  if (grid > 152 * 16) grid = 152 * 16;
  elementwise_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(op, a, b, nb, dst, n);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ failure-path self-test
// One thread waits, through the kernels' bounded wait, on a barrier phase that nothing
// completes (a fresh barrier's phase 0 with no arrivals expected).  The wait gives up after
// limit_ns, sets the abort flag and the device error word; a second wait then returns at
// once because of the abort flag.  out = {first wait succeeded, second wait succeeded,
// microseconds of the first wait, microseconds of the second}.
__global__ void selftest_wait_kernel(unsigned* err, uint64_t limit_ns, int* out) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  const uint64_t t0 = global_timer_ns();
  const bool first = mbar_wait_or_abort(b, 0, &abort_flag, err, limit_ns);
  const uint64_t t1 = global_timer_ns();
  const bool second = mbar_wait_or_abort(b, 0, &abort_flag, err, limit_ns);
  const uint64_t t2 = global_timer_ns();
  out[0] = first ? 1 : 0;
  out[1] = second ? 1 : 0;
  out[2] = static_cast<int>(min((t1 - t0) / 1000ull, 2000000000ull));
  out[3] = static_cast<int>(min((t2 - t1) / 1000ull, 2000000000ull));
}

int launch_selftest_wait(unsigned* err, uint64_t limit_ns, int* out, cudaStream_t st) {
  selftest_wait_kernel<<<1, 32, 0, st>>>(err, limit_ns, out);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ dequantize hook
// Same unit decoders as the streaming kernel (through a global-memory loader), one
// thread per 16-weight unit; the product with the block scale is exact in fp32.
template <int WT>
__global__ void dequantize_units_kernel(const uint8_t* W, int64_t M, int64_t K, int64_t row_bytes,
                                        float* out) {
  const int64_t units_per_row = K / kUnitElems;
  const int64_t total = M * units_per_row;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total; t += stride) {
    const int64_t row = t / units_per_row;
    const uint32_t u = static_cast<uint32_t>(t - row * units_per_row);
    const GmemLoader ld{W + row * row_bytes};
    float2 v[8];
    float d;
    decode_unit<WT>(ld, u, v, d);
    float* o = out + row * K;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t e = unit_pair_elem<WT>(u, k);
      o[e] = v[k].x * d;
      o[e + 1] = v[k].y * d;
    }
  }
}

// Q4_K: one thread per unit pair, through the stream kernel's pair decoder; each value
// d*sc*q - dmin*m with one rounding (d*sc*q and dmin*m are exact in fp32).
__global__ void dequantize_q4k_pairs_kernel(const uint8_t* W, int64_t M, int64_t K, int64_t row_bytes,
                                            float* out) {
  const int64_t pairs_per_row = K / (2 * kUnitElems);
  const int64_t total = M * pairs_per_row;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total; t += stride) {
    const int64_t row = t / pairs_per_row;
    const uint32_t p = static_cast<uint32_t>(t - row * pairs_per_row);
    const GmemLoader ld{W + row * row_bytes};
    float2 v[2][8];
    float dsc[2], dmn[2];
    const uint4 q = q4k_load_pair(ld, p, dsc, dmn);
    q4k_nibbles(q, 0, v[0]);
    q4k_nibbles(q, 1, v[1]);
    float* o = out + row * K;
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t e = unit_pair_elem<WT_Q4_K>(2 * p + n, k);
        o[e] = fmaf(dsc[n], v[n][k].x, -dmn[n]);
        o[e + 1] = fmaf(dsc[n], v[n][k].y, -dmn[n]);
      }
  }
}

// Element-wise decode for F32/F16 rows whose K is not a multiple of 8.
template <int WT>
__global__ void dequantize_elems_kernel(const uint8_t* W, int64_t M, int64_t K, int64_t row_bytes,
                                        float* out) {
  const int64_t total = M * K;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total; t += stride) {
    const int64_t row = t / K, k = t - row * K;
    out[t] = decode_elem<WT>(W + row * row_bytes, k);
  }
}

int launch_dequantize(int wtype, const uint8_t* W, int64_t M, int64_t K, int64_t row_bytes, float* out,
                      cudaStream_t st) {
  const bool by_unit = (K % kUnitElems == 0) &&
                       ((wtype != WT_F32 && wtype != WT_F16) ||
                        (reinterpret_cast<uintptr_t>(W) % 16 == 0 && row_bytes % 16 == 0));
  const int64_t work = by_unit ? M * (K / kUnitElems) : M * K;
  int64_t grid = (work + 255) / 256;
  if (grid > 152 * 16) grid = 152 * 16;
  if (grid < 1) grid = 1;
  const unsigned g = static_cast<unsigned>(grid);
  switch (wtype) {
    case WT_F32:
      if (by_unit) dequantize_units_kernel<WT_F32><<<g, 256, 0, st>>>(W, M, K, row_bytes, out);
      else dequantize_elems_kernel<WT_F32><<<g, 256, 0, st>>>(W, M, K, row_bytes, out);
      break;
    case WT_F16:
      if (by_unit) dequantize_units_kernel<WT_F16><<<g, 256, 0, st>>>(W, M, K, row_bytes, out);
      else dequantize_elems_kernel<WT_F16><<<g, 256, 0, st>>>(W, M, K, row_bytes, out);
      break;
    case WT_Q8_0: dequantize_units_kernel<WT_Q8_0><<<g, 256, 0, st>>>(W, M, K, row_bytes, out); break;
    case WT_Q4_0: dequantize_units_kernel<WT_Q4_0><<<g, 256, 0, st>>>(W, M, K, row_bytes, out); break;
    case WT_Q4_K: dequantize_q4k_pairs_kernel<<<g, 256, 0, st>>>(W, M, K, row_bytes, out); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace gf
