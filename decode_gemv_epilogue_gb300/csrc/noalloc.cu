// Allocation-free entry point for the transform-once signed-FWHT prologue path.
//
// Some callers cannot allocate device memory for a workspace: a C host that links only
// this library and has no device allocator of its own, or a serving process whose
// device memory is fixed at start-up and must not grow while requests are running.
// For them the prologue's scratch (the transformed x', ncols*K floats) lives in a
// file-scope device array owned by the library.  Every GPU that loads the library keeps
// this array (GF_NOALLOC_MAX_WORKSPACE_FLOATS floats, 1 MiB) until the process exits.
//
// Host code cannot use the array's name as a device address, so the address is looked
// up once per device with cudaGetSymbolAddress (the first call on a device does this,
// with that device current) and handed to the kernels through gemv_fused_ex's
// workspace option.  Nothing is allocated or freed, here or below.  The address stays
// valid as long as the device's primary context does: a cudaDeviceReset by the host
// invalidates it (and the device error word of api.cu), so the library must be
// reloaded after one.
#include <cstdint>
#include <mutex>

#include "gemvfuse.h"

namespace {

constexpr int64_t kMaxFloats = GF_NOALLOC_MAX_WORKSPACE_FLOATS;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_workspace[kMaxFloats];

// Device address of this device's array, looked up on first use; nullptr on failure.
float* workspace_address() {
  static std::mutex mu;
  static float* addr[kMaxDevices] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<float*>(p);
  }
  return addr[dev];
}

}  // namespace

extern "C" GF_API int gemv_fused_fwht_noalloc(const void* W, int wtype, const float* x, int64_t M, int64_t K,
                                              int epilogue, const float* aux, float* dst, int64_t ncols,
                                              const float* fwht_signs, int64_t fwht_block, int64_t nsigns,
                                              uint32_t flags, void* stream) {
  if (!fwht_signs) return GF_ERR_INVALID;
  const int64_t nc = ncols == 0 ? 1 : ncols;
  if (nc < 1 || K < 0 || M < 0) return GF_ERR_INVALID;
  if (K > 0 && nc > kMaxFloats / K) return GF_ERR_UNSUPPORTED;  // ncols*K above the static array
  gf_opts o = {};
  o.ncols = nc;
  o.fwht_signs = fwht_signs;
  o.fwht_block = fwht_block;
  o.nsigns = nsigns;
  o.flags = flags;
  o.fwht_workspace = nullptr;
  if (M > 0 && K > 0) {
    float* ws = workspace_address();
    if (!ws) return GF_ERR_CUDA;
    o.fwht_workspace = ws;
  }
  return gemv_fused_ex(W, wtype, x, M, K, epilogue, aux, dst, &o, stream);
}
