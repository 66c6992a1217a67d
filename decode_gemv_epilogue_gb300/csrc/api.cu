// C ABI of gemvfuse: argument validation (sizes, alignment, the aliasing contract),
// kernel planning for the TMA-streamed GEMV, dispatch, and the device error word.
//
// Aliasing contract ("feat(cuda): fuse activations and residual add into mmv f/q
// epilogues", What changed): dst may alias the mul/add operand only as the same
// element index (dst == aux, in place), and may not overlap the product inputs (W, the
// up matrix of the gated dual GEMV, x, the FWHT signs, the normalisation weight), which
// are read across the whole reduction.  Every call is validated on its own; no
// overlap-guard state is kept between calls.
#include <algorithm>
#include <cmath>
#include <new>
#include <cstdint>
#include <cstring>
#include <limits>
#include <mutex>

#include "gemvfuse.h"
#include "gf_device.cuh"
#include "gf_internal.h"

namespace gf {

// Per device: [0] the error bits of bounded waits that gave up, [1] the row chunks whose
// sums the integer path handed to the fp32 repair (see the streamed kernel).
__device__ unsigned int g_error_word[2];

static thread_local int t_last_cuda_error = 0;

static int cuda_fail(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return GF_ERR_CUDA;
}

unsigned* device_error_word() {
  static std::mutex mu;
  static unsigned* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<unsigned*>(p);
  }
  return addr[dev];
}

static DeviceLimits device_limits() {
  static std::mutex mu;
  static DeviceLimits lim[64];
  static bool have[64] = {false};
  DeviceLimits fallback{152, 232448};  // GB300: 152 SMs, 227 KB opt-in shared memory
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return fallback;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!have[dev]) {
    DeviceLimits l = fallback;
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      l.sm_count = v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess && v > 0)
      l.smem_optin = v;
    cudaGetLastError();
    lim[dev] = l;
    have[dev] = true;
  }
  return lim[dev];
}

// ------------------------------------------------------------------ helpers

static int64_t row_bytes_of(int wtype, int64_t K) {
  switch (wtype) {
    case GF_F32: return 4 * K;
    case GF_F16: return 2 * K;
    case GF_Q8_0: return (K / 32) * 34;
    case GF_Q4_K: return (K / 256) * 144;
    default: return (K / 32) * 18;
  }
}

static bool ranges_overlap(const void* a, int64_t abytes, const void* b, int64_t bbytes) {
  if (!a || !b || abytes <= 0 || bbytes <= 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + static_cast<uintptr_t>(bbytes) && b0 < a0 + static_cast<uintptr_t>(abytes);
}

static bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

static bool is_pow2(int64_t v) { return v >= 1 && (v & (v - 1)) == 0; }

struct Call {
  const void* W;
  int wtype;
  const float* x;
  int64_t M, K;
  int epi;
  const float* aux;
  const float* dst;
  int64_t ncols;
  const float* signs;
  int64_t fwht_block, nsigns;
  uint32_t flags;
  float* workspace;
  const void* W2;       // gated dual GEMV: the up matrix (epi == EPI_GLU)
  const float* gamma;   // RMS-normalisation prologue weight [K]
  float eps;
  int nseg = 0;         // several matrices sharing x (gemv_multi): M is their rows' sum
  gf_multi_item segs[kMaxSeg];
};

static int validate(const Call& c) {
  if (c.wtype < GF_F32 || c.wtype > GF_Q4_K) return GF_ERR_INVALID;
  if (c.epi == EPI_GLU) {
    if (!c.W2 && c.M > 0 && c.K > 0) return GF_ERR_INVALID;
  } else if (c.epi < GF_EPI_NONE || c.epi > GF_EPI_ADD || c.W2) {
    return GF_ERR_INVALID;
  }
  if (c.M < 0 || c.K < 0) return GF_ERR_INVALID;
  if (c.M > INT32_MAX || c.K > INT32_MAX / 8) return GF_ERR_UNSUPPORTED;
  if (c.ncols < 1 || c.ncols > kMaxBatch) return c.ncols < 1 ? GF_ERR_INVALID : GF_ERR_UNSUPPORTED;
  if ((c.wtype == GF_Q8_0 || c.wtype == GF_Q4_0) && c.K % 32 != 0) return GF_ERR_UNSUPPORTED;
  if (c.wtype == GF_Q4_K && c.K % 256 != 0) return GF_ERR_UNSUPPORTED;
  const bool need_aux = (c.epi == GF_EPI_SILU_MUL || c.epi == GF_EPI_ADD);
  if (c.M > 0) {
    if (!c.dst) return GF_ERR_INVALID;
    if (need_aux && !c.aux) return GF_ERR_INVALID;
    if (c.K > 0 && (!c.W || !c.x)) return GF_ERR_INVALID;
  }
  const uintptr_t walign = c.wtype == GF_F32 ? 4 : 2;
  if (c.W && !aligned(c.W, walign)) return GF_ERR_ALIGN;
  if (c.W2 && !aligned(c.W2, walign)) return GF_ERR_ALIGN;
  if (c.gamma) {
    if (!(c.eps >= 0.0f) || !(c.eps <= std::numeric_limits<float>::max())) return GF_ERR_INVALID;
    if (!aligned(c.gamma, 4)) return GF_ERR_ALIGN;
    if (c.signs) return GF_ERR_UNSUPPORTED;  // one prologue per call
  }
  if ((c.x && !aligned(c.x, 4)) || (c.dst && !aligned(c.dst, 4)) || (need_aux && c.aux && !aligned(c.aux, 4)))
    return GF_ERR_ALIGN;
  if (c.signs) {
    if (!aligned(c.signs, 4)) return GF_ERR_ALIGN;
    if (!is_pow2(c.fwht_block)) return GF_ERR_INVALID;
    if (c.fwht_block > kMaxFusedFwhtBlock) return GF_ERR_UNSUPPORTED;
    if (c.nsigns < 1) return GF_ERR_INVALID;
    if (c.K % c.fwht_block != 0 || c.K % c.nsigns != 0) return GF_ERR_INVALID;
  }
  // aliasing: dst against W, x, signs (never) and aux (only exactly equal)
  const int64_t dbytes = c.ncols * c.M * 4;
  const int64_t wbytes = c.M * row_bytes_of(c.wtype, c.K);
  const int64_t xbytes = c.ncols * c.K * 4;
  if (ranges_overlap(c.dst, dbytes, c.W, wbytes)) return GF_ERR_ALIAS;
  if (ranges_overlap(c.dst, dbytes, c.W2, wbytes)) return GF_ERR_ALIAS;
  if (c.gamma && ranges_overlap(c.dst, dbytes, c.gamma, c.K * 4)) return GF_ERR_ALIAS;
  if (ranges_overlap(c.dst, dbytes, c.x, xbytes)) return GF_ERR_ALIAS;
  if (c.signs && ranges_overlap(c.dst, dbytes, c.signs, c.nsigns * 4)) return GF_ERR_ALIAS;
  if (need_aux && c.aux != c.dst && ranges_overlap(c.dst, dbytes, c.aux, dbytes)) return GF_ERR_ALIAS;
  if (c.workspace && c.signs && c.M > 0 && c.K > 0) {
    if (!aligned(c.workspace, 16)) return GF_ERR_ALIGN;
    if (ranges_overlap(c.workspace, xbytes, c.W, wbytes) || ranges_overlap(c.workspace, xbytes, c.x, xbytes) ||
        ranges_overlap(c.workspace, xbytes, c.W2, wbytes) ||
        ranges_overlap(c.workspace, xbytes, c.dst, dbytes) || ranges_overlap(c.workspace, xbytes, c.signs, c.nsigns * 4) ||
        (need_aux && ranges_overlap(c.workspace, xbytes, c.aux, dbytes)))
      return GF_ERR_ALIAS;
  }
  return GF_OK;
}

// The tensor-core kernel takes F16 weights with a batch of at least kTcMinCols
// columns (no gated dual GEMV, no on-chip prologue), 16-byte aligned W and x, K a
// multiple of 64.  Measured on GB300 (signed FWHT + 5120^2, graph + PDL): 2 columns
// 15.7 us vs 14.2 us on the CUDA cores, 3 columns 15.7 vs 21.4 us, 8 columns 17.0 vs
// 31.9 us.
constexpr int kTcMinCols = 3;

static bool tc_eligible(const Call& c) {
  return c.wtype == GF_F16 && !c.W2 && !c.gamma && !c.signs && c.nseg == 0 && !(c.flags & GF_FLAG_NO_TENSOR_CORES) &&
         c.ncols >= kTcMinCols && c.K >= 64 && c.K % 64 == 0 && aligned(c.W, 16) && aligned(c.x, 16);
}

static int round_up(int v, int a) { return (v + a - 1) / a * a; }

// Plan the TMA-streamed kernel with S CTAs per cluster splitting K (S = 1: no split);
// returns false if the shape/alignment needs another S or the generic kernel.
static bool plan_stream_s(const Call& c, const DeviceLimits& lim, int S, Plan& p) {
  const int nc = static_cast<int>(c.ncols);
  const int K = static_cast<int>(c.K);
  const int64_t rb = row_bytes_of(c.wtype, c.K);
  const bool dual = c.W2 != nullptr;
  const int vr = dual ? 2 : 1;  // virtual rows per output row
  if (c.K < kUnitElems || K % kUnitElems != 0) return false;
  if (rb % 16 != 0 || !aligned(c.W, 16) || !aligned(c.x, 16)) return false;
  if (dual && !aligned(c.W2, 16)) return false;
  for (int i = 0; i < c.nseg; ++i)
    if (!aligned(c.segs[i].W, 16)) return false;
  if (c.gamma && !aligned(c.gamma, 16)) return false;
  if (rb > INT32_MAX / 2) return false;
  const int U = stream_u(c.wtype, nc), RT = stream_rt(c.wtype, nc);
  const int CS = stream_cs(c.wtype, nc);
  const int max_cw = stream_max_cw(c.wtype, nc);
  auto seg_of = [&](int klen) -> int { return static_cast<int>(row_bytes_of(c.wtype, klen)); };
  // K chunk: the whole row if x, one row's bytes and the units all fit; else a multiple
  // of the granule (256 elements, or the FWHT block) that does.  Split K caps the chunk
  // so that every CTA of a cluster gets at least one.
  int gran = 256;
  if (c.signs) gran = std::max<int>(gran, static_cast<int>(c.fwht_block));
  const int64_t cap_x = c.signs ? kXsMaxBytes / (4 * nc) : INT32_MAX;  // x staged only for the prologue
  const int64_t cap_units = static_cast<int64_t>(kUnitElems) * U * 32 * (max_cw / CS);
  const int cap_seg = std::min(kSegMaxBytes, kStageMaxBytes / RT);  // RT rows fit one stage
  int kc = K;
  if (K > cap_x || seg_of(K) > cap_seg || K > cap_units) {
    const int g_x = static_cast<int>(cap_x / gran);
    const int g_seg = cap_seg / seg_of(gran);
    const int g_u = static_cast<int>(cap_units / gran);
    const int gch = std::min(std::min(g_x, g_seg), g_u);
    if (gch < 1) return false;
    kc = gch * gran;
  }
  if (S > 1) {
    if (K % gran != 0) return false;
    kc = std::min(kc, std::max(gran, (K / S) / gran * gran));
  }
  const int n_kc = (K + kc - 1) / kc;
  if (n_kc < S) return false;
  const int seg_full = seg_of(kc);
  if (seg_full % 16 != 0) return false;
  if (n_kc > 1) {
    const int last = K - (n_kc - 1) * kc;
    if (seg_of(last) % 16 != 0 || last % kUnitElems != 0) return false;
  }
  const int units = kc / kUnitElems;
  const int wpc = (((units + U - 1) / U) + 31) / 32;
  const int wpg = CS * wpc;
  if (wpg > max_cw) return false;
  const int nclusters = static_cast<int>(std::min<int64_t>(lim.sm_count / S, c.M));
  if (nclusters < 1) return false;
  int rows_base = static_cast<int>(c.M / nclusters);
  int rows_extra = static_cast<int>(c.M % nclusters);
  int rows_max = rows_base + (rows_extra ? 1 : 0);
  int G = std::max(1, std::min(max_cw / wpg, (vr * rows_max + RT - 1) / RT));
  while (G > 1 && G * RT * seg_full > kStageMaxBytes) --G;
  int ncw = G * wpg;
  int R = G * RT;
  // With at least one full tile per CTA, hand out whole tiles: the CTAs with the highest
  // indices, which a launch behind another (PDL) starts last, take one tile fewer, and
  // no CTA decodes a part-filled tile of a full tile's cost.  Fewer rows than that: rows.
  int row_gran = 1;
  const int64_t tile_rows = R / vr;  // real rows of a full tile
  if (S == 1 && c.M >= tile_rows * nclusters) {
    const int64_t ntile = (c.M + tile_rows - 1) / tile_rows;
    row_gran = static_cast<int>(tile_rows);
    rows_base = static_cast<int>(ntile / nclusters);
    rows_extra = static_cast<int>(ntile % nclusters);
    rows_max = (rows_base + (rows_extra ? 1 : 0)) * row_gran;
  }
  int RC = std::min(rows_max, std::max(R, kRedMaxBytes / (vr * wpc * nc * 4)));
  RC = std::min(RC, 512);
  if (S > 1 && RC < rows_max) return false;  // split K exchanges one row chunk per CTA
  // x is staged in shared memory by the producer when the row is one chunk and the
  // staging costs at most one ring stage of a ring that keeps four or more
  // (with the RMS prologue gamma is staged after x)
  const int xcols = nc + (c.gamma ? 1 : 0);
  bool stage_x = !c.signs && n_kc == 1 && xcols * kc * 4 <= kXStageMaxBytes;
  int xs_bytes = c.signs ? round_up(nc * kc * 4, 128) : stage_x ? round_up(xcols * kc * 4, 128) : 0;
  const int aux_bytes = round_up(nc * RC * 4, 128);
  const int red_bytes = round_up(vr * RC * wpc * nc * 4, 128);
  const int norm_bytes = c.gamma ? round_up(wpc * nc * 4, 128) : 0;
  const int xchg_bytes = S > 1 ? round_up(S * nc * (vr * RC + 1) * 4, 128) : 0;
  int fixed = kBarBytes + xs_bytes + aux_bytes + red_bytes + norm_bytes + xchg_bytes + kRingSlackBytes;
  const int stage_bytes = round_up(R * seg_full, 128);
  int NS = std::min(kMaxStages, (lim.smem_optin - fixed) / stage_bytes);
  if (stage_x) {
    const int ns_plain = std::min(kMaxStages, (lim.smem_optin - (fixed - xs_bytes)) / stage_bytes);
    if (NS < std::min(ns_plain, 4) || NS < ns_plain - 1) {  // not worth the stages: load x directly
      stage_x = false;
      fixed -= xs_bytes;
      xs_bytes = 0;
      NS = ns_plain;
    }
  }
  if (NS < 2) return false;
  p.path = PATH_STREAM;
  p.grid = nclusters * S;
  p.threads = 32 * (1 + ncw);
  p.smem = fixed + NS * stage_bytes;
  StreamArgs& s = p.s;
  std::memset(&s, 0, sizeof(s));
  s.M = c.M;
  s.K = K;
  s.epi = c.epi;
  s.row_bytes = static_cast<int>(rb);
  s.kc_len = kc;
  s.n_kc = n_kc;
  s.R = R;
  s.G = G;
  s.wpg = wpg;
  s.wpc = wpc;
  s.NS = NS;
  s.stage_bytes = stage_bytes;
  s.RC = RC;
  s.ncw = ncw;
  s.rows_base = rows_base;
  s.rows_extra = rows_extra;
  s.gran = row_gran;
  s.fwht_B = c.signs ? static_cast<int>(c.fwht_block) : 0;
  s.nsigns = c.signs ? static_cast<int>(c.nsigns) : 1;
  s.fwht_scale = c.signs ? static_cast<float>(1.0 / std::sqrt(static_cast<double>(c.fwht_block))) : 1.0f;
  s.norm_eps = c.gamma ? c.eps : 0.0f;
  s.S = S;
  s.stage_x = stage_x ? 1 : 0;
  s.off_xs = kBarBytes;
  s.off_aux = s.off_xs + xs_bytes;
  s.off_red = s.off_aux + aux_bytes;
  s.off_norm = s.off_red + red_bytes;
  s.off_xchg = s.off_norm + norm_bytes;
  s.off_ring = s.off_xchg + xchg_bytes;
  return true;
}

// Split K when the rows alone would leave most SMs idle and each CTA would stream a
// long row range by itself: S = min(8, SMs / M) CTAs per cluster, each streaming a
// slice of every row's K chunks (and of x).  Measured on GB300: with under ~128 KB of x
// and weights per CTA the cluster launch costs more than the split saves.
constexpr int64_t kSplitMinCtaBytes = 128 * 1024;

static int split_factor(const Call& c, const DeviceLimits& lim) {
  if ((c.flags & GF_FLAG_NO_SPLIT_K) || c.nseg > 0) return 1;
  if (c.M < 1 || 2 * c.M > lim.sm_count) return 1;
  const int64_t vr = c.W2 ? 2 : 1;
  const int64_t cta_bytes = c.ncols * c.K * 4 + vr * row_bytes_of(c.wtype, c.K);  // one row per CTA
  if (cta_bytes < kSplitMinCtaBytes) return 1;
  return static_cast<int>(std::min<int64_t>(kMaxSplit, lim.sm_count / c.M));
}

static int split_max_clusters(const Call& c, const Plan& p) {
  const int nc = static_cast<int>(c.ncols);
  if (c.wtype == GF_Q4_K) return stream_split_max_clusters_q4k(nc, p);
  return (c.wtype == GF_F32 || c.wtype == GF_F16) ? stream_split_max_clusters_float(c.wtype, nc, p)
                                                  : stream_split_max_clusters_block(c.wtype, nc, p);
}

static bool plan_stream(const Call& c, const DeviceLimits& lim, Plan& p) {
  // the largest split whose clusters all fit on the device at once (when the device can
  // be asked; without one, the largest that plans)
  for (int S = split_factor(c, lim); S > 1; --S) {
    if (!plan_stream_s(c, lim, S, p)) continue;
    const int fit = split_max_clusters(c, p);
    if (fit == 0 || p.grid / S <= fit) return true;
  }
  return plan_stream_s(c, lim, 1, p);
}

static int plan_call(const Call& c, Plan& p, int* generic_smem, int* generic_grid, TcPlan* tc = nullptr) {
  const DeviceLimits lim = device_limits();
  if (tc && tc_eligible(c) && plan_tc(c.M, c.K, static_cast<int>(c.ncols), c.epi, lim, *tc)) return PATH_TC;
  if (plan_stream(c, lim, p)) return PATH_STREAM;
  const int64_t smem = generic_smem_floats(c.ncols, c.K) * 4;
  if (smem > lim.smem_optin) return GF_ERR_UNSUPPORTED;
  *generic_smem = static_cast<int>(smem);
  const int64_t rows_per_cta = 8;  // one row per warp of the 256-thread generic CTA
  int64_t grid = (c.M + rows_per_cta - 1) / rows_per_cta;
  grid = std::min<int64_t>(grid, 2 * lim.sm_count);
  *generic_grid = static_cast<int>(std::max<int64_t>(grid, 1));
  p.path = PATH_GENERIC;
  return PATH_GENERIC;
}

// One kernel launch with every argument resolved: what a call plans, and what a
// prepared call keeps (gf_prepare) so that launching it does no planning at all.
enum { REC_FWHT = 0, REC_TC = 1, REC_STREAM = 2, REC_GENERIC = 3, REC_COPY = 4 };
struct LaunchRec {
  int kind;
  bool pdl;
  const void* csrc;  // host staging copy (device-addressable pointers)
  void* cdst;
  int64_t cbytes;
  int wtype, ncols;
  const void* W;  // tensor-core path: the matrix of the tensor map
  const float* fx;  // stand-alone FWHT
  const float* fsigns;
  float* fdst;
  int64_t fn;
  int fB, fnsigns;
  TcPlan tp;
  Plan p;
  GenericArgs g;
  int ggrid, gsmem;
};
constexpr int kMaxRecs = 1 + kMaxSeg * (kMaxBatch / kMaxCols);  // transform + column blocks (per matrix)

// The operand pointers of a streamed launch of call c (the plan holds the shapes).
static void fill_stream_ptrs(const Call& c, float* dst, unsigned* err, StreamArgs& s) {
  s.W = static_cast<const uint8_t*>(c.W);
  s.x = c.x;
  s.aux = c.aux;
  s.dst = dst;
  s.signs = c.signs;
  s.err = err;
  s.W2 = static_cast<const uint8_t*>(c.W2);
  s.gamma = c.gamma;
  s.nseg = c.nseg;
  int64_t end = 0;
  for (int i = 0; i < c.nseg; ++i) {
    end += c.segs[i].M;
    s.seg_W[i] = static_cast<const uint8_t*>(c.segs[i].W);
    s.seg_end[i] = end;
    s.seg_epi[i] = c.segs[i].epilogue;
    s.seg_aux[i] = c.segs[i].aux;
    s.seg_dst[i] = c.segs[i].dst;
  }
}

// Plans one launch of at most one column block into r.
static int plan_one(const Call& c, float* dst, LaunchRec& r) {
  int gsmem = 0, ggrid = 0;
  const int path = plan_call(c, r.p, &gsmem, &ggrid, &r.tp);
  if (path < 0) return path;
  unsigned* err = device_error_word();
  if (!err) return cuda_fail(cudaGetLastError());
  r.pdl = (c.flags & GF_FLAG_PDL) != 0;
  r.wtype = c.wtype;
  r.ncols = static_cast<int>(c.ncols);
  r.W = c.W;
  if (path == PATH_TC) {
    r.kind = REC_TC;
    r.tp.a.x = c.x;
    r.tp.a.aux = c.aux;
    r.tp.a.dst = dst;
    r.tp.a.err = err;
  } else if (path == PATH_STREAM) {
    r.kind = REC_STREAM;
    fill_stream_ptrs(c, dst, err, r.p.s);
  } else {
    r.kind = REC_GENERIC;
    GenericArgs& g = r.g;
    g.W = static_cast<const uint8_t*>(c.W);
    g.x = c.x;
    g.aux = c.aux;
    g.dst = dst;
    g.signs = c.signs;
    g.err = err;
    g.M = c.M;
    g.K = static_cast<int>(c.K);
    g.epi = c.epi;
    g.row_bytes = row_bytes_of(c.wtype, c.K);
    g.fwht_B = c.signs ? static_cast<int>(c.fwht_block) : 0;
    g.nsigns = c.signs ? static_cast<int>(c.nsigns) : 1;
    g.fwht_scale = c.signs ? static_cast<float>(1.0 / std::sqrt(static_cast<double>(c.fwht_block))) : 1.0f;
    g.W2 = static_cast<const uint8_t*>(c.W2);
    g.gamma = c.gamma;
    g.norm_eps = c.gamma ? c.eps : 0.0f;
    r.ggrid = ggrid;
    r.gsmem = gsmem;
  }
  return GF_OK;
}

static int issue(const LaunchRec& r, cudaStream_t st) {
  int e;
  if (r.kind == REC_COPY) {
    e = launch_copy(r.cdst, r.csrc, r.cbytes, st, r.pdl);
  } else if (r.kind == REC_FWHT) {
    e = launch_fwht(r.fx, r.fsigns, r.fdst, r.fn, r.fB, r.fnsigns, st);
  } else if (r.kind == REC_TC) {
    e = launch_tc(r.tp, r.W, st, r.pdl);
  } else if (r.kind == REC_STREAM) {
    const StreamArgs& s = r.p.s;
    const int nc = r.ncols;
    const bool fl = (r.wtype == GF_F32 || r.wtype == GF_F16);
    const bool ext = s.W2 != nullptr || s.gamma != nullptr || s.nseg > 0;
    if (r.wtype == GF_Q4_K)
      e = s.S > 1 ? launch_stream_q4k_split(nc, r.p, st, r.pdl)
          : ext   ? launch_stream_q4k_ext(nc, r.p, st, r.pdl)
                  : launch_stream_q4k_plain(nc, r.p, st, r.pdl);
    else if (s.S > 1)
      e = fl ? launch_stream_float_split(r.wtype, nc, r.p, st, r.pdl)
             : launch_stream_block_split(r.wtype, nc, r.p, st, r.pdl);
    else if (ext)
      e = fl ? launch_stream_float_ext(r.wtype, nc, r.p, st, r.pdl)
             : launch_stream_block_ext(r.wtype, nc, r.p, st, r.pdl);
    else
      e = fl ? launch_stream_float_plain(r.wtype, nc, r.p, st, r.pdl)
             : launch_stream_block_plain(r.wtype, nc, r.p, st, r.pdl);
  } else {
    e = launch_generic(r.wtype, r.ncols, r.g, r.ggrid, r.gsmem, st, r.pdl);
  }
  return e != cudaSuccess ? cuda_fail(static_cast<cudaError_t>(e)) : GF_OK;
}

// The launches of a validated call, in order, into recs[0 .. *n).  A batch wider than
// one launch takes runs in column blocks (kMaxCols columns on the CUDA-core kernels,
// kTcMaxCols on the tensor cores) in consecutive launches (each streams W again); later
// blocks may start early (programmatic dependent launch): they read and write only
// their own columns.  With a workspace the prologue runs first as a stand-alone
// transform into it, and the GEMV on it is launched with programmatic dependent launch:
// it streams W while the transform runs and waits for it before reading x' (W is not
// written by the transform, so this holds whatever the caller's flags).
static int plan_launches(const Call& c0, float* dst, LaunchRec* recs, int cap, int* n) {
  *n = 0;
  if (c0.M == 0) return GF_OK;
  Call c = c0;
  if (c0.workspace && c0.K > 0) {
    if (cap < 1) return GF_ERR_UNSUPPORTED;
    LaunchRec& f = recs[(*n)++];
    f.kind = REC_FWHT;
    f.pdl = false;
    f.fx = c0.x;
    f.fsigns = c0.signs;
    f.fdst = c0.workspace;
    f.fn = c0.ncols * c0.K;
    f.fB = static_cast<int>(c0.fwht_block);
    f.fnsigns = static_cast<int>(c0.nsigns);
    c.x = c0.workspace;
    c.signs = nullptr;
    c.fwht_block = 0;
    c.nsigns = 0;
    c.workspace = nullptr;
    c.flags |= GF_FLAG_PDL;
  }
  const int64_t width = tc_eligible(c) ? kTcMaxCols : kMaxCols;
  if (c.nseg > 0) {
    // one pass over every matrix when the streamed kernel takes the block shape, else one
    // launch per matrix
    Call probe = c;
    probe.ncols = std::min<int64_t>(width, c.ncols);
    Plan pp;
    if (!plan_stream(probe, device_limits(), pp)) {
      for (int i = 0; i < c.nseg; ++i) {
        Call one = c;
        one.nseg = 0;
        one.W = c.segs[i].W;
        one.M = c.segs[i].M;
        one.epi = c.segs[i].epilogue;
        one.aux = c.segs[i].aux;
        one.dst = c.segs[i].dst;
        if (*n > 0) one.flags |= GF_FLAG_PDL;  // after the transform or the previous matrix
        int m = 0;
        const int e = plan_launches(one, c.segs[i].dst, recs + *n, cap - *n, &m);
        if (e != GF_OK) return e;
        *n += m;
      }
      return GF_OK;
    }
  }
  for (int64_t col = 0; col < c.ncols; col += width) {
    Call b = c;
    b.ncols = std::min<int64_t>(width, c.ncols - col);
    b.x = c.x + col * c.K;
    b.aux = c.aux ? c.aux + col * c.M : nullptr;
    b.dst = dst + col * c.M;
    for (int i = 0; i < c.nseg; ++i) {
      b.segs[i].aux = c.segs[i].aux ? c.segs[i].aux + col * c.segs[i].M : nullptr;
      b.segs[i].dst = c.segs[i].dst + col * c.segs[i].M;
    }
    if (col > 0) b.flags |= GF_FLAG_PDL;
    if (*n >= cap) return GF_ERR_UNSUPPORTED;
    const int e = plan_one(b, const_cast<float*>(b.dst), recs[*n]);
    if (e != GF_OK) return e;
    ++*n;
  }
  return GF_OK;
}

static int run_call(const Call& c, float* dst, cudaStream_t st) {
  LaunchRec recs[kMaxRecs];
  int n = 0;
  const int e = plan_launches(c, dst, recs, kMaxRecs, &n);
  if (e != GF_OK) return e;
  for (int i = 0; i < n; ++i) {
    const int r = issue(recs[i], st);
    if (r != GF_OK) return r;
  }
  return GF_OK;
}

static Call make_call(const void* W, int wtype, const float* x, int64_t M, int64_t K, int epilogue,
                      const float* aux, const float* dst, const gf_opts* opts) {
  Call c;
  c.W = W;
  c.wtype = wtype;
  c.x = x;
  c.M = M;
  c.K = K;
  c.epi = epilogue;
  c.aux = (epilogue == GF_EPI_SILU_MUL || epilogue == GF_EPI_ADD) ? aux : nullptr;
  c.dst = dst;
  c.ncols = 1;
  c.signs = nullptr;
  c.fwht_block = 0;
  c.nsigns = 0;
  c.flags = 0;
  c.workspace = nullptr;
  c.W2 = nullptr;
  c.gamma = nullptr;
  c.eps = 0.0f;
  if (opts) {
    c.ncols = opts->ncols == 0 ? 1 : opts->ncols;
    c.signs = opts->fwht_signs;
    c.fwht_block = opts->fwht_block;
    c.nsigns = opts->nsigns;
    c.flags = opts->flags;
    c.workspace = opts->fwht_signs ? opts->fwht_workspace : nullptr;
    c.gamma = opts->rms_norm_weight;
    c.eps = opts->rms_norm_eps;
  }
  return c;
}

// gemv_multi: each matrix is checked as the call gemv_fused_ex(W_i, ...) would be, then
// against the other matrices' operands.
static int make_multi_call(const gf_multi_item* items, int n, int wtype, const float* x, int64_t K,
                           const gf_opts* opts, Call* out) {
  if (!items || n < 1) return GF_ERR_INVALID;
  if (n > kMaxSeg) return GF_ERR_UNSUPPORTED;
  if (opts)
    for (int i = 0; i < 4; ++i)
      if (opts->view_ne[i] != 0) return GF_ERR_INVALID;
  int64_t rows = 0;
  for (int i = 0; i < n; ++i) {
    const gf_multi_item& it = items[i];
    const Call one = make_call(it.W, wtype, x, it.M, K, it.epilogue, it.aux, it.dst, opts);
    const int v = validate(one);
    if (v != GF_OK) return v;
    if (it.M > INT32_MAX - rows) return GF_ERR_UNSUPPORTED;
    rows += it.M;
  }
  Call c = make_call(items[0].W, wtype, x, rows, K, GF_EPI_NONE, nullptr, items[0].dst, opts);
  const int64_t nc = c.ncols;
  for (int i = 0; i < n; ++i) {
    const gf_multi_item& a = items[i];
    const bool aux_a = a.epilogue == GF_EPI_SILU_MUL || a.epilogue == GF_EPI_ADD;
    for (int j = 0; j < n; ++j) {
      if (j == i) continue;
      const gf_multi_item& b = items[j];
      const bool aux_b = b.epilogue == GF_EPI_SILU_MUL || b.epilogue == GF_EPI_ADD;
      const int64_t da = nc * a.M * 4;
      if (ranges_overlap(a.dst, da, b.W, b.M * row_bytes_of(wtype, K)) ||
          ranges_overlap(a.dst, da, b.dst, nc * b.M * 4) || (aux_b && ranges_overlap(a.dst, da, b.aux, nc * b.M * 4)))
        return GF_ERR_ALIAS;
      (void)aux_a;
    }
    c.segs[i] = items[i];
    if (!aux_a) c.segs[i].aux = nullptr;
  }
  c.nseg = n;
  *out = c;
  return GF_OK;
}

static int check_view(const gf_opts* opts, int64_t M) {
  if (!opts) return GF_OK;
  bool any = false;
  int64_t prod = 1;
  for (int i = 0; i < 4; ++i) {
    const int64_t v = opts->view_ne[i];
    if (v < 0) return GF_ERR_INVALID;
    if (v > 0) {
      any = true;
      if (prod > INT64_MAX / v) return GF_ERR_INVALID;
      prod *= v;
    }
  }
  if (any && prod != M) return GF_ERR_INVALID;
  return GF_OK;
}

}  // namespace gf

using namespace gf;

extern "C" {

int gemv_fused_ex(const void* W, int wtype, const float* x, int64_t M, int64_t K, int epilogue,
                  const float* aux, float* dst, const gf_opts* opts, void* stream) {
  const Call c = make_call(W, wtype, x, M, K, epilogue, aux, dst, opts);
  int v = validate(c);
  if (v != GF_OK) return v;
  v = check_view(opts, M);
  if (v != GF_OK) return v;
  return run_call(c, dst, static_cast<cudaStream_t>(stream));
}

int gemv_fused(const void* W, int wtype, const float* x, int64_t M, int64_t K, int epilogue,
               const float* aux, float* dst, void* stream) {
  return gemv_fused_ex(W, wtype, x, M, K, epilogue, aux, dst, nullptr, stream);
}

static Call make_glu_call(const void* W_gate, const void* W_up, int wtype, const float* x, int64_t M, int64_t K,
                          const float* dst, const gf_opts* opts) {
  Call c = make_call(W_gate, wtype, x, M, K, GF_EPI_NONE, nullptr, dst, opts);
  c.epi = EPI_GLU;
  c.W2 = W_up;
  return c;
}

int gemv_glu(const void* W_gate, const void* W_up, int wtype, const float* x, int64_t M, int64_t K, float* dst,
             const gf_opts* opts, void* stream) {
  const Call c = make_glu_call(W_gate, W_up, wtype, x, M, K, dst, opts);
  int v = validate(c);
  if (v != GF_OK) return v;
  v = check_view(opts, M);
  if (v != GF_OK) return v;
  return run_call(c, dst, static_cast<cudaStream_t>(stream));
}

int gemv_multi(const gf_multi_item* items, int n, int wtype, const float* x, int64_t K, const gf_opts* opts,
               void* stream) {
  Call c;
  const int v = make_multi_call(items, n, wtype, x, K, opts, &c);
  if (v != GF_OK) return v;
  return run_call(c, const_cast<float*>(c.dst), static_cast<cudaStream_t>(stream));
}

static int plan_info(const Call& c, const gf_opts* opts, int64_t info[8]) {
  int v = validate(c);
  if (v != GF_OK) return v;
  v = check_view(opts, c.M);
  if (v != GF_OK) return v;
  if (c.M == 0) return 0;  // nothing would be launched
  Call pc = c;
  if (pc.workspace) {  // the GEMV of the workspace path reads x' without a prologue
    pc.x = pc.workspace;
    pc.signs = nullptr;
  }
  pc.ncols = std::min<int64_t>(pc.ncols, tc_eligible(pc) ? kTcMaxCols : kMaxCols);  // each block's launch
  Plan p;
  TcPlan tp;
  int gsmem = 0, ggrid = 0;
  const int path = plan_call(pc, p, &gsmem, &ggrid, &tp);
  if (path < 0) return path;
  if (info) {
    for (int i = 0; i < 8; ++i) info[i] = 0;
    if (path == PATH_TC) {
      info[0] = tp.grid; info[1] = 192; info[2] = 128; info[3] = tp.a.NS;
      info[4] = 64 * tp.a.subs; info[5] = tp.smem; info[6] = 0; info[7] = tp.a.S;
    } else if (path == PATH_STREAM) {
      info[0] = p.grid; info[1] = p.threads; info[2] = p.s.R; info[3] = p.s.NS;
      info[4] = p.s.kc_len; info[5] = p.smem; info[6] = p.s.RC; info[7] = p.s.S;
    } else {
      info[0] = ggrid; info[1] = 256; info[5] = gsmem; info[7] = 1;
    }
  }
  return path;
}

int gf_plan(const void* W, int wtype, const float* x, int64_t M, int64_t K, int epilogue, const float* aux,
            const float* dst, const gf_opts* opts, int64_t info[8]) {
  return plan_info(make_call(W, wtype, x, M, K, epilogue, aux, dst, opts), opts, info);
}

int gf_plan_glu(const void* W_gate, const void* W_up, int wtype, const float* x, int64_t M, int64_t K,
                const float* dst, const gf_opts* opts, int64_t info[8]) {
  return plan_info(make_glu_call(W_gate, W_up, wtype, x, M, K, dst, opts), opts, info);
}

int fwht_signed(const float* x, const float* signs, float* dst, int64_t n, int64_t block, int64_t nsigns,
                void* stream) {
  if (n < 0 || !is_pow2(block)) return GF_ERR_INVALID;
  if (block > 16384) return GF_ERR_UNSUPPORTED;
  if (n % block != 0) return GF_ERR_INVALID;
  if (signs && (nsigns < 1 || n % nsigns != 0)) return GF_ERR_INVALID;
  if (n == 0) return GF_OK;
  if (!x || !dst) return GF_ERR_INVALID;
  if (!aligned(x, 4) || !aligned(dst, 4) || (signs && !aligned(signs, 4))) return GF_ERR_ALIGN;
  if (x != dst && ranges_overlap(x, n * 4, dst, n * 4)) return GF_ERR_ALIAS;
  if (signs && ranges_overlap(signs, nsigns * 4, dst, n * 4)) return GF_ERR_ALIAS;
  if (n > INT32_MAX) return GF_ERR_UNSUPPORTED;
  const int e = launch_fwht(x, signs, dst, n, static_cast<int>(block), signs ? static_cast<int>(nsigns) : 1,
                            static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(static_cast<cudaError_t>(e));
  return GF_OK;
}

int gf_elementwise(int op, const float* a, const float* b, int64_t nb, float* dst, int64_t n, void* stream) {
  if (op < GF_EW_SIGMOID || op > GF_EW_ADD) return GF_ERR_INVALID;
  if (n < 0) return GF_ERR_INVALID;
  const bool binary = (op == GF_EW_MUL || op == GF_EW_ADD);
  if (binary && (nb < 1 || n % nb != 0)) return GF_ERR_INVALID;
  if (n == 0) return GF_OK;
  if (!a || !dst || (binary && !b)) return GF_ERR_INVALID;
  if (!aligned(a, 4) || !aligned(dst, 4) || (binary && !aligned(b, 4))) return GF_ERR_ALIGN;
  if (a != dst && ranges_overlap(a, n * 4, dst, n * 4)) return GF_ERR_ALIAS;
  if (binary && b != dst && ranges_overlap(b, nb * 4, dst, n * 4)) return GF_ERR_ALIAS;
  const int e = launch_elementwise(op, a, binary ? b : nullptr, binary ? nb : 1, dst, n,
                                   static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(static_cast<cudaError_t>(e));
  return GF_OK;
}

int gf_dequantize(const void* W, int wtype, int64_t M, int64_t K, float* out, void* stream) {
  if (wtype < GF_F32 || wtype > GF_Q4_K) return GF_ERR_INVALID;
  if (M < 0 || K < 0) return GF_ERR_INVALID;
  if ((wtype == GF_Q8_0 || wtype == GF_Q4_0) && K % 32 != 0) return GF_ERR_UNSUPPORTED;
  if (wtype == GF_Q4_K && K % 256 != 0) return GF_ERR_UNSUPPORTED;
  if (M == 0 || K == 0) return GF_OK;
  if (!W || !out) return GF_ERR_INVALID;
  if (!aligned(W, wtype == GF_F32 ? 4 : 2) || !aligned(out, 4)) return GF_ERR_ALIGN;
  const int64_t rb = row_bytes_of(wtype, K);
  if (ranges_overlap(W, M * rb, out, M * K * 4)) return GF_ERR_ALIAS;
  const int e = launch_dequantize(wtype, static_cast<const uint8_t*>(W), M, K, rb, out,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(static_cast<cudaError_t>(e));
  return GF_OK;
}

int gf_selftest_wait_timeout(int64_t limit_us, int* out, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return GF_ERR_INVALID;
  if (!out) return GF_ERR_INVALID;
  if (!aligned(out, 4)) return GF_ERR_ALIGN;
  unsigned* err = device_error_word();
  if (!err) return cuda_fail(cudaGetLastError());
  const int e = launch_selftest_wait(err, static_cast<uint64_t>(limit_us) * 1000ull, out,
                                     static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(static_cast<cudaError_t>(e));
  return GF_OK;
}

int gf_device_status(int reset) {
  unsigned* err = device_error_word();
  if (!err) return cuda_fail(cudaGetLastError());
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned v = 0;
  e = cudaMemcpy(&v, err, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (reset) {
    e = cudaMemset(err, 0, sizeof(unsigned));
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return (v & ERRBIT_TIMEOUT) ? GF_ERR_TIMEOUT : GF_OK;
}

int64_t gf_repair_count(int reset) {
  unsigned* err = device_error_word();
  if (!err) return cuda_fail(cudaGetLastError());
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned v = 0;
  e = cudaMemcpy(&v, err + 1, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (reset) {
    e = cudaMemset(err + 1, 0, sizeof(unsigned));
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return static_cast<int64_t>(v);
}

const char* gf_status_string(int status) {
  switch (status) {
    case GF_OK: return "GF_OK";
    case GF_ERR_INVALID: return "GF_ERR_INVALID: bad argument";
    case GF_ERR_ALIAS: return "GF_ERR_ALIAS: dst overlaps an input it may not alias";
    case GF_ERR_UNSUPPORTED: return "GF_ERR_UNSUPPORTED: shape or option not implemented";
    case GF_ERR_ALIGN: return "GF_ERR_ALIGN: misaligned pointer";
    case GF_ERR_CUDA: return "GF_ERR_CUDA: CUDA call failed";
    case GF_ERR_TIMEOUT: return "GF_ERR_TIMEOUT: a kernel gave up on a bounded wait";
    default: return "unknown gf_status";
  }
}

int gf_last_cuda_error(void) { return t_last_cuda_error; }

int gf_version(void) { return 5; }

// ------------------------------------------------------------------ prepared calls
struct gf_prepared {
  int device;
  int n;
  gf::LaunchRec recs[gf::kMaxRecs];
};

static int prepare(const Call& c, const gf_opts* opts, gf_prepared** out) {
  if (!out) return GF_ERR_INVALID;
  *out = nullptr;
  int v = c.nseg > 0 ? GF_OK : validate(c);  // a multi-matrix call was checked per matrix
  if (v != GF_OK) return v;
  v = c.nseg > 0 ? GF_OK : check_view(opts, c.M);
  if (v != GF_OK) return v;
  gf_prepared* p = new (std::nothrow) gf_prepared;
  if (!p) return GF_ERR_INVALID;
  if (cudaGetDevice(&p->device) != cudaSuccess) {
    delete p;
    return cuda_fail(cudaGetLastError());
  }
  v = plan_launches(c, const_cast<float*>(c.dst), p->recs, kMaxRecs, &p->n);  // dst came in as float*
  if (v != GF_OK) {
    delete p;
    return v;
  }
  *out = p;
  return GF_OK;
}

int gf_prepare(const void* W, int wtype, const float* x, int64_t M, int64_t K, int epilogue, const float* aux,
               float* dst, const gf_opts* opts, gf_prepared** out) {
  return prepare(make_call(W, wtype, x, M, K, epilogue, aux, dst, opts), opts, out);
}

int gf_prepare_glu(const void* W_gate, const void* W_up, int wtype, const float* x, int64_t M, int64_t K, float* dst,
                   const gf_opts* opts, gf_prepared** out) {
  return prepare(make_glu_call(W_gate, W_up, wtype, x, M, K, dst, opts), opts, out);
}

int gf_prepare_multi(const gf_multi_item* items, int n, int wtype, const float* x, int64_t K, const gf_opts* opts,
                     gf_prepared** out) {
  if (!out) return GF_ERR_INVALID;
  *out = nullptr;
  Call c;
  const int v = make_multi_call(items, n, wtype, x, K, opts, &c);
  if (v != GF_OK) return v;
  return prepare(c, opts, out);
}

int gf_launch_prepared(const gf_prepared* const* calls, int n, void* stream) {
  if (n < 0 || (n > 0 && !calls)) return GF_ERR_INVALID;
  for (int i = 0; i < n; ++i)
    if (!calls[i]) return GF_ERR_INVALID;
  int dev = -1;
  if (n > 0 && cudaGetDevice(&dev) != cudaSuccess) return cuda_fail(cudaGetLastError());
  for (int i = 0; i < n; ++i)
    if (calls[i]->device != dev) return GF_ERR_INVALID;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (int i = 0; i < n; ++i)
    for (int k = 0; k < calls[i]->n; ++k) {
      const int e = gf::issue(calls[i]->recs[k], st);
      if (e != GF_OK) return e;
    }
  return GF_OK;
}

void gf_free_prepared(gf_prepared* p) {
  if (!p) return;
  delete p;
}

// ------------------------------------------------------------------ host staging copies
// Checks a gf_copy request; on GF_OK *ks / *kd are the addresses the kernel uses (the
// device view of pinned host memory).  Shape checks come first and need no device.
static int check_copy(void* dst, const void* src, int64_t bytes, const void** ks, void** kd) {
  if (bytes < 0 || bytes % 16 != 0) return GF_ERR_INVALID;
  if (bytes == 0) return GF_OK;
  if (!dst || !src) return GF_ERR_INVALID;
  if (!aligned(dst, 16) || !aligned(src, 16)) return GF_ERR_ALIGN;
  if (ranges_overlap(src, bytes, dst, bytes)) return GF_ERR_ALIAS;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cuda_fail(cudaGetLastError());
  const void* in[2] = {src, dst};
  void* outp[2] = {nullptr, nullptr};
  for (int i = 0; i < 2; ++i) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, in[i]) != cudaSuccess) {
      (void)cudaGetLastError();
      return GF_ERR_INVALID;
    }
    if (at.type == cudaMemoryTypeDevice) {
      if (at.device != dev) return GF_ERR_INVALID;
      outp[i] = const_cast<void*>(in[i]);
    } else if (at.type == cudaMemoryTypeHost) {
      if (!at.devicePointer) return GF_ERR_INVALID;
      outp[i] = at.devicePointer;  // the address of `in[i]` in the device's view
    } else if (at.type == cudaMemoryTypeManaged) {
      outp[i] = const_cast<void*>(in[i]);
    } else {  // pageable host memory: not taken, even where the device could read it
      return GF_ERR_INVALID;
    }
  }
  *ks = outp[0];
  *kd = outp[1];
  return GF_OK;
}

int gf_copy(void* dst, const void* src, int64_t bytes, uint32_t flags, void* stream) {
  const void* ks = nullptr;
  void* kd = nullptr;
  const int v = check_copy(dst, src, bytes, &ks, &kd);
  if (v != GF_OK || bytes == 0) return v;
  const int e = gf::launch_copy(kd, ks, bytes, static_cast<cudaStream_t>(stream), (flags & GF_FLAG_PDL) != 0);
  return e != cudaSuccess ? cuda_fail(static_cast<cudaError_t>(e)) : GF_OK;
}

int gf_prepare_copy(void* dst, const void* src, int64_t bytes, uint32_t flags, gf_prepared** out) {
  if (!out) return GF_ERR_INVALID;
  *out = nullptr;
  const void* ks = nullptr;
  void* kd = nullptr;
  const int v = check_copy(dst, src, bytes, &ks, &kd);
  if (v != GF_OK) return v;
  gf_prepared* p = new (std::nothrow) gf_prepared;
  if (!p) return GF_ERR_INVALID;
  if (cudaGetDevice(&p->device) != cudaSuccess) {
    delete p;
    return cuda_fail(cudaGetLastError());
  }
  p->n = 0;
  if (bytes > 0) {
    gf::LaunchRec& r = p->recs[0];
    r.kind = gf::REC_COPY;
    r.pdl = (flags & GF_FLAG_PDL) != 0;
    r.csrc = ks;
    r.cdst = kd;
    r.cbytes = bytes;
    p->n = 1;
  }
  *out = p;
  return GF_OK;
}

// ------------------------------------------------------------------ step graphs
struct gf_graph {
  int device;
  cudaGraph_t graph;
  cudaGraphExec_t exec;
};

int gf_graph_create(const gf_prepared* const* calls, int n, gf_graph** out) {
  if (!out) return GF_ERR_INVALID;
  *out = nullptr;
  if (n < 1 || !calls) return GF_ERR_INVALID;
  for (int i = 0; i < n; ++i)
    if (!calls[i]) return GF_ERR_INVALID;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return cuda_fail(cudaGetLastError());
  for (int i = 0; i < n; ++i)
    if (calls[i]->device != dev) return GF_ERR_INVALID;
  cudaStream_t s = nullptr;
  cudaError_t e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
  if (e != cudaSuccess) return cuda_fail(e);
  cudaGraph_t g = nullptr;
  e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
  int st = GF_OK;
  if (e == cudaSuccess) {
    st = gf_launch_prepared(calls, n, s);
    e = cudaStreamEndCapture(s, &g);  // ends the capture whatever the launches returned
  }
  cudaStreamDestroy(s);
  if (e != cudaSuccess || st != GF_OK) {
    if (g) cudaGraphDestroy(g);
    return st != GF_OK ? st : cuda_fail(e);
  }
  cudaGraphExec_t x = nullptr;
  e = cudaGraphInstantiate(&x, g, 0);
  if (e != cudaSuccess) {
    cudaGraphDestroy(g);
    return cuda_fail(e);
  }
  gf_graph* r = new (std::nothrow) gf_graph;
  if (!r) {
    cudaGraphExecDestroy(x);
    cudaGraphDestroy(g);
    return GF_ERR_INVALID;
  }
  r->device = dev;
  r->graph = g;
  r->exec = x;
  *out = r;
  return GF_OK;
}

int gf_graph_launch(const gf_graph* g, void* stream) {
  if (!g) return GF_ERR_INVALID;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return cuda_fail(cudaGetLastError());
  if (dev != g->device) return GF_ERR_INVALID;
  const cudaError_t e = cudaGraphLaunch(g->exec, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GF_OK : cuda_fail(e);
}

void gf_graph_free(gf_graph* g) {
  if (!g) return;
  cudaGraphExecDestroy(g->exec);
  cudaGraphDestroy(g->graph);
  delete g;
}

}  // extern "C"
