// Host/device shared declarations for the gemvfuse library (not part of the C ABI).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

struct CUtensorMap_st;  // the driver's tensor-map descriptor (cuda.h)

namespace gf {

// Kernel-side limits of the TMA-streamed GEMV.
constexpr int kMaxCols = 8;      // columns per GEMV launch
constexpr int kMaxBatch = 256;   // columns per call (wider batches run in blocks of kMaxCols)
constexpr int kMaxStages = 8;
constexpr int kBarBytes = 256;              // mbarrier area at the start of shared memory
constexpr int kXsMaxBytes = 64 * 1024;      // x chunk (all columns) kept in shared memory
constexpr int kXStageMaxBytes = 32 * 1024;  // x staged without a prologue (whole rows only)
constexpr int kSegMaxBytes = 32 * 1024;     // bytes of one row's K chunk
constexpr int kStageMaxBytes = 72 * 1024;
constexpr int kRedMaxBytes = 16 * 1024;
constexpr int kRingSlackBytes = 16;         // aligned-word decoders may read 3 bytes past a row
constexpr int kMaxFusedFwhtBlock = 8192;
constexpr int kUnitElems = 16;              // weights per decode unit (half a quant block)
constexpr int kMaxSplit = 8;                // CTAs of a split-K cluster (portable cluster size)
constexpr int kMaxSeg = 4;                  // matrices sharing x in one multi-matrix launch

// Tiling of the consumer warps, per (format, columns):
//  U   units (16 weights) per thread per K chunk, RT rows per thread per tile;
//  NCT columns per thread, CS = ceil(NC / NCT) column groups.
// A tile of R = G * RT rows is split over G row groups of consumer warps; a row group is
// CS column groups of wpc warps; within a column group every thread owns U units of the
// K chunk and keeps their x values (NCT columns) in registers for the whole chunk.
// F32/F16 decode is cheap, so batches are split two columns per thread (more warps);
// Q8_0/Q4_0 keep up to four columns per thread so each weight is decoded once per four
// columns.  Q4_K threads always own one unit pair (two units sharing a code load) and
// one column: with 17 warps a thread has at most 96 registers (a quarter of the SM's
// register file serves up to five warps), and a second column of x spills.  Single-
// column Q4_0 and Q8_0 (integer dot products, below) keep one unit and eight rows per
// thread per tile: the x conversion per unit is the costly part of a chunk's start, the
// rows share it, and the per-tile reduction is spread over more rows (Q8_0 with four
// rows per thread: 5-8% slower at 4096..14336 rows).
__host__ __device__ constexpr bool stream_quant(int wt) { return wt == 2 || wt == 3 || wt == 4; }
__host__ __device__ constexpr int stream_nct(int wt, int nc) {
  return wt == 4 ? 1 : stream_quant(wt) ? (nc <= 4 ? nc : 4) : (nc <= 2 ? nc : 2);
}
__host__ __device__ constexpr int stream_cs(int wt, int nc) {
  return (nc + stream_nct(wt, nc) - 1) / stream_nct(wt, nc);
}
__host__ __device__ constexpr int stream_u(int wt, int nc) {
  return wt == 4 ? 2 : ((wt == 3 || wt == 2) && nc == 1) ? 1 : (nc == 1 && stream_quant(wt)) ? 2 : 1;
}
__host__ __device__ constexpr int stream_rt(int wt, int nc) {
  return (nc == 1 && (wt == 3 || wt == 2)) ? 8 : 4;
}
__host__ __device__ constexpr int stream_max_cw(int wt, int nc) { return stream_nct(wt, nc) <= 2 ? 16 : 8; }
__host__ __device__ constexpr int stream_threads(int wt, int nc) { return 32 * (1 + stream_max_cw(wt, nc)); }
// Q4_0, Q8_0 and Q4_K with up to kIntMaxCols columns take integer dot products (x as
// shared-exponent 24-bit integers, dp4a on the codes): a third to a half of the
// instructions per weight of the float decode.  With more columns per thread the float
// decode, done once for all of them, is cheaper.
constexpr int kIntMaxCols = 1;
__host__ __device__ constexpr bool stream_int(int wt, int nc) { return (wt >= 2 && wt <= 4) && nc <= kIntMaxCols; }

struct StreamArgs {
  const uint8_t* W;
  const float* x;
  const float* aux;
  float* dst;
  const float* signs;
  unsigned* err;
  int64_t M;
  int K;
  int epi;
  int row_bytes;     // bytes of a full row
  int kc_len;        // elements per K chunk
  int n_kc;          // K chunks
  int R;             // rows per tile (= G * RT)
  int G;             // row groups of consumer warps
  int wpg;           // warps per row group (= CS * wpc)
  int wpc;           // warps per column group
  int NS;            // ring stages
  int stage_bytes;   // bytes reserved per stage
  int RC;            // rows per finalize chunk
  int ncw;           // consumer warps (= G * wpg)
  int rows_base;     // granules of rows per CTA (the first rows_extra CTAs take one more)
  int rows_extra;
  int gran;          // rows per granule: 1, or a full tile's real rows
  int fwht_B;        // 0 = no prologue
  int nsigns;
  float fwht_scale;
  const uint8_t* W2; // up-projection rows of the gated dual GEMV (nullptr: one matrix)
  const float* gamma;  // RMS-normalisation weight [K] (nullptr: no normalisation)
  float norm_eps;
  // Several matrices sharing x in one pass (nseg > 0): virtual row r belongs to segment
  // i = the first with r < seg_end[i]; its rows are seg_W[i], its tail seg_epi[i] with
  // seg_aux[i], its output seg_dst[i] ([ncols][rows of the segment]).  W, epi, aux and dst
  // above are then unused.
  int nseg;
  const uint8_t* seg_W[kMaxSeg];
  int64_t seg_end[kMaxSeg];
  int seg_epi[kMaxSeg];
  const float* seg_aux[kMaxSeg];
  float* seg_dst[kMaxSeg];
  int S;             // CTAs per cluster sharing a row range, each a slice of the K chunks
  int stage_x;       // 1: the producer bulk-copies x (one K chunk, every column) into xs
  int off_xs, off_aux, off_red, off_norm, off_xchg, off_ring;
};

struct GenericArgs {
  const uint8_t* W;
  const float* x;
  const float* aux;
  float* dst;
  const float* signs;
  unsigned* err;
  int64_t M;
  int K;
  int epi;
  int64_t row_bytes;
  int fwht_B;
  int nsigns;
  float fwht_scale;
  const uint8_t* W2;
  const float* gamma;
  float norm_eps;
};

struct DeviceLimits;

// Tensor-core GEMV (F16 weights, batches): see gemv_tc.cu.
struct TcArgs {
  const float* x;
  const float* aux;
  float* dst;
  unsigned* err;
  int64_t M;
  int K;
  int epi;
  int ncols;          // columns of this launch (<= kTcMaxCols)
  int Np;             // columns rounded up to 8: B holds Np rows of hi, then Np of lo
  int S;              // CTAs per cluster splitting K (1: none)
  int subs;           // 64-element sub-tiles per stage
  int nst;            // stages of a row (K / (64 subs))
  int NS;             // pipeline stages
  int tmem_cols;      // tensor-memory columns allocated (power of two >= 2 Np, >= 32)
  int off_a, off_b;   // stage offsets from the 1024-aligned shared-memory base
  int b_stage_bytes;  // 2 Np rows of 128 bytes
  int off_x;          // x stages: ncols rows of 64 * subs floats per stage
  int x_stage_bytes;
};

struct TcPlan {
  int grid, smem;
  TcArgs a;
};

constexpr int kTcMaxCols = 16;  // columns per tensor-core launch (one B chunk per converter thread)

// Shapes only (pointers are filled by the caller); false if the kernel cannot take them.
bool plan_tc(int64_t M, int64_t K, int ncols, int epi, const DeviceLimits& lim, TcPlan& p);
// Encodes the tensor map of W ([M][K] f16, row stride 2K) and launches.
int launch_tc(const TcPlan& p, const void* W, cudaStream_t st, bool pdl);

// A 2-D tensor map of element type dtype (kMapU8, kMapF16, kMapF32) over rows of `inner`
// elements, `stride_bytes` apart, with boxes of box_inner x box_rows (128-byte swizzle or
// none).  `map` points to a 64-byte aligned CUtensorMap.  Returns a cudaError_t.
enum { kMapU8 = 0, kMapF16 = 1, kMapF32 = 2 };
int encode_map_2d(::CUtensorMap_st* map, int dtype, const void* base, uint64_t inner, uint64_t rows,
                  uint64_t stride_bytes, uint32_t box_inner, uint32_t box_rows, bool swizzle128);


// Generic kernel: 256 threads; shared memory x [ncols][K], 1/rms [ncols], warp
// partials [8][ncols].
constexpr int kGenericWarps = 8;
__host__ __device__ constexpr int64_t generic_smem_floats(int64_t ncols, int64_t K) {
  return ncols * K + ncols + kGenericWarps * ncols;
}

enum { PATH_STREAM = 1, PATH_GENERIC = 2, PATH_TC = 3 };

struct Plan {
  int path;
  int grid, threads, smem;
  StreamArgs s;   // valid when path == PATH_STREAM (pointers filled by the caller)
};

struct DeviceLimits {
  int sm_count;
  int smem_optin;
};

// Kernel feature sets of the streamed GEMV (separate instantiations).
enum { FEAT_PLAIN = 0, FEAT_EXT = 1, FEAT_SPLIT = 2 };

// Launchers (return cudaError_t).  `pdl` requests programmatic stream serialization.
// FEAT_SPLIT launches group the grid into clusters of p.s.S CTAs.  One function per
// (format family, feature set), each in its own translation unit.
int launch_stream_float_plain(int wtype, int ncols, const Plan& p, cudaStream_t st, bool pdl);  // F32, F16
int launch_stream_float_ext(int wtype, int ncols, const Plan& p, cudaStream_t st, bool pdl);
int launch_stream_float_split(int wtype, int ncols, const Plan& p, cudaStream_t st, bool pdl);
int launch_stream_block_plain(int wtype, int ncols, const Plan& p, cudaStream_t st, bool pdl);  // Q8_0, Q4_0
int launch_stream_block_ext(int wtype, int ncols, const Plan& p, cudaStream_t st, bool pdl);
int launch_stream_block_split(int wtype, int ncols, const Plan& p, cudaStream_t st, bool pdl);
int launch_stream_q4k_plain(int ncols, const Plan& p, cudaStream_t st, bool pdl);              // Q4_K
int launch_stream_q4k_ext(int ncols, const Plan& p, cudaStream_t st, bool pdl);
int launch_stream_q4k_split(int ncols, const Plan& p, cudaStream_t st, bool pdl);
// Resident clusters of the split-K kernel for this plan (0 if unknown, e.g. no device).
int stream_split_max_clusters_float(int wtype, int ncols, const Plan& p);
int stream_split_max_clusters_block(int wtype, int ncols, const Plan& p);
int stream_split_max_clusters_q4k(int ncols, const Plan& p);
int launch_generic(int wtype, int ncols, const GenericArgs& a, int grid, int smem,
                   cudaStream_t st, bool pdl);
int launch_fwht(const float* x, const float* signs, float* dst, int64_t n, int B, int nsigns,
                cudaStream_t st);
// Kernel copy of `bytes` (a multiple of 16) between device-addressable ranges.
int launch_copy(void* dst, const void* src, int64_t bytes, cudaStream_t st, bool pdl);
int launch_elementwise(int op, const float* a, const float* b, int64_t nb, float* dst, int64_t n,
                       cudaStream_t st);
int launch_dequantize(int wtype, const uint8_t* W, int64_t M, int64_t K, int64_t row_bytes,
                      float* out, cudaStream_t st);

unsigned* device_error_word();  // this device's error word (nullptr on failure)
int launch_selftest_wait(unsigned* err, uint64_t limit_ns, int* out, cudaStream_t st);

}  // namespace gf
