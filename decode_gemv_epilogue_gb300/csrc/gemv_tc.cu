// Tensor-core GEMV for F16 weights and a batch of columns (5th-generation tensor cores:
// tcgen05.mma with the accumulator in tensor memory).
//
// A CTA owns one tile of 128 rows of W and a slice of its K range.  Per 64-element K
// stage, warp 0 loads the 128 x 64 f16 tile of W with one 2-D TMA copy (128-byte
// swizzle, K-major: the tensor cores read it straight from shared memory); warps 2..5
// write the batch's x for the same 64 elements next to it as f16 rows in the same
// swizzled layout.  x is fp32, so each column is scaled by an exact power of two
// (its largest |x| over the CTA's K slice lands in [2^14, 2^15)) and split into
// hi = f16(x) and lo = f16(x - hi): B holds Np rows of hi followed by Np rows of lo
// (Np = columns rounded up to 8).  One thread of warp 1 issues four
// 128 x (2 Np) x 16 MMAs per stage into a TMEM accumulator and releases the stage
// with tcgen05.commit.  After the last stage the same four warps read their lane
// quarter of TMEM (one row per thread), form y = (hi part + lo part) * 2^-s, apply the
// tail and write dst.  hi + lo represents x to about 2^-22 relative, products of f16
// values are exact in fp32 and the accumulation is fp32.
//
// Rows alone give too few tiles for 152 SMs (e.g. 40 for 5120 rows), so K is split
// over a cluster of S CTAs per tile (S = SMs / tiles, at most 8); ranks 1..S-1 store
// their per-row partial sums into rank 0's shared memory and rank 0 adds them in rank
// order (deterministic).  Every wait is bounded; on a timeout the kernel sets the error
// word, drains its copies and MMAs, frees its tensor memory and returns.
#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "gf_device.cuh"
#include "gf_internal.h"

namespace gf {

constexpr int kTcRows = 128;                    // rows per tile (MMA M)
constexpr int kTcK = 64;                        // K elements per stage: one 128-byte f16 row
constexpr int kTcKSteps = kTcK / 16;            // MMAs per stage (K = 16 each)
constexpr int kTcThreads = 192;                 // warp 0 TMA, warp 1 MMA, warps 2..5 x / epilogue
constexpr int kTcABytes = kTcRows * kTcK * 2;   // 16 KB per stage
constexpr int kTcPrefetch = 4;                  // stages of x in flight per converter thread
constexpr int kTcMaxStages = 12;                // W tiles in flight: a 16 KB tile lands ~2.7 us after issue

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot_saddr, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_saddr), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A * B^T, A and B K-major f16 in shared memory (descriptors), fp32 D.
__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(da), "l"(db), "r"(idesc), "r"(accum)
      : "memory");
}

// Arrive on `bar` once every MMA this thread has issued so far has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// Eight consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzled layout
// (rows of 128 bytes, 8-row groups 1024 bytes apart; the tile starts 1024-aligned).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
  d |= static_cast<uint64_t>(1) << 16;                          // leading offset (unused when swizzled)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;                  // stride between 8-row groups
  d |= static_cast<uint64_t>(1) << 46;                          // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                          // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp32 D, f16 A and B, both K-major, M x N.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Byte offset of element (row, k) of a 64-wide K-major f16 tile in the 128-byte
// swizzle: the 16-byte chunk index is XORed with the row's position in its 8-row group.
__device__ __forceinline__ uint32_t sw128_offset(int row, int k) {
  return static_cast<uint32_t>(row) * 128u + ((static_cast<uint32_t>(k >> 3) ^ (row & 7)) << 4) +
         static_cast<uint32_t>(k & 7) * 2u;
}

// ------------------------------------------------------------------ kernel
// Shared memory from a 1024-aligned base: barriers and the TMEM address slot [0, 512);
// per-warp column maxima [512, 1536); scales and inverse scales [1536, 2048); the
// split-K exchange [2048, off_a); NS A stages (16 KB each) at off_a; NS B stages at
// off_b (2 Np rows of 128 bytes each).
template <bool SPLIT>
__global__ void __launch_bounds__(kTcThreads, 1) gemv_tc_kernel(const __grid_constant__ CUtensorMap tmap,
                                                                const TcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t pad = ((raw_s + 1023u) & ~1023u) - raw_s;
  uint8_t* base = smem_raw + pad;
  const uint32_t sb = raw_s + pad;
  const int NS = a.NS;
  const uint32_t fullA0 = sb, fullB0 = sb + 8u * NS, empty0 = sb + 16u * NS;
  const uint32_t accbar = sb + 24u * NS, xchbar = accbar + 8u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + 24 * NS + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + 24 * NS + 20);
  float* smax = reinterpret_cast<float*>(base + 512);   // [4 warps][64] column maxima
  float* scl = reinterpret_cast<float*>(base + 1536);   // [64]
  float* iscl = scl + 64;                               // [64]
  float* xch = reinterpret_cast<float*>(base + 2048);   // [S][Np][128]
  const uint32_t sA = sb + static_cast<uint32_t>(a.off_a), sB = sb + static_cast<uint32_t>(a.off_b);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int crank = 0;
  if constexpr (SPLIT) crank = static_cast<int>(cluster_ctarank());
  const int S = SPLIT ? a.S : 1;
  const int row0 = (static_cast<int>(blockIdx.x) / S) * kTcRows;
  const int st0 = crank * a.nst / S, st1 = (crank + 1) * a.nst / S;  // this CTA's K stages
  const int nmy = st1 - st0;
  const int Np = a.Np;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < NS; ++i) {
      mbar_init(fullA0 + 8u * i, 1);
      mbar_init(fullB0 + 8u * i, 128);
      mbar_init(empty0 + 8u * i, 1);
    }
    mbar_init(accbar, 1);
    mbar_init(xchbar, static_cast<uint32_t>(SPLIT ? (S - 1) * 128 : 1));
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), static_cast<uint32_t>(a.tmem_cols));
  tc_fence_before();
  if constexpr (SPLIT)
    cluster_sync_all();
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();

  if (warp == 0) {
    // ------------------------------------------------------------ W tiles (TMA)
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nmy; ++i) {
        const int slot = i % NS, round = i / NS;
        if (!mbar_wait_or_abort(empty0 + 8u * slot, static_cast<uint32_t>((round & 1) ^ 1), abort_flag, a.err))
          break;
        mbar_arrive_expect_tx(fullA0 + 8u * slot, static_cast<uint32_t>(kTcABytes));
        tma_load_2d(sA + static_cast<uint32_t>(slot * kTcABytes), &tmap, (st0 + i) * kTcK, row0,
                    fullA0 + 8u * slot);
        ++issued;
      }
      if (issued < nmy)  // aborted: wait (bounded) for the copies in flight
        for (int i = max(0, issued - NS); i < issued; ++i)
          (void)mbar_wait(fullA0 + 8u * (i % NS), static_cast<uint32_t>((i / NS) & 1));
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_f16(kTcRows, 2 * Np);
      for (int i = 0; i < nmy; ++i) {
        const int slot = i % NS, round = i / NS;
        if (!mbar_wait_or_abort(fullA0 + 8u * slot, static_cast<uint32_t>(round & 1), abort_flag, a.err)) break;
        if (!mbar_wait_or_abort(fullB0 + 8u * slot, static_cast<uint32_t>(round & 1), abort_flag, a.err)) break;
        tc_fence_after();
        const uint64_t da = umma_desc_sw128(sA + static_cast<uint32_t>(slot * kTcABytes));
        const uint64_t db = umma_desc_sw128(sB + static_cast<uint32_t>(slot * a.b_stage_bytes));
#pragma unroll
        for (int kk = 0; kk < kTcKSteps; ++kk)  // +32 bytes of K per step inside the swizzled rows
          umma_f16(tmem, da + 2u * kk, db + 2u * kk, idesc, (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(empty0 + 8u * slot);
      }
      umma_commit(accbar);  // also after an abort: arrives once every issued MMA is done
    }
  } else {
    // ------------------------------------------------------------ x rows of B, then the epilogue
    const int ctid = threadIdx.x - 64, cw = warp - 2;
    auto xbar = [&]() { named_bar_sync(1, 128); };
    pdl_wait();  // x, aux and dst may belong to the preceding grid
    // scale 2^s per column with its largest |x| * 2^s in [2^14, 2^15): maxima over this
    // CTA's K slice, four columns per pass so their loads are in flight together
    const int k0 = st0 * kTcK, klen4 = nmy * kTcK / 4;
    for (int n0 = 0; n0 < a.ncols; n0 += 4) {
      float m[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 4
      for (int i = ctid; i < klen4; i += 128) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (n0 + u < a.ncols) {
            const float4 v = reinterpret_cast<const float4*>(a.x + static_cast<int64_t>(n0 + u) * a.K + k0)[i];
            m[u] = fmaxf(m[u], fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) m[u] = fmaxf(m[u], __shfl_xor_sync(0xffffffffu, m[u], off));
        if (lane == 0 && n0 + u < a.ncols) smax[cw * 64 + n0 + u] = m[u];
      }
    }
    xbar();
    if (ctid < Np) {
      float m = 0.0f;
      if (ctid < a.ncols)
        for (int w = 0; w < 4; ++w) m = fmaxf(m, smax[w * 64 + ctid]);
      const uint32_t bits = __float_as_uint(m);
      const int E = static_cast<int>((bits >> 23) & 255u);
      int sh = 0;
      if (m > 0.0f && E < 255) sh = min(120, max(-120, 15 - (E == 0 ? -126 : E - 126)));
      scl[ctid] = __uint_as_float(static_cast<uint32_t>(127 + sh) << 23);
      iscl[ctid] = __uint_as_float(static_cast<uint32_t>(127 - sh) << 23);
    }
    xbar();
    // B rows per stage: chunk ch = (column n, 8 elements c8) with Np * 8 <= 128 chunks, so
    // thread ctid owns chunk ctid of every stage; the x of the next kTcPrefetch stages
    // is in flight in registers while this stage waits for its slot and converts
    const bool has_chunk = ctid < Np * 8;
    const int n_own = ctid >> 3, c8_own = ctid & 7;
    const bool live = has_chunk && n_own < a.ncols;
    const float* xcol = a.x + static_cast<int64_t>(live ? n_own : 0) * a.K + st0 * kTcK + 8 * c8_own;
    float4 pre[kTcPrefetch][2];
#pragma unroll
    for (int d = 0; d < kTcPrefetch; ++d)
      if (live && d < nmy) {
        pre[d][0] = reinterpret_cast<const float4*>(xcol + d * kTcK)[0];
        pre[d][1] = reinterpret_cast<const float4*>(xcol + d * kTcK)[1];
      }
    const float sc_own = live ? scl[n_own] : 1.0f;
    bool ok = true;
    for (int i0 = 0; i0 < nmy; i0 += kTcPrefetch) {
#pragma unroll
      for (int d = 0; d < kTcPrefetch; ++d) {  // register slot d holds stage i0 + d
        const int i = i0 + d;
        if (i >= nmy) break;
        const float4 c0 = pre[d][0], c1 = pre[d][1];
        if (live && i + kTcPrefetch < nmy) {
          pre[d][0] = reinterpret_cast<const float4*>(xcol + (i + kTcPrefetch) * kTcK)[0];
          pre[d][1] = reinterpret_cast<const float4*>(xcol + (i + kTcPrefetch) * kTcK)[1];
        }
        const int slot = i % NS, round = i / NS;
        ok = ok && mbar_wait_or_abort(empty0 + 8u * slot, static_cast<uint32_t>((round & 1) ^ 1), abort_flag, a.err);
        if (ok && has_chunk) {
          uint8_t* bt = base + a.off_b + slot * a.b_stage_bytes;
          uint4 hv = make_uint4(0u, 0u, 0u, 0u), lv = make_uint4(0u, 0u, 0u, 0u);
          if (live) {
            const float v[8] = {c0.x * sc_own, c0.y * sc_own, c0.z * sc_own, c0.w * sc_own,
                                c1.x * sc_own, c1.y * sc_own, c1.z * sc_own, c1.w * sc_own};
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const __half h0 = __float2half_rn(v[2 * t]), h1 = __float2half_rn(v[2 * t + 1]);
              const __half l0 = __float2half_rn(v[2 * t] - __half2float(h0));
              const __half l1 = __float2half_rn(v[2 * t + 1] - __half2float(h1));
              hw[t] = static_cast<uint32_t>(__half_as_ushort(h0)) | (static_cast<uint32_t>(__half_as_ushort(h1)) << 16);
              lw[t] = static_cast<uint32_t>(__half_as_ushort(l0)) | (static_cast<uint32_t>(__half_as_ushort(l1)) << 16);
            }
            hv = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            lv = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
          *reinterpret_cast<uint4*>(bt + sw128_offset(n_own, 8 * c8_own)) = hv;
          *reinterpret_cast<uint4*>(bt + sw128_offset(Np + n_own, 8 * c8_own)) = lv;
          fence_proxy_async_smem();  // generic-proxy writes, read by the tensor cores
        }
        mbar_arrive(fullB0 + 8u * slot);
      }
    }
    // epilogue: wait for every MMA (bounded, regardless of an abort: tensor memory is
    // freed below), then this warp's quarter of the accumulator rows
    const bool acc_ok = mbar_wait(accbar, 0);
    if (!acc_ok) set_error(a.err, ERRBIT_TIMEOUT);
    ok = ok && acc_ok && !*abort_flag;
    tc_fence_after();
    const int q = warp & 3;           // TMEM lane quarter this warp can read
    const int r = 32 * q + lane;      // row within the tile
    const int64_t row = static_cast<int64_t>(row0) + r;
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * q) << 16);
    const bool need_aux = (a.epi == EPI_SILU_MUL || a.epi == EPI_ADD);
    for (int c0 = 0; c0 < Np; c0 += 8) {
      float hv[8], lv[8];
      tmem_ld8(trow + static_cast<uint32_t>(c0), hv);
      tmem_ld8(trow + static_cast<uint32_t>(Np + c0), lv);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = c0 + j;
        if (c >= a.ncols) continue;
        const float y = (hv[j] + lv[j]) * iscl[c];
        if constexpr (SPLIT) {
          float* slot = xch + (crank * Np + c) * kTcRows + r;
          if (crank == 0)
            *slot = y;
          else
            st_cluster_f32(map_to_rank(smem_u32(slot), 0), y);
        } else if (ok && row < a.M) {
          const int64_t o = static_cast<int64_t>(c) * a.M + row;
          a.dst[o] = apply_tail(a.epi, y, need_aux ? a.aux[o] : 0.0f);
        }
      }
    }
    if constexpr (SPLIT) {
      if (crank != 0) {
        mbar_arrive_remote(map_to_rank(xchbar, 0));
      } else {
        ok = mbar_wait_cluster_or_abort(xchbar, 0, abort_flag, a.err) && ok;
        if (ok && row < a.M)
          for (int c = 0; c < a.ncols; ++c) {
            float y = 0.0f;
            for (int sl = 0; sl < S; ++sl) y += xch[(sl * Np + c) * kTcRows + r];  // rank order
            const int64_t o = static_cast<int64_t>(c) * a.M + row;
            a.dst[o] = apply_tail(a.epi, y, need_aux ? a.aux[o] : 0.0f);
          }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (SPLIT) cluster_sync_all();  // no CTA leaves while a peer may still store into it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, static_cast<uint32_t>(a.tmem_cols));
  }
}

// ------------------------------------------------------------------ host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime (no link-time
// dependence on the driver library).
static EncodeTiledFn encode_tiled() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

static int round_up_i(int v, int a) { return (v + a - 1) / a * a; }

bool plan_tc(int64_t M, int64_t K, int ncols, int epi, const DeviceLimits& lim, TcPlan& p) {
  if (M < 1 || K < kTcK || K % kTcK != 0 || K > INT32_MAX / 2 || M > INT32_MAX - kTcRows) return false;
  if (ncols < 1 || ncols > kTcMaxCols) return false;
  const int Np = round_up_i(ncols, 8);
  const int nb = 2 * Np;  // MMA N: a multiple of 16 in [16, 128]
  int tmem_cols = 32;
  while (tmem_cols < nb) tmem_cols *= 2;
  const int nst = static_cast<int>(K / kTcK);
  const int64_t tiles = (M + kTcRows - 1) / kTcRows;
  // split K while the tiles leave SMs idle; the exchange holds S * Np * 128 floats
  int S = static_cast<int>(std::min<int64_t>(kMaxSplit, lim.sm_count / std::max<int64_t>(tiles, 1)));
  S = std::min(S, nst);
  S = std::min(S, (64 * 1024) / (Np * kTcRows * 4));
  if (S < 2) S = 1;
  const int xch_bytes = S > 1 ? S * Np * kTcRows * 4 : 0;
  const int off_a = round_up_i(2048 + xch_bytes, 1024);
  const int b_stage = nb * 128;
  const int stage = kTcABytes + b_stage;
  const int avail = lim.smem_optin - 1024 - off_a;  // 1024: alignment slack of the dynamic base
  const int NS = std::min(kTcMaxStages, avail / stage);
  if (NS < 2 || 24 * NS + 24 > 512) return false;
  if (tiles * S > INT32_MAX) return false;
  TcArgs& a = p.a;
  std::memset(&a, 0, sizeof(a));
  a.M = M;
  a.K = static_cast<int>(K);
  a.epi = epi;
  a.ncols = ncols;
  a.Np = Np;
  a.S = S;
  a.nst = nst;
  a.NS = NS;
  a.tmem_cols = tmem_cols;
  a.off_a = off_a;
  a.off_b = off_a + NS * kTcABytes;
  a.b_stage_bytes = b_stage;
  p.grid = static_cast<int>(tiles * S);
  p.smem = 1024 + a.off_b + NS * b_stage;
  return true;
}

template <bool SPLIT>
static int launch_tc_t(const CUtensorMap& map, const TcPlan& p, cudaStream_t st, bool pdl) {
  auto kern = gemv_tc_kernel<SPLIT>;
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && configured[dev] < p.smem) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem);
    if (e != cudaSuccess) return e;
    configured[dev] = p.smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(p.smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (SPLIT) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(p.a.S);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, map, p.a);
}

int launch_tc(const TcPlan& p, const void* W, cudaStream_t st, bool pdl) {
  const EncodeTiledFn enc = encode_tiled();
  if (!enc) return cudaErrorNotSupported;
  alignas(64) CUtensorMap map;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.a.K), static_cast<cuuint64_t>(p.a.M)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.a.K) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kTcK), static_cast<cuuint32_t>(kTcRows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(W), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  return p.a.S > 1 ? launch_tc_t<true>(map, p, st, pdl) : launch_tc_t<false>(map, p, st, pdl);
}

}  // namespace gf
