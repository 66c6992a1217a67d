// Tensor-core GEMV for F16 weights and a batch of columns (5th-generation tensor cores:
// tcgen05.mma with the accumulator in tensor memory).
//
// A CTA owns one tile of 128 rows of W and a slice of its K range.  Per stage of
// 64-element K sub-tiles, warp 0 loads the 128 x 64 f16 tiles of W with 2-D TMA copies
// (128-byte swizzle, K-major: the tensor cores read them straight from shared memory)
// and the batch's x for the same elements (one bulk copy per column up to 8 columns, one
// 2-D copy of all columns beyond), x once the preceding grid, which may write it, has
// finished (the first W stage goes out before that).  Warps 2..5 turn the staged x into
// f16 rows of B in the same swizzled layout.  x is fp32, so each column is scaled by an
// exact power of two (its largest |x| over the CTA's K slice lands in [2^14, 2^15)) and
// split into hi = f16(x) and lo = f16(x - hi): B holds Np rows of hi followed by Np rows
// of lo (Np = columns rounded up to 8).  One thread of warp 1 issues the stage's
// 128 x (2 Np) x 16 MMAs, rotating over four TMEM accumulators, and releases the stage
// with tcgen05.commit.  After the last stage the same four warps read their lane quarter
// of TMEM (one row per thread), form y = (hi part + lo part) * 2^-s, apply the tail and
// write dst.  hi + lo represents x to about 2^-22 relative, products of f16 values are
// exact in fp32 and the accumulation is fp32.
//
// Rows alone give too few tiles for 152 SMs (e.g. 40 for 5120 rows), so K is split over
// a cluster of S CTAs per tile (S = SMs / tiles, at most 8).  Column c of the batch is
// finalised by rank c % S: every rank sends its per-row partial sums of the other ranks'
// columns into their shared memory (st.async, completing bytes on the owner's mbarrier),
// and each owner adds the S partials in rank order (deterministic) and writes its
// columns, so the ranks share the final stores.  Every wait is bounded; on a timeout the
// kernel sets the error word, drains its copies and MMAs, frees its tensor memory and
// returns.
#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "gf_device.cuh"
#include "gf_internal.h"
#include "tc_device.cuh"

namespace gf {

constexpr int kTcRows = 128;                    // rows per tile (MMA M)
constexpr int kTcK = 64;                        // K elements per sub-tile: one 128-byte f16 row
constexpr int kTcKSteps = kTcK / 16;            // MMAs per sub-tile (K = 16 each)
constexpr int kTcThreads = 192;                 // warp 0 TMA, warp 1 MMA, warps 2..5 x / epilogue
constexpr int kTcABytes = kTcRows * kTcK * 2;   // 16 KB per sub-tile (a stage holds a.subs of them)
constexpr int kTcMaxStages = 12;                // W tiles in flight
constexpr int kTcMaxSubs = 4;                   // sub-tiles per stage
// MMA m accumulates into accumulator m % kTcAcc: MMAs into the same TMEM columns wait
// for each other's full latency, which a 128 x N x 16 MMA with small N does not amortise
// (one accumulator held the kernel to ~240 cycles per MMA); the epilogue adds them.
constexpr int kTcAcc = 4;

// ------------------------------------------------------------------ kernel
// Shared memory from a 1024-aligned base: barriers (per stage: W landed, B written, slot
// empty, x landed; the accumulator and exchange barriers) and the TMEM address slot
// [0, 512);
// per-warp column maxima [512, 1536); scales and inverse scales [1536, 2048); the
// split-K exchange [2048, off_a); NS A stages (16 KB each) at off_a; NS B stages at
// off_b (2 Np rows of 128 bytes each).
template <bool SPLIT>
__global__ void __launch_bounds__(kTcThreads, 1) gemv_tc_kernel(const __grid_constant__ CUtensorMap tmap,
                                                                const __grid_constant__ CUtensorMap xmap,
                                                                const TcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t pad = ((raw_s + 1023u) & ~1023u) - raw_s;
  uint8_t* base = smem_raw + pad;
  const uint32_t sb = raw_s + pad;
  const int NS = a.NS;
  const uint32_t fullA0 = sb, fullB0 = sb + 8u * NS, empty0 = sb + 16u * NS;
  const uint32_t accbar = sb + 24u * NS, xchbar = accbar + 8u;
  const uint32_t xfull0 = sb + 24u * NS + 24u;  // NS barriers: a stage's x has landed
  const uint32_t tmemdone = xfull0 + 8u * NS;    // every epilogue thread's TMEM reads are done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + 24 * NS + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + 24 * NS + 20);
  float* smax = reinterpret_cast<float*>(base + 512);   // [4 warps][64] column maxima
  float* scl = reinterpret_cast<float*>(base + 1536);   // [64]
  float* iscl = scl + 64;                               // [64]
  float* xch = reinterpret_cast<float*>(base + 2048);   // [Np][128][SP] partial sums (split K)
  const uint32_t sA = sb + static_cast<uint32_t>(a.off_a), sB = sb + static_cast<uint32_t>(a.off_b);
  const uint32_t sX = sb + static_cast<uint32_t>(a.off_x);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int crank = 0;
  if constexpr (SPLIT) crank = static_cast<int>(cluster_ctarank());
  const int S = SPLIT ? a.S : 1;
  const int row0 = (static_cast<int>(blockIdx.x) / S) * kTcRows;
  const int st0 = crank * a.nst / S, st1 = (crank + 1) * a.nst / S;  // this CTA's K stages
  const int nmy = st1 - st0;
  const int Np = a.Np;
  const int SP = S <= 4 ? 4 : 8;            // exchange slots per (column, row): S rounded up
  const int subs = a.subs;                  // 64-element sub-tiles per stage
  const int b_sub_bytes = 2 * Np * 128;     // B rows of one sub-tile

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmap);
    if (a.ncols > 8) prefetch_tmap(&xmap);
    *abort_flag = 0;
    for (int i = 0; i < NS; ++i) {
      mbar_init(fullA0 + 8u * i, 1);
      mbar_init(xfull0 + 8u * i, 1);
      mbar_init(fullB0 + 8u * i, 128);
      mbar_init(empty0 + 8u * i, 1);
    }
    mbar_init(accbar, 1);
    mbar_init(tmemdone, 128);
    mbar_init(xchbar, 1);
    if constexpr (SPLIT) {  // the partials this CTA receives: S - 1 peers x its columns x 128 rows
      const int nown = a.ncols > crank ? (a.ncols - 1 - crank) / S + 1 : 0;
      mbar_arrive_expect_tx(xchbar, static_cast<uint32_t>((S - 1) * nown * kTcRows * 4));
    }
    fence_mbar_init();
  }
  __syncwarp();  // warp 0 reaches the CTA-wide barrier below converged
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
    // ------------------------------------------------------------ W tiles and x (TMA)
    if (lane == 0) {
      const int xrow = subs * kTcK;  // floats of one column per stage
      // the stage's x: one 2-D copy of every column for wide batches, one bulk copy per
      // column up to 8 columns (measured faster there behind the transform-once prologue)
      const bool x2d = a.ncols > 8;
      // x lands on its own barrier: the converters start on a stage as soon as its x is
      // there (an L2 read) instead of waiting for its W tiles (a DRAM read), and the MMAs
      // find B ready when W lands.  x of stage i goes out after the producer saw the slot
      // empty, so its arrival also tells the converters that the slot's B is free.
      auto issue_x = [&](int i, int slot) {
        const uint32_t xb = xfull0 + 8u * slot;
        mbar_arrive_expect_tx(xb, static_cast<uint32_t>(a.ncols * xrow * 4));
        if (x2d) {
          tma_load_2d(sX + static_cast<uint32_t>(slot * a.x_stage_bytes), &xmap, (st0 + i) * xrow, 0, xb);
        } else {
          for (int c = 0; c < a.ncols; ++c)
            bulk_g2s(sX + static_cast<uint32_t>(slot * a.x_stage_bytes + c * xrow * 4),
                     a.x + static_cast<int64_t>(c) * a.K + static_cast<int64_t>(st0 + i) * xrow,
                     static_cast<uint32_t>(xrow * 4), xb);
        }
      };
      int issued = 0, x_done = 0;  // stages whose W / x copies are out
      bool waited = false;
      // slot = i % NS and the phase parity (i / NS) & 1, kept incrementally (no division
      // on the issue path)
      for (int i = 0, slot = 0, par = 0; i < nmy; ++i, slot = (slot + 1 == NS) ? 0 : slot + 1, par ^= (slot == 0)) {
        // the first NS stages are empty: no wait (see the stream kernel)
        if (i >= NS && !mbar_wait_or_abort(empty0 + 8u * slot, static_cast<uint32_t>(par ^ 1), abort_flag, a.err))
          break;
        mbar_arrive_expect_tx(fullA0 + 8u * slot, static_cast<uint32_t>(subs * kTcABytes));
        for (int sbt = 0; sbt < subs; ++sbt)
          tma_load_2d(sA + static_cast<uint32_t>((slot * subs + sbt) * kTcABytes), &tmap,
                      ((st0 + i) * subs + sbt) * kTcK, row0, fullA0 + 8u * slot);
        ++issued;
        if (!waited) {  // first W stage out: now x, once the preceding grid has finished
          pdl_wait();
          waited = true;
        }
        if (waited)
          for (; x_done < issued; ++x_done) issue_x(x_done, x_done == i ? slot : x_done % NS);
      }
      if (issued < nmy) {  // aborted: complete the stages' x, then wait (bounded) for the copies in flight
        if (!waited) pdl_wait();
        for (; x_done < issued; ++x_done) issue_x(x_done, x_done % NS);
        for (int i = max(0, issued - NS); i < issued; ++i) {
          (void)mbar_wait(fullA0 + 8u * (i % NS), static_cast<uint32_t>((i / NS) & 1));
          (void)mbar_wait(xfull0 + 8u * (i % NS), static_cast<uint32_t>((i / NS) & 1));
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_f16(kTcRows, 2 * Np);
      const uint32_t acc_cols = static_cast<uint32_t>(2 * Np);
      for (int i = 0, slot = 0, par = 0; i < nmy; ++i, slot = (slot + 1 == NS) ? 0 : slot + 1, par ^= (slot == 0)) {
        if (!mbar_wait_or_abort(fullA0 + 8u * slot, static_cast<uint32_t>(par), abort_flag, a.err)) break;
        if (!mbar_wait_or_abort(fullB0 + 8u * slot, static_cast<uint32_t>(par), abort_flag, a.err)) break;
        tc_fence_after();
        for (int sbt = 0; sbt < subs; ++sbt) {
          const uint64_t da = umma_desc_sw128(sA + static_cast<uint32_t>((slot * subs + sbt) * kTcABytes));
          const uint64_t db =
              umma_desc_sw128(sB + static_cast<uint32_t>(slot * a.b_stage_bytes + sbt * b_sub_bytes));
#pragma unroll
          for (int kk = 0; kk < kTcKSteps; ++kk) {  // +32 bytes of K per step inside the swizzled rows
            const int m = (i * subs + sbt) * kTcKSteps + kk;
            umma_f16(tmem + static_cast<uint32_t>(m % kTcAcc) * acc_cols, da + 2u * kk, db + 2u * kk, idesc,
                     m >= kTcAcc ? 1u : 0u);
          }
        }
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
    // CTA's K slice, eight columns per pass so their loads are in flight together (under
    // the weight stream an L2 round trip takes ~1-2 us)
    const int k0 = st0 * subs * kTcK, klen4 = nmy * subs * kTcK / 4;
    for (int n0 = 0; n0 < a.ncols; n0 += 8) {
      float m[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 4
      for (int i = ctid; i < klen4; i += 128) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (n0 + u < a.ncols) {
            const float4 v = reinterpret_cast<const float4*>(a.x + static_cast<int64_t>(n0 + u) * a.K + k0)[i];
            m[u] = fmaxf(m[u], fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
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
    // thread ctid owns chunk ctid of every sub-tile; a stage's x lands with its W tile
    // (same barrier), by which time the MMAs that read the slot's previous B are done
    const bool has_chunk = ctid < Np * 8;
    const int n_own = ctid >> 3, c8_own = ctid & 7;
    const bool live = has_chunk && n_own < a.ncols;
    const float sc_own = live ? scl[n_own] : 1.0f;
    const uint32_t sw_hi = sw128_offset(n_own, 8 * c8_own), sw_lo = sw128_offset(Np + n_own, 8 * c8_own);
    bool ok = true;
    // per stage: one wait, the loads of every sub-tile in flight together, then the
    // conversions and stores (one warp per SM sub-partition runs this, so independent
    // work is what hides the latencies); ring slot and phase kept incrementally
    for (int i = 0, slot = 0, par = 0; i < nmy; ++i, slot = (slot + 1 == NS) ? 0 : slot + 1, par ^= (slot == 0)) {
      ok = ok && mbar_wait_or_abort(xfull0 + 8u * slot, static_cast<uint32_t>(par), abort_flag, a.err);
      float4 c[kTcMaxSubs][2];
      const float* xs = reinterpret_cast<const float*>(base + a.off_x + slot * a.x_stage_bytes) +
                        n_own * subs * kTcK + 8 * c8_own;
#pragma unroll
      for (int sbt = 0; sbt < kTcMaxSubs; ++sbt) {
        c[sbt][0] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        c[sbt][1] = c[sbt][0];
        if (sbt < subs && ok && live) {
          c[sbt][0] = reinterpret_cast<const float4*>(xs + sbt * kTcK)[0];
          c[sbt][1] = reinterpret_cast<const float4*>(xs + sbt * kTcK)[1];
        }
      }
      if (ok && has_chunk) {
        uint8_t* bt = base + a.off_b + slot * a.b_stage_bytes;
#pragma unroll
        for (int sbt = 0; sbt < kTcMaxSubs; ++sbt) {
          if (sbt >= subs) break;
          // hi = f16(x * 2^s), lo = f16(x * 2^s - hi), two elements per conversion (zero
          // rows for the padding columns)
          const float2 sc2 = make_float2(sc_own, sc_own);
          const float2 v[4] = {fmul2(make_float2(c[sbt][0].x, c[sbt][0].y), sc2),
                               fmul2(make_float2(c[sbt][0].z, c[sbt][0].w), sc2),
                               fmul2(make_float2(c[sbt][1].x, c[sbt][1].y), sc2),
                               fmul2(make_float2(c[sbt][1].z, c[sbt][1].w), sc2)};
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const __half2 h = __floats2half2_rn(v[t].x, v[t].y);
            const float2 rr = fsub2(v[t], __half22float2(h));
            const __half2 l = __floats2half2_rn(rr.x, rr.y);
            hw[t] = *reinterpret_cast<const uint32_t*>(&h);
            lw[t] = *reinterpret_cast<const uint32_t*>(&l);
          }
          *reinterpret_cast<uint4*>(bt + sbt * b_sub_bytes + sw_hi) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(bt + sbt * b_sub_bytes + sw_lo) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        fence_proxy_async_smem();  // generic-proxy writes, read by the tensor cores
      }
      mbar_arrive(fullB0 + 8u * slot);
    }
    // This thread's epilogue row (TMEM lane quarter of its warp).  Column c is finalised
    // by cluster rank c % S: own_tbl holds that rank in 4 bits per column, `mine` flags
    // this CTA's columns (a chain of compares: the epilogue runs one warp per SM
    // sub-partition, where every dependent instruction is paid in full, so integer
    // division stays out of it).  Their aux values are loaded here, before the wait for
    // the last MMAs hides their latency (at the start they would delay the scale pass;
    // in the tail each would wait behind the previous column's dst store, as dst may
    // alias aux).
    const int q = warp & 3;           // TMEM lane quarter this warp can read
    const int r = 32 * q + lane;      // row within the tile
    const int64_t row = static_cast<int64_t>(row0) + r;
    const bool need_aux = (a.epi == EPI_SILU_MUL || a.epi == EPI_ADD);
    uint64_t own_tbl = 0;
    uint32_t mine = 0;
    {
      int o = 0;
#pragma unroll
      for (int c = 0; c < kTcMaxCols; ++c) {
        own_tbl |= static_cast<uint64_t>(o) << (4 * c);
        if (o == crank && c < a.ncols) mine |= 1u << c;
        o = (o + 1 == S) ? 0 : o + 1;
      }
    }
    float auxv[kTcMaxCols];
#pragma unroll
    for (int c = 0; c < kTcMaxCols; ++c) {
      auxv[c] = 0.0f;
      if (need_aux && ((mine >> c) & 1u) && row < a.M) auxv[c] = a.aux[static_cast<int64_t>(c) * a.M + row];
    }
    // epilogue: wait for every MMA (bounded, regardless of an abort: tensor memory is
    // freed below), then this warp's quarter of the accumulator rows
    const bool acc_ok = mbar_wait(accbar, 0);
    if (!acc_ok) set_error(a.err, ERRBIT_TIMEOUT);
    ok = ok && acc_ok && !*abort_flag;
    tc_fence_after();
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * q) << 16);
    const int nacc = min(kTcAcc, nmy * subs * kTcKSteps);  // accumulators written
    float* const dcol = a.dst + row;                         // column c at dcol[c * M]
    const bool plain_add = a.epi == EPI_ADD;
#pragma unroll
    for (int c0 = 0; c0 < kTcMaxCols; c0 += 8) {
      if (c0 >= Np) break;
      // all accumulators of these 8 columns (hi and lo) in flight, then one wait
      uint32_t hr[kTcAcc][8], lr[kTcAcc][8];
#pragma unroll
      for (int t = 0; t < kTcAcc; ++t)
        if (t < nacc) {
          tmem_ld8_nowait(trow + static_cast<uint32_t>(t * 2 * Np + c0), hr[t]);
          tmem_ld8_nowait(trow + static_cast<uint32_t>(t * 2 * Np + Np + c0), lr[t]);
        }
      tmem_wait_ld();
      float hv[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
      float lv[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int t = 0; t < kTcAcc; ++t)  // the accumulators, in order
        if (t < nacc) {
          tmem_pin8(hr[t]);
          tmem_pin8(lr[t]);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            hv[j] += __uint_as_float(hr[t][j]);
            lv[j] += __uint_as_float(lr[t][j]);
          }
        }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = c0 + j;
        if (c >= a.ncols) break;
        const float y = (hv[j] + lv[j]) * iscl[c];
        if constexpr (SPLIT) {  // this rank's partial, into the exchange of the column's owner
          const uint32_t own = static_cast<uint32_t>(own_tbl >> (4 * c)) & 15u;
          float* slot = xch + (c * kTcRows + r) * SP + crank;
          if (own == static_cast<uint32_t>(crank))
            *slot = y;
          else
            st_async_f32(map_to_rank(smem_u32(slot), own), y, map_to_rank(xchbar, own));
        } else if (ok && row < a.M) {
          dcol[static_cast<int64_t>(c) * a.M] = plain_add ? y + auxv[c] : apply_tail(a.epi, y, auxv[c]);
        }
      }
    }
    // the tensor memory may be freed once every epilogue thread is past its reads (an
    // explicit barrier: the freeing warp does not rely on the CTA-wide one below)
    tc_fence_before();
    mbar_arrive(tmemdone);
    if constexpr (SPLIT) {
      // wait until every peer's partials of this CTA's columns have landed, then add the
      // S partials of each column in rank order and apply the tail
      ok = mbar_wait_cluster_or_abort(xchbar, 0, abort_flag, a.err) && ok;
      if (ok && row < a.M) {
        float yv[kTcMaxCols];
#pragma unroll
        for (int c = 0; c < kTcMaxCols; ++c) {
          yv[c] = 0.0f;
          if ((mine >> c) & 1u) {
            const float4* pp = reinterpret_cast<const float4*>(xch + (c * kTcRows + r) * SP);
            const float4 p0 = pp[0];
            yv[c] = (0.0f + p0.x) + p0.y;  // S >= 2 here
            if (S >= 3) yv[c] += p0.z;
            if (S >= 4) yv[c] += p0.w;
            if (S >= 5) {
              const float4 p1 = pp[1];
              yv[c] += p1.x;
              if (S >= 6) yv[c] += p1.y;
              if (S >= 7) yv[c] += p1.z;
              if (S >= 8) yv[c] += p1.w;
            }
          }
        }
        if (plain_add) {
#pragma unroll
          for (int c = 0; c < kTcMaxCols; ++c)
            if ((mine >> c) & 1u) dcol[static_cast<int64_t>(c) * a.M] = yv[c] + auxv[c];
        } else {
#pragma unroll
          for (int c = 0; c < kTcMaxCols; ++c)
            if ((mine >> c) & 1u) dcol[static_cast<int64_t>(c) * a.M] = apply_tail(a.epi, yv[c], auxv[c]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (SPLIT) cluster_sync_all();  // no CTA leaves while a peer may still store into it
  if (warp == 1) {
    (void)mbar_wait(tmemdone, 0u);  // bounded; every epilogue thread arrives, also after an abort
    __syncwarp();                    // the dealloc is a warp-wide instruction
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

// Clusters of S CTAs of the split kernel that can be resident at once (0 if the device
// cannot be asked): a cluster's CTAs share a GPC, so clusters of S may fit fewer times
// than SMs / S.  Every plan holds one CTA per SM; the answer is kept per device and S.
// The query raises the kernel's shared-memory limit to the device maximum, which keeps
// every later launch's own (smaller) setting valid.
static int tc_max_clusters(int S, int smem_max) {
  static int cache[64][kMaxSplit + 1];
  static bool init[64][kMaxSplit + 1];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || S < 2 || S > kMaxSplit) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (init[dev][S]) return cache[dev][S];
  int n = 0;
  auto kern = gemv_tc_kernel<true>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S * 64);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = 160 * 1024;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  cache[dev][S] = n;
  init[dev][S] = true;
  return n;
}

bool plan_tc(int64_t M, int64_t K, int ncols, int epi, const DeviceLimits& lim, TcPlan& p) {
  if (M < 1 || K < kTcK || K % kTcK != 0 || K > INT32_MAX / 2 || M > INT32_MAX - kTcRows) return false;
  if (ncols < 1 || ncols > kTcMaxCols) return false;
  const int Np = round_up_i(ncols, 8);
  const int nb = 2 * Np;  // MMA N: a multiple of 16 in [16, 32]
  int tmem_cols = 32;
  while (tmem_cols < kTcAcc * nb) tmem_cols *= 2;  // kTcAcc accumulators of nb columns
  const int64_t tiles = (M + kTcRows - 1) / kTcRows;
  // split K while the tiles leave SMs idle; the exchange holds S * Np * 128 floats
  const int nsub_all = static_cast<int>(K / kTcK);
  int S = static_cast<int>(std::min<int64_t>(kMaxSplit, lim.sm_count / std::max<int64_t>(tiles, 1)));
  S = std::min(S, nsub_all);
  while (S >= 2 && Np * kTcRows * 4 * (S <= 4 ? 4 : 8) > 64 * 1024) --S;
  while (S >= 2) {  // every cluster resident at once (when the device can say)
    const int fit = tc_max_clusters(S, lim.smem_optin);
    if (fit == 0 || tiles <= fit) break;
    --S;
  }
  if (S < 2) S = 1;
  const int xch_bytes = S > 1 ? Np * kTcRows * 4 * (S <= 4 ? 4 : 8) : 0;
  const int off_a = round_up_i(2048 + xch_bytes, 1024);
  const int avail = lim.smem_optin - 1024 - off_a;  // 1024: alignment slack of the dynamic base
  // stages of `subs` sub-tiles: the MMA thread's per-stage cost (its waits and commits) is
  // spread over more data; the widest that divides K, gives every split rank a stage and
  // keeps at least three stages in flight
  int subs = 1, NS = 0;
  for (int cand = 4; cand >= 1; cand /= 2) {
    if (nsub_all % cand != 0 || nsub_all / cand < S) continue;
    const int ns = std::min(kTcMaxStages, avail / (cand * (kTcABytes + nb * 128 + ncols * kTcK * 4)));
    if (ns >= 3 || cand == 1) {
      subs = cand;
      NS = ns;
      break;
    }
  }
  if (NS < 2 || 32 * NS + 32 > 512) return false;
  if (tiles * S > INT32_MAX) return false;
  TcArgs& a = p.a;
  std::memset(&a, 0, sizeof(a));
  a.M = M;
  a.K = static_cast<int>(K);
  a.epi = epi;
  a.ncols = ncols;
  a.Np = Np;
  a.S = S;
  a.subs = subs;
  a.nst = nsub_all / subs;
  a.NS = NS;
  a.tmem_cols = tmem_cols;
  a.off_a = off_a;
  a.off_b = off_a + NS * subs * kTcABytes;
  a.b_stage_bytes = subs * nb * 128;
  a.off_x = a.off_b + NS * a.b_stage_bytes;
  a.x_stage_bytes = subs * ncols * kTcK * 4;
  p.grid = static_cast<int>(tiles * S);
  p.smem = 1024 + a.off_x + NS * a.x_stage_bytes;
  return true;
}

template <bool SPLIT>
static int launch_tc_t(const CUtensorMap& map, const CUtensorMap& xmap, const TcPlan& p, cudaStream_t st, bool pdl) {
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
  return cudaLaunchKernelEx(&cfg, kern, map, xmap, p.a);
}

int encode_map_2d(CUtensorMap* map, int dtype, const void* base, uint64_t inner, uint64_t rows, uint64_t stride_bytes,
                  uint32_t box_inner, uint32_t box_rows, bool swizzle128) {
  const EncodeTiledFn enc = encode_tiled();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(stride_bytes)};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map,
                         dtype == kMapF16   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                         : dtype == kMapF32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                            : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                         2,
                         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Encoded tensor maps of recent operands: a map holds only the address, shape, stride
// and box, so an entry with the same key is always the right one.
namespace {
struct MapEntry {
  const void* base;
  uint64_t inner, rows;
  uint32_t box_inner, box_rows;
  int dtype;
  CUtensorMap map;  // the type carries the 64-byte alignment the driver requires
};
constexpr int kMapCache = 64;
std::mutex g_map_mu;
MapEntry g_maps[kMapCache];
int g_map_used = 0, g_map_next = 0;
}  // namespace

// A dense row-major [rows][inner] operand (rows `inner` elements apart).
static int cached_map(const void* base, int dtype, uint64_t inner, uint64_t rows, uint32_t box_inner,
                      uint32_t box_rows, bool swizzle128, CUtensorMap* out) {
  std::lock_guard<std::mutex> lock(g_map_mu);
  for (int i = 0; i < g_map_used; ++i) {
    const MapEntry& e = g_maps[i];
    if (e.base == base && e.dtype == dtype && e.inner == inner && e.rows == rows && e.box_inner == box_inner &&
        e.box_rows == box_rows) {
      *out = e.map;
      return cudaSuccess;
    }
  }
  const uint64_t esize = dtype == kMapF32 ? 4 : dtype == kMapF16 ? 2 : 1;
  CUtensorMap fresh;
  const int r = encode_map_2d(&fresh, dtype, base, inner, rows, inner * esize, box_inner, box_rows, swizzle128);
  if (r != cudaSuccess) return r;
  MapEntry& e = g_maps[g_map_next];
  e.map = fresh;
  e.base = base;
  e.dtype = dtype;
  e.inner = inner;
  e.rows = rows;
  e.box_inner = box_inner;
  e.box_rows = box_rows;
  *out = e.map;
  g_map_next = (g_map_next + 1) % kMapCache;
  if (g_map_used < kMapCache) ++g_map_used;
  return cudaSuccess;
}

int launch_tc(const TcPlan& p, const void* W, cudaStream_t st, bool pdl) {
  CUtensorMap wmap, xmap;  // the type carries the 64-byte alignment the driver requires
  // W: 128 x 64 f16 boxes, 128-byte swizzle; x (beyond 8 columns): [ncols][K] fp32, one
  // stage of every column
  int e = cached_map(W, kMapF16, static_cast<uint64_t>(p.a.K), static_cast<uint64_t>(p.a.M), kTcK, kTcRows, true,
                     &wmap);
  if (e != cudaSuccess) return e;
  std::memset(&xmap, 0, sizeof(xmap));  // unused up to 8 columns
  if (p.a.ncols > 8) {
    e = cached_map(p.a.x, kMapF32, static_cast<uint64_t>(p.a.K), static_cast<uint64_t>(p.a.ncols),
                   static_cast<uint32_t>(p.a.subs * kTcK), static_cast<uint32_t>(p.a.ncols), false, &xmap);
    if (e != cudaSuccess) return e;
  }
  return p.a.S > 1 ? launch_tc_t<true>(wmap, xmap, p, st, pdl) : launch_tc_t<false>(wmap, xmap, p, st, pdl);
}

}  // namespace gf
