// TMA-streamed persistent GEMV with fused prologue/epilogue.
//
// One CTA per SM owns a contiguous range of rows (whole tiles when every CTA gets one,
// the remainder to the lowest block indices, which a launch behind another starts
// first).  Warp 0 is the producer: one lane streams the CTA's weight bytes, tile by
// tile (R rows x one K chunk), into a ring of shared-memory stages with 1-D bulk async
// copies (no multicast), signalling a "full" mbarrier per stage.  Warps 1..ncw are
// consumers: each thread owns fixed 16-weight units of the K chunk and keeps the
// matching x in registers while it walks the R rows of a stage, issuing every row's
// shared-memory loads before the arithmetic.  F32/F16 (and batched block formats)
// decode to floats and accumulate with packed f32x2 FMAs; single-column Q8_0, Q4_0 and
// Q4_K take exact integer dot products (dp4a) against x held as 24-bit integers with a
// shared exponent per unit.  Per tile, each warp reduces its per-row partial sums with
// shuffles and stores them to shared memory; after the last K chunk the partials of
// the consumer warps are added in a fixed order (deterministic), the fused tail is
// applied with the prefetched aux operand, and dst is written once.
//
// x: when a row fits one K chunk, the producer stages x (all columns) in shared memory
// with a bulk copy issued right behind the first weight tile; otherwise each consumer
// loads its x values from global memory.
//
// Prologues: with the signed FWHT, x (all columns of one K chunk) is staged in shared
// memory with a bulk copy and transformed in place, so x' never leaves the chip.  With
// RMS normalisation, gamma multiplies x as it is loaded into registers and the
// per-column 1/rms scales the finished dot product before the tail; the sum of squares
// is taken from the same register loads during the first row chunk (each column
// group's threads together load every x value of a chunk exactly once) and reduced in
// a fixed order with the row sums.
//
// Gated dual GEMV: every tile holds h rows of the gate matrix followed by the same h
// rows of the up matrix ("virtual rows"), and the tail is silu(gate) * up.
//
// Several matrices sharing x (nseg > 0): their rows are streamed as one matrix; tile
// copies are cut at matrix boundaries and each row's tail, aux and dst are its matrix's.
//
// Split K: with S > 1 the grid is made of clusters of S CTAs; the CTAs of a cluster
// share one row range and each takes a slice of its K chunks.  The per-row partial
// sums of ranks 1..S-1 are stored into rank 0's shared memory (distributed shared
// memory), rank 0 adds the S slices in rank order (deterministic) and applies the tail.
//
// Each (format, columns) pair is compiled three times (FEAT): the plain GEMV, the
// extended one (dual GEMV, several matrices, RMS prologue) and the split-K one
// (clusters, with the same extensions).  The plain kernel carries none of the
// extension code: cluster instructions in a kernel image alone add about a
// microsecond per launch on GB300.
//
// Every wait is bounded; a timeout sets the device error word and the kernel returns
// after draining its own copies.
#pragma once

#include "gf_device.cuh"
#include "gf_internal.h"

namespace gf {

// Segment of virtual row r of a multi-matrix launch (a.nseg > 0) and the row's index in it.
__device__ __forceinline__ int seg_of(const StreamArgs& a, int64_t r, int64_t& local) {
  int i = 0;
#pragma unroll
  for (int k = 0; k < kMaxSeg - 1; ++k)
    if (k < a.nseg - 1 && r >= a.seg_end[i]) ++i;
  local = r - (i ? a.seg_end[i - 1] : 0);
  return i;
}

template <int WT>
__host__ __device__ constexpr int seg_bytes_of(int klen) {
  return WT == WT_F32    ? 4 * klen
         : WT == WT_F16  ? 2 * klen
         : WT == WT_Q8_0 ? (klen / 32) * 34
         : WT == WT_Q4_0 ? (klen / 32) * 18
                         : (klen / 256) * 144;
}

// Unit i (< U) of the thread at position tg (of tg_n) in its column group: strided over
// the chunk, except Q4_K, whose two units are the pair sharing one code load.
template <int WT, int U>
__device__ __forceinline__ int unit_index(int tg, int i, int tg_n) {
  if constexpr (WT == WT_Q4_K) {
    static_assert(U == 2, "Q4_K threads own one unit pair");
    return 2 * tg + i;
  } else {
    return tg + i * tg_n;
  }
}

// x values of one unit for the thread's NCT columns (starting at column c0; columns
// past the batch are zero) as eight float2 pairs each, in decode_unit()'s pair order.
// xs is either the K chunk staged in shared memory (column stride xstride) or x itself
// in global memory (column stride K, offset to the chunk); both are read with 16-byte
// loads.
// With GAMMA, each x value is multiplied by the RMS-normalisation weight at the same
// element (gsrc: the weight at the chunk's offset) as it is loaded, and (with SQ) its
// square is added to ssq[c] first.
template <int WT, int NCT, bool GAMMA>
__device__ __forceinline__ void load_unit_x(const float* xs, int64_t xstride, const float* gsrc, int u, uint32_t qr,
                                            int c0, int nc, float2 (&xv)[NCT][8], bool sq = false,
                                            float* ssq = nullptr) {
  if constexpr (!GAMMA) {
#pragma unroll
    for (int c = 0; c < NCT; ++c) {
      const bool live = (c0 + c) < nc;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float4 t = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (live)
          t = *reinterpret_cast<const float4*>(
              xs + (c0 + c) * xstride + unit_pair_elem<WT>(static_cast<uint32_t>(u), 2 * static_cast<int>((q + qr) & 3u)));
        xv[c][2 * q] = make_float2(t.x, t.y);
        xv[c][2 * q + 1] = make_float2(t.z, t.w);
      }
    }
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t e = unit_pair_elem<WT>(static_cast<uint32_t>(u), 2 * static_cast<int>((q + qr) & 3u));
      const float4 gm = *reinterpret_cast<const float4*>(gsrc + e);
#pragma unroll
      for (int c = 0; c < NCT; ++c) {
        float4 t = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if ((c0 + c) < nc) t = *reinterpret_cast<const float4*>(xs + (c0 + c) * xstride + e);
        if (sq) {
          ssq[c] = fmaf(t.x, t.x, ssq[c]);
          ssq[c] = fmaf(t.y, t.y, ssq[c]);
          ssq[c] = fmaf(t.z, t.z, ssq[c]);
          ssq[c] = fmaf(t.w, t.w, ssq[c]);
        }
        t.x *= gm.x; t.y *= gm.y; t.z *= gm.z; t.w *= gm.w;
        xv[c][2 * q] = make_float2(t.x, t.y);
        xv[c][2 * q + 1] = make_float2(t.z, t.w);
      }
    }
  }
}

// acc[c] += sum of the unit's 16 products for each of the thread's columns (quant
// formats: the block partial first, then scaled by d into the running sum).
template <int WT, int NCT>
__device__ __forceinline__ void unit_rows_fma(const float2 (&v)[8], float d, const float2 (&xv)[NCT][8],
                                              float2 (&acc)[NCT]) {
#pragma unroll
  for (int c = 0; c < NCT; ++c) {
    if constexpr (WT == WT_F32 || WT == WT_F16) {
      float2 t = acc[c];
#pragma unroll
      for (int k = 0; k < 8; ++k) t = ffma2(v[k], xv[c][k], t);
      acc[c] = t;
    } else {
      float2 p0 = make_float2(0.0f, 0.0f), p1 = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int k = 0; k < 8; k += 2) {
        p0 = ffma2(v[k], xv[c][k], p0);
        p1 = ffma2(v[k + 1], xv[c][k + 1], p1);
      }
      acc[c] = ffma2(make_float2(d, d), fadd2(p0, p1), acc[c]);
    }
  }
}

// One thread's share of a tile: U units (16 weights each, stride tg_n within the
// column group) times RT rows (stride G within the tile), against x in registers.
// Q4_K: per row, one decode of the thread's unit pair; the scaled-code term through
// packed FMAs, the min term through the units' sums of x (xsum).
template <int NCT, int RT>
__device__ __forceinline__ void consume_tile_q4k(uint32_t st, int seg, int rows, int units, int tg, int g, int G,
                                                 const float2 (&xr)[2][NCT][8], const float (&xsum)[2][NCT],
                                                 float2 (&acc)[RT][NCT]) {
  if (2 * tg >= units) return;
#pragma unroll
  for (int j = 0; j < RT; ++j) {
    const int r = g + j * G;
    if (r < rows) {
      const SmemLoader ld{st + static_cast<uint32_t>(r * seg)};
      float dsc[2], dmn[2];
      const uint4 q = q4k_load_pair(ld, static_cast<uint32_t>(tg), dsc, dmn);
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        float2 v[8];
        q4k_nibbles(q, static_cast<uint32_t>(n), v);
#pragma unroll
        for (int c = 0; c < NCT; ++c) {
          float2 p0 = make_float2(0.0f, 0.0f), p1 = make_float2(0.0f, 0.0f);
#pragma unroll
          for (int k = 0; k < 8; k += 2) {
            p0 = ffma2(v[k], xr[n][c][k], p0);
            p1 = ffma2(v[k + 1], xr[n][c][k + 1], p1);
          }
          float2 t = ffma2(make_float2(dsc[n], dsc[n]), fadd2(p0, p1), acc[j][c]);
          t.x = fmaf(-dmn[n], xsum[n][c], t.x);
          acc[j][c] = t;
        }
      }
    }
  }
}

// Q4_K through integer dot products: per row, one 16-byte code load and one unpack of the
// scales for the thread's unit pair; each unit's nibbles against its XInt, scaled by
// d * sc[j] * 2^-s, and the min term through the unit's sum of x.  Every row's loads
// come first, as in consume_tile_int.
template <int RT>
__device__ __forceinline__ void consume_tile_q4k_int(uint32_t st, int seg, int rows, int units, int tg, int g,
                                                     int G, const XInt (&xq)[2][1], const float (&xsum)[2][1],
                                                     float2 (&acc)[RT][1]) {
  if (2 * tg >= units) return;
  const uint32_t p = static_cast<uint32_t>(tg), pp = p & 7u, gq = pp >> 1;
  const uint32_t boff = (p >> 3) * kQ4kBytes;
  uint32_t hdr[RT], sw[RT][3];
  uint4 q[RT];
#pragma unroll
  for (int j = 0; j < RT; ++j) {
    const int r = min(g + j * G, rows - 1);
    const SmemLoader ld{st + static_cast<uint32_t>(r * seg)};
    hdr[j] = ld.word(boff);
#pragma unroll
    for (int k = 0; k < 3; ++k) sw[j][k] = ld.word(boff + 4u + 4u * k);
    q[j] = ld.quad(boff + 16u + 16u * pp);
  }
#pragma unroll
  for (int j = 0; j < RT; ++j) {
    float dsc[2], dmn[2];
    q4k_scales_from(hdr[j], sw[j][0], sw[j][1], sw[j][2], gq, dsc, dmn);
    const uint32_t w[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      uint32_t nb[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) nb[k] = (w[k] >> (4u * n)) & 0x0F0F0F0Fu;
      const XInt (&xn)[1] = xq[n];
      int t[1];
      nibble_words_int<1, false>(nb, xn, t);
      float a = fmaf(dsc[n] * xq[n][0].sc, static_cast<float>(t[0]), acc[j][0].x);
      acc[j][0].x = fmaf(-dmn[n], xsum[n][0], a);
    }
  }
}

// Q4_0 / Q8_0 through integer dot products: per row, the unit's codes against each
// column's XInt; the block scale d times 2^-s scales the exact integer sum.  All rows'
// shared-memory words are loaded before any arithmetic (the loads are ordered asm, so
// this leaves the scheduler every row's dp4a chains to interleave); rows past the tile's
// end read its last row and their sums are never stored.
template <int WT, int NCT, int U, int RT>
__device__ __forceinline__ void consume_tile_int(uint32_t st, int seg, int rows, int units, int tg, int tg_n,
                                                 int g, int G, const XInt (&xq)[U][NCT], float2 (&acc)[RT][NCT]) {
  constexpr bool kQ8 = WT == WT_Q8_0;
  constexpr uint32_t kBlk = kQ8 ? 34u : 18u, kHalf = kQ8 ? 16u : 8u;
  constexpr int kW = kQ8 ? 5 : 3;  // aligned words covering the unit's code bytes
#pragma unroll
  for (int i = 0; i < U; ++i) {
    const uint32_t u = static_cast<uint32_t>(tg + i * tg_n);
    if (u < static_cast<uint32_t>(units)) {
      const uint32_t off = (u >> 1) * kBlk, start = off + 2u + kHalf * (u & 1u);
      const uint32_t wa = start & ~3u, sh = (start & 3u) * 8u;
      uint32_t dr[RT], wr[RT][kW];
#pragma unroll
      for (int j = 0; j < RT; ++j) {
        const int r = min(g + j * G, rows - 1);
        const SmemLoader ld{st + static_cast<uint32_t>(r * seg)};
        dr[j] = ld.u16(off);
#pragma unroll
        for (int k = 0; k < kW; ++k) wr[j][k] = ld.u32(wa + 4u * k);
      }
#pragma unroll
      for (int j = 0; j < RT; ++j) {
        float t[NCT];
        if constexpr (kQ8) {
          uint32_t w[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) w[k] = __funnelshift_r(wr[j][k], wr[j][k + 1], sh);
          q8_0_words_int<NCT>(w, xq[i], t);
        } else {
          int ti[NCT];
          q4_0_words_int<NCT>(__funnelshift_r(wr[j][0], wr[j][1], sh), __funnelshift_r(wr[j][1], wr[j][2], sh),
                              xq[i], ti);
#pragma unroll
          for (int c = 0; c < NCT; ++c) t[c] = static_cast<float>(ti[c]);
        }
        const float d = h2f(dr[j]);
#pragma unroll
        for (int c = 0; c < NCT; ++c) acc[j][c].x = fmaf(d * xq[i][c].sc, t[c], acc[j][c].x);
      }
    }
  }
}

// BATCH: load every row's raw unit before any arithmetic (else row by row; F32 always
// goes row by row).
template <int WT, int NCT, int U, int RT, bool BATCH>
__device__ __forceinline__ void consume_tile(uint32_t st, int seg, int rows, int units, int tg, int tg_n,
                                             int g, int G, uint32_t qr, const float2 (&xr)[U][NCT][8],
                                             float2 (&acc)[RT][NCT]) {
#pragma unroll
  for (int i = 0; i < U; ++i) {
    const int u = tg + i * tg_n;
    if (u < units) {
      if constexpr (WT == WT_F32 || !BATCH) {
#pragma unroll
        for (int j = 0; j < RT; ++j) {
          const int r = g + j * G;
          if (r < rows) {
            const SmemLoader ld{st + static_cast<uint32_t>(r * seg)};
            float2 v[8];
            float d;
            decode_unit<WT>(ld, static_cast<uint32_t>(u), v, d, qr);
            unit_rows_fma<WT, NCT>(v, d, xr[i], acc[j]);
          }
        }
      } else {
        // every row's loads first (rows past the tile's end read its last row; their
        // sums are never stored), then the arithmetic
        RawUnit<WT> raw[RT];
#pragma unroll
        for (int j = 0; j < RT; ++j) {
          const int r = min(g + j * G, rows - 1);
          load_raw<WT>(SmemLoader{st + static_cast<uint32_t>(r * seg)}, static_cast<uint32_t>(u), qr, raw[j]);
        }
#pragma unroll
        for (int j = 0; j < RT; ++j) {
          float2 v[8];
          float d;
          decode_raw<WT>(raw[j], static_cast<uint32_t>(u), v, d);
          unit_rows_fma<WT, NCT>(v, d, xr[i], acc[j]);
        }
      }
    }
  }
}

// Rows [r0, r0 + nrows) of call a owned by the CTA (cluster) with row-range index rg.
__device__ __forceinline__ void cta_rows(const StreamArgs& a, int rg, int64_t& r0, int& nrows) {
  r0 = (static_cast<int64_t>(rg) * a.rows_base + min(rg, a.rows_extra)) * a.gran;
  const int64_t n = min(static_cast<int64_t>((a.rows_base + (rg < a.rows_extra ? 1 : 0)) * a.gran), a.M - r0);
  nrows = static_cast<int>(max(n, static_cast<int64_t>(0)));
}

// A consumer warp's walk over the tiles of one K chunk: wait for each stage, let
// `consume` add the warp's products into its per-row partial sums, release the stage,
// reduce the sums over the warp and store them to `red` (the first K chunk of the CTA
// stores, later ones add).  The ring position and the status carry over between chunks.
struct TileWalk {
  uint32_t ring, full0, empty0;
  float* red;
  volatile int* abort_flag;
  unsigned* err;
  int stage_bytes, NS, R, G, wpc;
  int nvr;    // virtual rows of the row chunk
  bool first; // the CTA's first K chunk
  int g, c0, wc, lane;
  int slot;
  uint32_t fphase;
  bool ok;
};

template <int NC, int NCT, int RT, class F>
__device__ __forceinline__ void walk_tiles(TileWalk& w, F&& consume) {
  for (int t0 = 0; t0 < w.nvr; t0 += w.R) {
    const int rows = min(w.R, w.nvr - t0);
    w.ok = w.ok && mbar_wait_or_abort(w.full0 + 8u * w.slot, w.fphase, w.abort_flag, w.err);
    float2 acc[RT][NCT];
#pragma unroll
    for (int j = 0; j < RT; ++j)
#pragma unroll
      for (int c = 0; c < NCT; ++c) acc[j][c] = make_float2(0.0f, 0.0f);
    if (w.ok) consume(w.ring + static_cast<uint32_t>(w.slot) * w.stage_bytes, rows, acc);
    __syncwarp();
    if (w.lane == 0) mbar_arrive(w.empty0 + 8u * w.slot);
    if (++w.slot == w.NS) {
      w.slot = 0;
      w.fphase ^= 1u;
    }
    // warp reduction of the RT*NCT partial sums (padded to a power of two)
    constexpr int V = RT * NCT;
    constexpr int VP = V > 16 ? 32 : V > 8 ? 16 : V > 4 ? 8 : V > 2 ? 4 : V > 1 ? 2 : 1;
    float vals[VP];
#pragma unroll
    for (int j = 0; j < VP; ++j) vals[j] = j < V ? acc[j / NCT][j % NCT].x + acc[j / NCT][j % NCT].y : 0.0f;
    const float sum = WarpVecReduce<VP>::run(vals, w.lane);
    const int jv = w.lane >> (5 - WarpVecReduce<VP>::kLog);
    if (w.lane == WarpVecReduce<VP>::owner(jv) && jv < V) {
      const int r = w.g + (jv / NCT) * w.G, c = w.c0 + jv % NCT;
      if (r < rows && c < NC) {
        float* p = w.red + ((t0 + r) * w.wpc + w.wc) * NC + c;
        *p = w.first ? sum : (*p + sum);
      }
    }
  }
}

// fp32 dot product of one row's K chunk (weights from global memory through the
// 16-bit-load decoders, x from where the chunk lives) over the 32 lanes of a warp: the
// repair of rows whose x the integer path cannot carry.  Single column.  Every lane gets
// the sum.  IEEE semantics throughout (an infinite x gives the definition's Inf or NaN).
template <int WT, bool GAMMA>
__device__ __forceinline__ float repair_dot(const uint8_t* rowp, int units, const float* xsrc, int64_t xstride,
                                            const float* gsrc, bool norm, int lane) {
  const GmemLoader ld{rowp};
  float s = 0.0f;
  auto load_x = [&](int u, float2 (&xv)[1][8]) {
    if (norm)
      load_unit_x<WT, 1, GAMMA>(xsrc, xstride, gsrc, u, 0u, 0, 1, xv);
    else
      load_unit_x<WT, 1, false>(xsrc, xstride, nullptr, u, 0u, 0, 1, xv);
  };
  if constexpr (WT == WT_Q4_K) {
    for (int p = lane; 2 * p < units; p += 32) {
      float dsc[2], dmn[2];
      const uint4 q = q4k_load_pair(ld, static_cast<uint32_t>(p), dsc, dmn);
#pragma unroll 1
      for (int n = 0; n < 2; ++n) {
        float2 v[8], xv[1][8];
        q4k_nibbles(q, static_cast<uint32_t>(n), v);
        load_x(2 * p + n, xv);
        float2 t = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < 8; ++k)  // the weight d*sc*q - dmin*m first, then its product
          t = ffma2(ffma2(make_float2(dsc[n], dsc[n]), v[k], make_float2(-dmn[n], -dmn[n])), xv[0][k], t);
        s += t.x + t.y;
      }
    }
  } else {
    for (int u = lane; u < units; u += 32) {
      float2 v[8], xv[1][8];
      float d;
      decode_unit<WT>(ld, static_cast<uint32_t>(u), v, d);
      load_x(u, xv);
      float2 t = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int k = 0; k < 8; ++k) t = ffma2(v[k], xv[0][k], t);
      s = fmaf(d, t.x + t.y, s);
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  return s;
}

template <int WT, int NC, int FEAT>
__global__ void __launch_bounds__(stream_threads(WT, NC), 1)
    gemv_stream_kernel(const __grid_constant__ StreamArgs a) {
  constexpr bool kExt = FEAT != FEAT_PLAIN;     // dual GEMV / several matrices / RMS prologue compiled in
  constexpr bool kSplit = FEAT == FEAT_SPLIT;   // cluster split K compiled in
  constexpr int U = stream_u(WT, NC);
  constexpr int RT = stream_rt(WT, NC);
  constexpr int NCT = stream_nct(WT, NC);
  constexpr bool kInt = stream_int(WT, NC);
  // batched tile loads, except where they would spill (two F16 columns per thread with
  // the extension code)
  constexpr bool kBatch = !(kExt && WT == WT_F16 && NCT > 1);
  static_assert(U * NCT * 16 <= 64, "x registers per thread");
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t full0 = sbase, empty0 = sbase + 8u * a.NS, xbar = sbase + 16u * a.NS;
  const uint32_t xchbar = xbar + 8u;  // split K: arrivals of the peer CTAs (rank 0 only)
  float* xs = reinterpret_cast<float*>(smem + a.off_xs);
  float* auxs = reinterpret_cast<float*>(smem + a.off_aux);
  float* red = reinterpret_cast<float*>(smem + a.off_red);
  float* normv = reinterpret_cast<float*>(smem + a.off_norm);  // [wpc][NC] sums of squares
  float* xch = reinterpret_cast<float*>(smem + a.off_xchg);    // split K: [S][NC][XR], then [S][NC]
  const uint32_t ring = sbase + static_cast<uint32_t>(a.off_ring);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kBarBytes - 8);
  // integer path: some unit of x cannot be carried (its rows are recomputed in fp32)
  volatile int* xflag = reinterpret_cast<volatile int*>(smem + kBarBytes - 16);

  const int S = kSplit ? a.S : 1;
  int crank = 0;
  if constexpr (kSplit) crank = static_cast<int>(cluster_ctarank());
  const int rg = static_cast<int>(blockIdx.x) / S;  // row range of this CTA (its cluster's)

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    *xflag = 0;
    for (int i = 0; i < a.NS; ++i) {
      mbar_init(full0 + 8u * i, 1);
      mbar_init(empty0 + 8u * i, static_cast<uint32_t>(a.ncw));
    }
    mbar_init(xbar, 1);
    mbar_init(xchbar, static_cast<uint32_t>(S > 1 ? (S - 1) * a.ncw * 32 : 1));
    fence_mbar_init();
  }
  __syncwarp();  // warp 0 reaches the CTA-wide barrier below converged
  if constexpr (kSplit)
    cluster_sync_all();  // peers arrive on rank 0's barrier only after it is initialised
  else
    __syncthreads();
  pdl_trigger();

  int64_t r0;
  int nrows;
  cta_rows(a, rg, r0, nrows);
  const int kc_lo = crank * a.n_kc / S, kc_hi = (crank + 1) * a.n_kc / S;
  const bool dual = kExt && a.W2 != nullptr;
  const bool multi = kExt && a.nseg > 0;  // several matrices sharing x (never with dual)
  const bool norm = kExt && a.gamma != nullptr;
  const bool xnew = a.stage_x && nrows > 0;  // the producer copies x (and gamma) into xs

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      int it = 0, slot = 0;  // tiles issued; ring slot of the next one
      uint32_t ephase = 1u;   // parity of the empty-barrier phase that frees `slot`
      bool ok = true;
      bool x_issued = false;
      for (int rc0 = 0; rc0 < nrows && ok; rc0 += a.RC) {
        const int nrc = min(a.RC, nrows - rc0);
        const int nvr = dual ? 2 * nrc : nrc;
        for (int kc = kc_lo; kc < kc_hi && ok; ++kc) {
          const int klen = min(a.kc_len, a.K - kc * a.kc_len);
          const int seg = seg_bytes_of<WT>(klen);
          const int64_t segoff = seg_bytes_of<WT>(kc * a.kc_len);
          for (int t0 = 0; t0 < nvr; t0 += a.R) {
            const int rows = min(a.R, nvr - t0);
            const int h = dual ? rows / 2 : rows;  // rows taken from each matrix
            // the first NS tiles go to empty slots: no wait (a wait on the phase before a
            // fresh barrier's first one took ~0.9 us on GB300)
            if (it >= a.NS && !mbar_wait_or_abort(empty0 + 8u * slot, ephase, abort_flag, a.err)) {
              ok = false;
              break;
            }
            const uint32_t full = full0 + 8u * slot;
            const uint32_t dst = ring + static_cast<uint32_t>(slot) * a.stage_bytes;
            const int64_t row = r0 + rc0 + (dual ? t0 / 2 : t0);
            mbar_arrive_expect_tx(full, static_cast<uint32_t>(rows * seg));
            if (multi) {
              // the tile's rows, cut at segment boundaries (rows are contiguous within one)
              for (int r = 0; r < rows;) {
                int64_t local;
                const int i = seg_of(a, row + r, local);
                const int n = static_cast<int>(min(static_cast<int64_t>(rows - r), a.seg_end[i] - (row + r)));
                if (a.n_kc == 1) {
                  bulk_g2s(dst + static_cast<uint32_t>(r * seg), a.seg_W[i] + local * a.row_bytes,
                           static_cast<uint32_t>(n * seg), full, pol);
                } else {
                  for (int q = 0; q < n; ++q)
                    bulk_g2s(dst + static_cast<uint32_t>((r + q) * seg), a.seg_W[i] + (local + q) * a.row_bytes + segoff,
                             static_cast<uint32_t>(seg), full, pol);
                }
                r += n;
              }
            } else if (a.n_kc == 1) {
              bulk_g2s(dst, a.W + row * a.row_bytes, static_cast<uint32_t>(h * seg), full, pol);
              if (dual)
                bulk_g2s(dst + static_cast<uint32_t>(h * seg), a.W2 + row * a.row_bytes,
                         static_cast<uint32_t>(h * seg), full, pol);
            } else if (!dual) {
              for (int r = 0; r < rows; ++r)
                bulk_g2s(dst + static_cast<uint32_t>(r * seg), a.W + (row + r) * a.row_bytes + segoff,
                         static_cast<uint32_t>(seg), full, pol);
            } else {
              for (int r = 0; r < rows; ++r) {
                const bool up = r >= h;
                const uint8_t* src = (up ? a.W2 : a.W) + (row + (up ? r - h : r)) * a.row_bytes + segoff;
                bulk_g2s(dst + static_cast<uint32_t>(r * seg), src, static_cast<uint32_t>(seg), full, pol);
              }
            }
            ++it;
            if (++slot == a.NS) {
              slot = 0;
              ephase ^= 1u;
            }
            if (xnew && !x_issued) {
              // x staged by bulk copy right behind the first weight tile, once the preceding
              // grid (which may write x) has finished: later in the queue it would wait
              // behind the whole ring of weight tiles (with the RMS prologue, gamma follows
              // x on the same barrier)
              pdl_wait();
              mbar_arrive_expect_tx(xbar, static_cast<uint32_t>((NC + (norm ? 1 : 0)) * a.K * 4));
              for (int c = 0; c < NC; ++c)
                bulk_g2s(smem_u32(xs + c * a.K), a.x + static_cast<int64_t>(c) * a.K,
                         static_cast<uint32_t>(a.K * 4), xbar);
              if (norm) bulk_g2s(smem_u32(xs + NC * a.K), a.gamma, static_cast<uint32_t>(a.K * 4), xbar);
              x_issued = true;
            }
          }
        }
      }
      if (!ok) {
        // Drain: wait (bounded) until every copy this thread issued has landed.
        for (int i = max(0, it - a.NS); i < it; ++i)
          (void)mbar_wait(full0 + 8u * (i % a.NS), static_cast<uint32_t>((i / a.NS) & 1));
        if (x_issued) (void)mbar_wait(xbar, 0u);
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    // Every consumer thread runs the same sequence of named barriers whether or not a
    // wait gave up; after an abort the remaining work is skipped, not the barriers.
    const int cw = warp - 1, ctid = threadIdx.x - 32, nt = a.ncw * 32;
    const uint32_t qr = lane_quad_rot<WT>(lane);
    auto epi_aux = [](int e) { return e == EPI_SILU_MUL || e == EPI_ADD; };
    const bool finalizer = (crank == 0);
    pdl_wait();  // x, aux and dst may belong to the preceding grid
    int slot = 0;            // ring slot of the next tile
    uint32_t fphase = 0;     // parity of its full-barrier phase
    uint32_t xphase = 0;
    bool ok = true;
    auto cbar = [&]() { named_bar_sync(1, static_cast<uint32_t>(nt)); };
    const int XR = dual ? 2 * a.RC : a.RC;  // virtual rows per row chunk
    const int g = cw / a.wpg;               // row group of this warp
    const int wr = cw - g * a.wpg;          // warp within the row group
    const int cgi = wr / a.wpc;             // column group
    const int wc = wr - cgi * a.wpc;        // warp within the column group
    const int c0 = cgi * NCT;               // first column of this thread
    const int tg = wc * 32 + lane, tg_n = a.wpc * 32;
    bool need_aux = epi_aux(a.epi);
    if (multi)
      for (int i = 0; i < a.nseg; ++i) need_aux = need_aux || epi_aux(a.seg_epi[i]);
    // aux of column c at virtual row gr (0 for a segment whose tail takes none)
    auto aux_at = [&](int c, int64_t gr) -> float {
      if (!multi) return a.aux[c * a.M + gr];
      int64_t local;
      const int i = seg_of(a, gr, local);
      if (!epi_aux(a.seg_epi[i])) return 0.0f;
      const int64_t mi = a.seg_end[i] - (i ? a.seg_end[i - 1] : 0);
      return a.seg_aux[i][c * mi + local];
    };
    // Repair (integer path): when some unit of x could not be carried (xflag), the sums
    // of the row chunk starting at global row rb are recomputed in fp32 -- a warp per
    // virtual row, every K chunk of the row, x' rebuilt in shared memory chunk by chunk
    // with the on-chip prologue -- and stored where the finalisation reads them: red
    // (warp slot 0) or, with split K, slice 0 of rank 0's exchange buffer.  Every
    // consumer thread takes every barrier; after an abort the work is skipped.
    auto repair = [&](int64_t rb, int nrc_, int nvr_) {
      if constexpr (kInt) {
        if (ctid == 0 && a.err) atomicAdd(a.err + 1, 1u);  // counted for gf_repair_count
        if constexpr (kSplit) {
          for (int i = ctid; i < S * NC * XR; i += nt) xch[i] = 0.0f;
        } else {
          for (int i = ctid; i < nvr_ * a.wpc * NC; i += nt) red[i] = 0.0f;
        }
        cbar();
        const int H = a.R / 2;
        for (int kc2 = 0; kc2 < a.n_kc; ++kc2) {
          const int klen2 = min(a.kc_len, a.K - kc2 * a.kc_len);
          const float* xsrc2;
          int64_t xstride2;
          if (a.fwht_B > 0) {
            for (int i = ctid; i < NC * klen2; i += nt) {
              const int c = i / klen2, e = i - c * klen2;
              xs[i] = a.x[static_cast<int64_t>(c) * a.K + static_cast<int64_t>(kc2) * a.kc_len + e];
            }
            cbar();
            fwht_smem(xs, NC * klen2, a.fwht_B, klen2, static_cast<int64_t>(kc2) * a.kc_len, a.signs, a.nsigns,
                      a.fwht_scale, ctid, nt, cbar);
            xsrc2 = xs;
            xstride2 = klen2;
          } else if (a.stage_x) {
            xsrc2 = xs;
            xstride2 = a.K;
          } else {
            xsrc2 = a.x + static_cast<int64_t>(kc2) * a.kc_len;
            xstride2 = a.K;
          }
          const float* gsrc2 = !norm ? nullptr
                               : a.stage_x ? xs + NC * a.K
                                           : a.gamma + static_cast<int64_t>(kc2) * a.kc_len;
          const int64_t segoff = seg_bytes_of<WT>(kc2 * a.kc_len);
          for (int v = cw; v < nvr_ && !*abort_flag; v += a.ncw) {
            const uint8_t* rowp;
            if (dual) {  // tile t: gate rows t*H .. t*H+ht-1, then the same up rows
              const int t = v / a.R, l = v - t * a.R, ht = min(H, nrc_ - t * H);
              rowp = l < ht ? a.W + (rb + t * H + l) * a.row_bytes : a.W2 + (rb + t * H + l - ht) * a.row_bytes;
            } else if (multi) {
              int64_t local;
              const int i = seg_of(a, rb + v, local);
              rowp = a.seg_W[i] + local * a.row_bytes;
            } else {
              rowp = a.W + (rb + v) * a.row_bytes;
            }
            const float y = repair_dot<WT, kExt>(rowp + segoff, klen2 / kUnitElems, xsrc2, xstride2, gsrc2, norm, lane);
            if (lane == 0) {
              float* slot = kSplit ? xch + v : red + v * a.wpc * NC;
              *slot += y;
            }
          }
          cbar();  // the next chunk's x' overwrites xs
        }
      }
    };
    bool x_loaded = false;
    float ssq[NCT];  // this thread's share of the sum of squares of x (first row chunk)
#pragma unroll
    for (int c = 0; c < NCT; ++c) ssq[c] = 0.0f;
    for (int rc0 = 0; rc0 < nrows; rc0 += a.RC) {
      const int nrc = min(a.RC, nrows - rc0);
      const int nvr = dual ? 2 * nrc : nrc;
      for (int kc = kc_lo; kc < kc_hi; ++kc) {
        const int klen = min(a.kc_len, a.K - kc * a.kc_len);
        if (a.fwht_B > 0 && (a.n_kc > 1 || !x_loaded)) {
          // prologue: stage the chunk of every column in shared memory, transform it there
          if (x_loaded) cbar();  // nobody still reads the previous x chunk
          if (ctid == 0 && !*abort_flag) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(xbar, static_cast<uint32_t>(NC * klen * 4));
            for (int c = 0; c < NC; ++c)
              bulk_g2s(smem_u32(xs + c * klen), a.x + static_cast<int64_t>(c) * a.K + kc * a.kc_len,
                       static_cast<uint32_t>(klen * 4), xbar);
          }
          x_loaded = true;
          if (kc == 0 && need_aux)  // aux loads overlap the x copy
            for (int i = ctid; i < nrc * NC; i += nt) {
              const int c = i / nrc, r = i - c * nrc;
              auxs[c * a.RC + r] = aux_at(c, r0 + rc0 + r);  // plain load: aux may alias dst
            }
          ok = ok && mbar_wait_or_abort(xbar, xphase, abort_flag, a.err);
          xphase ^= 1u;
          fwht_smem(xs, NC * klen, a.fwht_B, klen, static_cast<int64_t>(kc) * a.kc_len, a.signs, a.nsigns,
                    a.fwht_scale, ctid, nt, cbar);
        } else if (kc == 0 && need_aux) {
          for (int i = ctid; i < nrc * NC; i += nt) {
            const int c = i / nrc, r = i - c * nrc;
            auxs[c * a.RC + r] = aux_at(c, r0 + rc0 + r);
          }
        }
        const int units = klen / kUnitElems;
        const int seg = seg_bytes_of<WT>(klen);
        // this thread's x (its units, its columns) in registers for the whole chunk: from
        // the transformed chunk in shared memory, or straight from global memory
        if (xnew && kc == kc_lo && rc0 == 0) {
          ok = ok && mbar_wait_or_abort(xbar, xphase, abort_flag, a.err);
          xphase ^= 1u;
        }
        const bool x_smem = a.fwht_B > 0 || a.stage_x;
        const float* xsrc = x_smem ? xs : a.x + static_cast<int64_t>(kc) * a.kc_len;
        const int64_t xstride = x_smem ? klen : a.K;
        const float* gsrc = !norm ? nullptr
                            : a.stage_x ? xs + NC * a.K  // staged after x
                                        : a.gamma + static_cast<int64_t>(kc) * a.kc_len;
        // (integer path: each unit's x is converted as soon as it is loaded)
        float2 xr[kInt ? 1 : U][NCT][8];
        XInt xq[kInt ? U : 1][kInt ? NCT : 1];
        float xsum[U][NCT];
        // integer path: per unit, whether its own values allow it, its largest |x| and the
        // sum of its 14 smaller |x| (see x_to_int)
        bool xlocal[U];
        float xmax[U], xrest[U];
#pragma unroll
        for (int i = 0; i < U; ++i) {
          const int u = unit_index<WT, U>(tg, i, tg_n);
          if (u < units && ok) {
            float2 (&xv)[NCT][8] = xr[kInt ? 0 : i];
            if (norm)
              load_unit_x<WT, NCT, kExt>(xsrc, xstride, gsrc, u, qr, c0, NC, xv, rc0 == 0, ssq);
            else
              load_unit_x<WT, NCT, false>(xsrc, xstride, nullptr, u, qr, c0, NC, xv);
            if constexpr (WT == WT_Q4_K) {  // the unit's sum of (scaled) x, for the sub-block min term
#pragma unroll
              for (int c = 0; c < NCT; ++c) {
                float2 t = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int k = 0; k < 8; ++k) t = fadd2(t, xv[c][k]);
                xsum[i][c] = t.x + t.y;
              }
            }
            if constexpr (kInt) xlocal[i] = x_to_int(xv[0], xq[i][0], xmax[i], xrest[i]);
          }
        }
        TileWalk w{ring, full0, empty0, red, abort_flag, a.err, a.stage_bytes, a.NS, a.R, a.G, a.wpc,
                   nvr, kc == kc_lo, g, c0, wc, lane, slot, fphase, ok};
        if constexpr (kInt) {
          // a unit the integer path cannot carry sets xflag: the rows are recomputed in fp32
          // before the tails (the integer sums stay finite meanwhile).  Units whose own
          // values do not allow it are judged against the warp's typical magnitude: the
          // mean of the units' trimmed means (a non-finite unit never passes).
          bool xbad = false;
          bool lbad = false;
#pragma unroll
          for (int i = 0; i < U; ++i)
            if (unit_index<WT, U>(tg, i, tg_n) < units && ok) lbad = lbad || !xlocal[i];
          if (__any_sync(0xffffffffu, lbad)) {
            float rsum = 0.0f, nun = 0.0f;
#pragma unroll
            for (int i = 0; i < U; ++i)
              if (unit_index<WT, U>(tg, i, tg_n) < units && ok) {
                rsum += fmaxf(xrest[i], 0.0f);  // 0 for a non-finite unit
                nun += 14.0f;
              }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
              rsum += __shfl_xor_sync(0xffffffffu, rsum, off);
              nun += __shfl_xor_sync(0xffffffffu, nun, off);
            }
            const float mu = rsum / fmaxf(nun, 1.0f);
#pragma unroll
            for (int i = 0; i < U; ++i)
              if (unit_index<WT, U>(tg, i, tg_n) < units && ok)
                xbad = xbad || !(xlocal[i] || (xmax[i] <= 256.0f * mu && xrest[i] == xrest[i]));
          }
          if (xbad) *xflag = 1;
          walk_tiles<NC, NCT, RT>(w, [&](uint32_t st, int rows, float2 (&acc)[RT][NCT]) {
            if constexpr (WT == WT_Q4_K)
              consume_tile_q4k_int<RT>(st, seg, rows, units, tg, g, a.G, xq, xsum, acc);
            else
              consume_tile_int<WT, NCT, U, RT>(st, seg, rows, units, tg, tg_n, g, a.G, xq, acc);
          });
        } else {
          walk_tiles<NC, NCT, RT>(w, [&](uint32_t st, int rows, float2 (&acc)[RT][NCT]) {
            if constexpr (WT == WT_Q4_K)
              consume_tile_q4k<NCT, RT>(st, seg, rows, units, tg, g, a.G, xr, xsum, acc);
            else
              consume_tile<WT, NCT, U, RT, kBatch>(st, seg, rows, units, tg, tg_n, g, a.G, qr, xr, acc);
          });
        }
        slot = w.slot;
        fphase = w.fphase;
        ok = w.ok;
      }
      if (norm && rc0 == 0 && g == 0) {
        // sum of squares: row group 0's column groups saw every x value of this CTA's K
        // range once; one slot per (warp of the column group, column)
#pragma unroll
        for (int c = 0; c < NCT; ++c) {
          float v = ssq[c];
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
          if (lane == 0 && c0 + c < NC) normv[wc * NC + c0 + c] = v;
        }
      }
      cbar();  // all partial sums of this row chunk are in `red` (and `normv`)
      if constexpr (kInt && !kSplit) {
        if (*xflag) repair(r0 + rc0, nrc, nvr);
      }
      // sum of squares of column c over this CTA's K range, warps in order
      auto ssum = [&](int c) -> float {
        float t = 0.0f;
        for (int w = 0; w < a.wpc; ++w) t += normv[w * NC + c];
        return t;
      };
      if constexpr (kSplit) {
        // split K (one row chunk per CTA): each rank's per-row sums go to slice `crank`
        // of rank 0's exchange buffer; rank 0 waits for every peer thread's arrival
        for (int i = ctid; i < nvr * NC; i += nt) {
          const int c = i / nvr, v = i - c * nvr;
          float y = 0.0f;
          for (int w = 0; w < a.wpc; ++w) y += red[(v * a.wpc + w) * NC + c];
          float* slot = xch + (crank * NC + c) * XR + v;
          if (finalizer)
            *slot = y;
          else
            st_cluster_f32(map_to_rank(smem_u32(slot), 0), y);
        }
        if (norm && ctid < NC) {  // this rank's sum of squares, after the S row slices
          float* slot = xch + S * NC * XR + crank * NC + ctid;
          const float t = ssum(ctid);
          if (finalizer)
            *slot = t;
          else
            st_cluster_f32(map_to_rank(smem_u32(slot), 0), t);
        }
        if constexpr (kInt) {  // rank 0 repairs if any rank's x could not be carried
          if (!finalizer && ctid == 0 && *xflag) st_cluster_u32(map_to_rank(smem_u32(const_cast<int*>(xflag)), 0), 1u);
        }
        if (!finalizer)
          mbar_arrive_remote(map_to_rank(xchbar, 0));
        else
          ok = ok && mbar_wait_cluster_or_abort(xchbar, 0, abort_flag, a.err);
        cbar();  // rank 0: its own slice is complete too
        if constexpr (kInt) {
          if (finalizer && *xflag) repair(r0 + rc0, nrc, nvr);
        }
      }
      if (ok && finalizer) {
        // sum of virtual row v for column c: the consumer warps' partials (one CTA),
        // or the S slices in rank order (split K)
        auto vsum = [&](int v, int c) -> float {
          float y = 0.0f;
          if constexpr (!kSplit) {
            for (int w = 0; w < a.wpc; ++w) y += red[(v * a.wpc + w) * NC + c];
          } else {
            for (int sl = 0; sl < S; ++sl) y += xch[(sl * NC + c) * XR + v];
          }
          return y;
        };
        const int H = a.R / 2;
        for (int i = ctid; i < nrc * NC; i += nt) {
          const int c = i / nrc, r = i - c * nrc;
          float inv = 1.0f;
          if (norm) {
            float t = 0.0f;
            if constexpr (kSplit) {
              for (int sl = 0; sl < S; ++sl) t += xch[S * NC * XR + sl * NC + c];
            } else {
              t = ssum(c);
            }
            inv = 1.0f / sqrtf(t / static_cast<float>(a.K) + a.norm_eps);
          }
          float out;
          if (dual) {
            // tile t holds gate rows t*H .. t*H+ht-1 then the same up rows
            const int t = r / H, l = r - t * H, ht = min(H, nrc - t * H);
            float yg = vsum(t * a.R + l, c), yu = vsum(t * a.R + ht + l, c);
            if (norm) {
              yg *= inv;
              yu *= inv;
            }
            out = tail_silu(yg) * yu;
          } else if (multi) {
            float y = vsum(r, c);
            if (norm) y *= inv;
            int64_t local;
            const int si = seg_of(a, r0 + rc0 + r, local);
            const int64_t mi = a.seg_end[si] - (si ? a.seg_end[si - 1] : 0);
            a.seg_dst[si][c * mi + local] = apply_tail(a.seg_epi[si], y, need_aux ? auxs[c * a.RC + r] : 0.0f);
            continue;
          } else {
            float y = vsum(r, c);
            if (norm) y *= inv;
            const float av = need_aux ? auxs[c * a.RC + r] : 0.0f;
            out = apply_tail(a.epi, y, av);
          }
          a.dst[c * a.M + r0 + rc0 + r] = out;
        }
      }
      cbar();  // red / auxs may be reused by the next row chunk
    }
  }
  __syncthreads();
  if constexpr (kSplit) cluster_sync_all();  // no CTA leaves while a peer may still store into it
}

template <int WT, int NC, int FEAT>
int launch_stream_t(const Plan& p, cudaStream_t st, bool pdl) {
  auto kern = gemv_stream_kernel<WT, NC, FEAT>;
  static int configured_smem[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && configured_smem[dev] < p.smem) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem);
    if (e != cudaSuccess) return e;
    configured_smem[dev] = p.smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(p.threads);
  cfg.dynamicSmemBytes = static_cast<size_t>(p.smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (FEAT == FEAT_SPLIT) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(p.s.S);
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
  return cudaLaunchKernelEx(&cfg, kern, p.s);
}

// Clusters of p.s.S CTAs of this kernel that can be resident at once (0 if the query
// fails); p gives the threads and dynamic shared memory of the launch.
template <int WT, int NC>
int max_active_clusters_t(const Plan& p) {
  auto kern = gemv_stream_kernel<WT, NC, FEAT_SPLIT>;
  // raise the limit to the device maximum, never below what a launch of this kernel set
  int dev = 0, smem_max = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      smem_max < p.smem ||
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.s.S * 64);
  cfg.blockDim = dim3(p.threads);
  cfg.dynamicSmemBytes = static_cast<size_t>(p.smem);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.s.S);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int WT, int FEAT>
int dispatch_cols(int ncols, const Plan& p, cudaStream_t st, bool pdl) {
  switch (ncols) {
    case 1: return launch_stream_t<WT, 1, FEAT>(p, st, pdl);
    case 2: return launch_stream_t<WT, 2, FEAT>(p, st, pdl);
    case 3: return launch_stream_t<WT, 3, FEAT>(p, st, pdl);
    case 4: return launch_stream_t<WT, 4, FEAT>(p, st, pdl);
    case 5: return launch_stream_t<WT, 5, FEAT>(p, st, pdl);
    case 6: return launch_stream_t<WT, 6, FEAT>(p, st, pdl);
    case 7: return launch_stream_t<WT, 7, FEAT>(p, st, pdl);
    case 8: return launch_stream_t<WT, 8, FEAT>(p, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

template <int WT>
int occupancy_cols(int ncols, const Plan& p) {
  switch (ncols) {
    case 1: return max_active_clusters_t<WT, 1>(p);
    case 2: return max_active_clusters_t<WT, 2>(p);
    case 3: return max_active_clusters_t<WT, 3>(p);
    case 4: return max_active_clusters_t<WT, 4>(p);
    case 5: return max_active_clusters_t<WT, 5>(p);
    case 6: return max_active_clusters_t<WT, 6>(p);
    case 7: return max_active_clusters_t<WT, 7>(p);
    case 8: return max_active_clusters_t<WT, 8>(p);
    default: return 0;
  }
}

}  // namespace gf
