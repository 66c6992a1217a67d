// Device helpers shared by the gemvfuse kernels: inline-PTX wrappers (mbarrier,
// bulk async copy, programmatic dependent launch, packed f32x2 arithmetic), the
// weight unit decoders, the fused tails and the shared-memory Walsh-Hadamard passes.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace gf {

enum { WT_F32 = 0, WT_F16 = 1, WT_Q8_0 = 2, WT_Q4_0 = 3, WT_Q4_K = 4 };
enum { EPI_NONE = 0, EPI_SIGMOID = 1, EPI_SILU = 2, EPI_SILU_MUL = 3, EPI_ADD = 4 };
// Internal tail of the gated dual GEMV: silu(gate row) * (up row).
enum { EPI_GLU = 5 };
enum { ERRBIT_TIMEOUT = 1u };

// A bounded wait gives up after this many nanoseconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Suspend-time hint for try_wait: a waiting thread sleeps in hardware (it is woken when
// the phase completes) for up to this long instead of spinning on issue slots.
constexpr uint32_t kTryWaitHintNs = 100000u;

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kTryWaitHintNs)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase with the given parity to complete; false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// As mbar_wait, but also gives up as soon as *abort is set, and sets *abort (and the
// error word) when its own time limit runs out, so the rest of the CTA stops waiting.
__device__ __forceinline__ bool mbar_wait_or_abort(uint32_t bar, uint32_t parity,
                                                   volatile int* abort, unsigned* err,
                                                   uint64_t limit_ns = kWaitLimitNs) {
  if (*abort) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort = 1;
      if (err) atomicOr(err, static_cast<unsigned>(ERRBIT_TIMEOUT));
      return false;
    }
  }
}

// ------------------------------------------------------------------ clusters
// Split-K CTAs of one cluster push their partial sums into the shared memory of the
// cluster's rank-0 CTA (remote stores, then a release-arrive on its mbarrier); rank 0
// waits with cluster-scope acquire.

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster (release, then acquire).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address in the shared memory of CTA `rank` of this cluster matching local `addr`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kTryWaitHintNs)
      : "memory");
  return ok != 0;
}

// mbar_wait_or_abort with cluster-scope acquire (for arrivals from peer CTAs).
__device__ __forceinline__ bool mbar_wait_cluster_or_abort(uint32_t bar, uint32_t parity,
                                                           volatile int* abort, unsigned* err) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      if (err) atomicOr(err, static_cast<unsigned>(ERRBIT_TIMEOUT));
      return false;
    }
  }
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 1-D bulk async copy global -> shared (no multicast), completion counted on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Programmatic dependent launch: wait for the preceding grid's memory; allow the
// following grid to launch.  Both are no-ops without a programmatic dependency.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }

__device__ __forceinline__ void set_error(unsigned* err, unsigned bit) {
  if (err) atomicOr(err, bit);
}

// Packed two-lane fp32 arithmetic (one instruction, two IEEE-rounded results).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// ------------------------------------------------------------------ loaders
// The unit decoders read weight bytes through a loader so the same decode code runs
// on a shared-memory stage (the streaming kernel) and on global memory (dequantize).
// words<N>(start) returns N consecutive 32-bit words starting at a 2-byte-aligned
// offset.  The shared-memory loader reads the N+1 aligned words around them and
// funnel-shifts (it may read up to 3 bytes past the last byte: the stage ring keeps
// slack for that); the global-memory loader assembles them from 16-bit loads and
// never reads outside the requested bytes.

struct SmemLoader {
  uint32_t base;  // shared-state-space address of row start
  __device__ __forceinline__ uint32_t u16(uint32_t off) const {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(base + off));
    return v;
  }
  __device__ __forceinline__ uint32_t u32(uint32_t off) const {  // 4-byte aligned
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(base + off));
    return v;
  }
  __device__ __forceinline__ uint4 v4(uint32_t off) const {  // 16-byte aligned
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(base + off));
    return v;
  }
  __device__ __forceinline__ uint32_t word(uint32_t off) const { return u32(off); }   // 4-byte aligned
  __device__ __forceinline__ uint4 quad(uint32_t off) const { return v4(off); }       // 16-byte aligned
  template <int N>
  __device__ __forceinline__ void words(uint32_t start, uint32_t (&w)[N]) const {
    const uint32_t a = start & ~3u, sh = (start & 3u) * 8u;
    uint32_t r[N + 1];
#pragma unroll
    for (int i = 0; i <= N; ++i) r[i] = u32(a + 4u * i);
#pragma unroll
    for (int i = 0; i < N; ++i) w[i] = __funnelshift_r(r[i], r[i + 1], sh);
  }
};

struct GmemLoader {
  const uint8_t* base;
  __device__ __forceinline__ uint32_t u16(uint32_t off) const {
    return *reinterpret_cast<const uint16_t*>(base + off);
  }
  __device__ __forceinline__ uint4 v4(uint32_t off) const {
    return *reinterpret_cast<const uint4*>(base + off);
  }
  template <int N>
  __device__ __forceinline__ void words(uint32_t start, uint32_t (&w)[N]) const {
#pragma unroll
    for (int i = 0; i < N; ++i) w[i] = __byte_perm(u16(start + 4u * i), u16(start + 4u * i + 2u), 0x5410);
  }
  // word / quad from 16-bit loads: rows in global memory may be only 2-byte aligned
  __device__ __forceinline__ uint32_t word(uint32_t off) const {
    return __byte_perm(u16(off), u16(off + 2u), 0x5410);
  }
  __device__ __forceinline__ uint4 quad(uint32_t off) const {
    return make_uint4(word(off), word(off + 4u), word(off + 8u), word(off + 12u));
  }
};

// ------------------------------------------------------------------ unit decoders
// A "unit" is 16 weights of one row (half a quant block).  Unit u covers, within a
// row (or K chunk):
//   F32, F16, Q8_0 : elements 16u .. 16u+15
//   Q4_0           : block b = u/2, half h = u%2: code bytes 8h .. 8h+7 of the block,
//                    i.e. elements 32b+8h .. +7 (low nibbles) and 32b+16+8h .. +7 (high)
// decode_unit() returns the 16 values as eight float2 pairs (pair k = elements
// unit_pair_elem(u, k) and +1) together with the block scale d (1 for F32/F16).  Quant
// codes are turned into floats exactly: the byte goes into the low mantissa bits of
// 2^23 and 2^23 + offset is subtracted with a packed add, exact for every code.

constexpr float kMagic = 8388608.0f;  // 2^23

__device__ __forceinline__ float2 magic_pair(uint32_t w, uint32_t sel0, float bias) {
  const float a = __uint_as_float(__byte_perm(w, 0x4B000000u, sel0));
  const float b = __uint_as_float(__byte_perm(w, 0x4B000000u, sel0 + 1));
  return fadd2(make_float2(a, b), make_float2(bias, bias));
}

__device__ __forceinline__ float h2f(uint32_t bits16) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16)));
}

__device__ __forceinline__ float2 h2pair(uint32_t w) {
  __half2 h;
  *reinterpret_cast<uint32_t*>(&h) = w;
  return __half22float2(h);
}

// qr (F32/F16 only) rotates the order in which a thread visits the unit's four 16-byte
// quads: slot quad q holds natural quad (q + qr) & 3.  Lanes of a quarter warp use
// different rotations so their 16-byte shared-memory reads hit distinct banks; the x
// values are loaded with the same rotation, so every product pairs the same element.
template <int WT, class L>
__device__ __forceinline__ void decode_unit(const L& ld, uint32_t u, float2 (&v)[8], float& d,
                                            uint32_t qr = 0) {
  if constexpr (WT == WT_F32) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 a = ld.v4(u * 64u + 16u * ((q + qr) & 3u));
      v[2 * q] = make_float2(__uint_as_float(a.x), __uint_as_float(a.y));
      v[2 * q + 1] = make_float2(__uint_as_float(a.z), __uint_as_float(a.w));
    }
    d = 1.0f;
  } else if constexpr (WT == WT_F16) {
    const uint32_t h0 = (qr >> 1) & 1u;
    const uint4 a = ld.v4(u * 32u + 16u * h0);
    const uint4 b = ld.v4(u * 32u + 16u * (h0 ^ 1u));
    v[0] = h2pair(a.x); v[1] = h2pair(a.y); v[2] = h2pair(a.z); v[3] = h2pair(a.w);
    v[4] = h2pair(b.x); v[5] = h2pair(b.y); v[6] = h2pair(b.z); v[7] = h2pair(b.w);
    d = 1.0f;
  } else if constexpr (WT == WT_Q8_0) {
    const uint32_t b = u >> 1, h = u & 1u;
    const uint32_t off = b * 34u;
    d = h2f(ld.u16(off));
    uint32_t w[4];
    ld.template words<4>(off + 2u + 16u * h, w);
    const float bias = -(kMagic + 128.0f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t t = w[i] ^ 0x80808080u;  // bytes q + 128
      v[2 * i] = magic_pair(t, 0x7540u, bias);
      v[2 * i + 1] = magic_pair(t, 0x7542u, bias);
    }
  } else {  // WT_Q4_0
    const uint32_t b = u >> 1, h = u & 1u;
    const uint32_t off = b * 18u;
    d = h2f(ld.u16(off));
    uint32_t w[2];
    ld.template words<2>(off + 2u + 8u * h, w);
    const float bias = -(kMagic + 8.0f);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t lo = w[i] & 0x0F0F0F0Fu;
      const uint32_t hi = (w[i] >> 4) & 0x0F0F0F0Fu;
      v[2 * i] = magic_pair(lo, 0x7540u, bias);
      v[2 * i + 1] = magic_pair(lo, 0x7542u, bias);
      v[4 + 2 * i] = magic_pair(hi, 0x7540u, bias);
      v[4 + 2 * i + 1] = magic_pair(hi, 0x7542u, bias);
    }
  }
}

// The same decode for a shared-memory stage, split into the loads (RawUnit, so a
// thread can issue the loads of all its rows before any arithmetic) and the arithmetic
// (decode_raw).  F32 (16 registers per unit) keeps decode_unit.
template <int WT> struct RawUnit;
template <> struct RawUnit<WT_F16> { uint4 a, b; };
template <> struct RawUnit<WT_Q8_0> { uint32_t d, w[5]; };
template <> struct RawUnit<WT_Q4_0> { uint32_t d, w[3]; };

template <int WT>
__device__ __forceinline__ void load_raw(const SmemLoader& ld, uint32_t u, uint32_t qr, RawUnit<WT>& r) {
  if constexpr (WT == WT_F16) {
    const uint32_t h0 = (qr >> 1) & 1u;
    r.a = ld.v4(u * 32u + 16u * h0);
    r.b = ld.v4(u * 32u + 16u * (h0 ^ 1u));
  } else {
    constexpr uint32_t kBlk = WT == WT_Q8_0 ? 34u : 18u, kHalf = WT == WT_Q8_0 ? 16u : 8u;
    constexpr int kW = WT == WT_Q8_0 ? 5 : 3;
    const uint32_t off = (u >> 1) * kBlk;
    r.d = ld.u16(off);
    const uint32_t a = (off + 2u + kHalf * (u & 1u)) & ~3u;
#pragma unroll
    for (int i = 0; i < kW; ++i) r.w[i] = ld.u32(a + 4u * i);
  }
}

template <int WT>
__device__ __forceinline__ void decode_raw(const RawUnit<WT>& r, uint32_t u, float2 (&v)[8], float& d) {
  if constexpr (WT == WT_F16) {
    v[0] = h2pair(r.a.x); v[1] = h2pair(r.a.y); v[2] = h2pair(r.a.z); v[3] = h2pair(r.a.w);
    v[4] = h2pair(r.b.x); v[5] = h2pair(r.b.y); v[6] = h2pair(r.b.z); v[7] = h2pair(r.b.w);
    d = 1.0f;
  } else {
    constexpr uint32_t kBlk = WT == WT_Q8_0 ? 34u : 18u, kHalf = WT == WT_Q8_0 ? 16u : 8u;
    const uint32_t sh = (((u >> 1) * kBlk + 2u + kHalf * (u & 1u)) & 3u) * 8u;
    d = h2f(r.d);
    if constexpr (WT == WT_Q8_0) {
      const float bias = -(kMagic + 128.0f);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t t = __funnelshift_r(r.w[i], r.w[i + 1], sh) ^ 0x80808080u;  // bytes q + 128
        v[2 * i] = magic_pair(t, 0x7540u, bias);
        v[2 * i + 1] = magic_pair(t, 0x7542u, bias);
      }
    } else {
      const float bias = -(kMagic + 8.0f);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint32_t w = __funnelshift_r(r.w[i], r.w[i + 1], sh);
        const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
        v[2 * i] = magic_pair(lo, 0x7540u, bias);
        v[2 * i + 1] = magic_pair(lo, 0x7542u, bias);
        v[4 + 2 * i] = magic_pair(hi, 0x7540u, bias);
        v[4 + 2 * i + 1] = magic_pair(hi, 0x7542u, bias);
      }
    }
  }
}

// ---- Q4_K (super-blocks of 256 elements, 144 bytes: binary16 d and dmin, 12 bytes of
// packed 6-bit sub-block scales sc[j] and mins m[j], 128 code bytes; value
// d*sc[j]*q - dmin*m[j]).  Units come in pairs that share one 16-byte load of codes:
// pair p of a row (or K chunk) is super-block b = p / 8, pair-in-block pp = p % 8
// (group g = pp / 2, half h = pp % 2), code bytes 16 + 16*pp of the super-block.  Unit
// 2p + n is nibble n of those bytes: sub-block j = 2g + n, elements 32j + 16h .. + 15.
constexpr uint32_t kQ4kBytes = 144;

// d*sc[j] and dmin*m[j] (both exact in fp32) of sub-blocks 2g and 2g+1 of a super-block,
// from its first four words (hdr = d | dmin << 16, then the 12 packed scale bytes).
__device__ __forceinline__ void q4k_scales_from(uint32_t hdr, uint32_t s0, uint32_t s1, uint32_t s2, uint32_t g,
                                                float (&dsc)[2], float (&dmn)[2]) {
  const float d = h2f(hdr & 0xFFFFu), dmin = h2f(hdr >> 16);
  const bool upper = g >= 2u;  // sub-blocks 4..7: low bits in bytes 8..11, high bits in 0..7
#pragma unroll
  for (uint32_t n = 0; n < 2; ++n) {
    const uint32_t sh = 8u * ((2u * g + n) & 3u);
    const uint32_t a = (s0 >> sh) & 0xFFu, b = (s1 >> sh) & 0xFFu, c = (s2 >> sh) & 0xFFu;
    const uint32_t sc = upper ? ((c & 15u) | ((a >> 6) << 4)) : (a & 63u);
    const uint32_t m = upper ? ((c >> 4) | ((b >> 6) << 4)) : (b & 63u);
    dsc[n] = d * static_cast<float>(sc);
    dmn[n] = dmin * static_cast<float>(m);
  }
}

// The same for the super-block at boff.
template <class L>
__device__ __forceinline__ void q4k_scales(const L& ld, uint32_t boff, uint32_t g, float (&dsc)[2],
                                           float (&dmn)[2]) {
  q4k_scales_from(ld.word(boff), ld.word(boff + 4u), ld.word(boff + 8u), ld.word(boff + 12u), g, dsc, dmn);
}

// The 16 code bytes of unit pair p and its two sub-blocks' scale and min.
template <class L>
__device__ __forceinline__ uint4 q4k_load_pair(const L& ld, uint32_t p, float (&dsc)[2], float (&dmn)[2]) {
  const uint32_t pp = p & 7u;
  const uint32_t boff = (p >> 3) * kQ4kBytes;
  q4k_scales(ld, boff, pp >> 1, dsc, dmn);
  return ld.quad(boff + 16u + 16u * pp);
}

// Nibble n of the 16 code bytes as exact floats 0..15: eight pairs of consecutive
// elements of unit 2p + n.
__device__ __forceinline__ void q4k_nibbles(const uint4 q, uint32_t n, float2 (&v)[8]) {
  const float bias = -kMagic;
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t c = (w[i] >> (4u * n)) & 0x0F0F0F0Fu;
    v[2 * i] = magic_pair(c, 0x7540u, bias);
    v[2 * i + 1] = magic_pair(c, 0x7542u, bias);
  }
}

// ---- integer dot products (Q4_0, Q8_0 and Q4_K, single columns)
// A unit's 16 x values become integers X_j = rn(x_j * 2^s) (round to nearest) that share
// the exponent s, chosen so that m * 2^s lies in [2^22, 2^23) for m = max |x_j|; when
// m's significand is all ones (m * 2^s would round up to 2^23) s is one less.  Hence
// -2^23 <= X_j <= 2^23 - 1.  Each X_j is split into three bytes
// X = D2 * 2^16 + D1 * 2^8 + D0 (D2 signed, D1 and D0 unsigned), packed four elements
// to a register in the order of the unit's code bytes: group g holds the elements of the
// low nibbles (g = 0, 1) or high nibbles (g = 2, 3) of code word g % 2.
// sum_j (q_j - 8) X_j is then exact in 32-bit integers (|.| <= 2^30): three chains of
// four dp4a (one per digit) on the unpacked nibbles, combined at the end with
// -8 sum_j X_j (modulo 2^32; the result fits).  The block's d times 2^-s scales the
// converted sum.  Rounding x * 2^s moves each x_j by at most 2^-s / 2 <= m * 2^-23.
//
// That error is m * 2^-23 at most for every value of the unit: small next to the row's
// products unless m stands far above the values around it.  A unit is carried by the
// integer path when all 16 values are finite and
//  - m <= 1024 * (mean |x| of its 14 values left after the two largest): each value moves
//    by at most 1.2e-4 of that mean, even when the two largest carry zero weights; or
//  - at most two values are non-zero and the second is within 2^7 of m (one-hot and
//    two-hot units); or
//  - m <= 256 * mu, mu the mean of that trimmed mean over the 32 units of the warp
//    (512 values of x): the unit's rounding is then small next to the typical products of
//    the row, however small its own other values are (a SwiGLU output, whose units often
//    hold a few large values among near-zero ones, stays on the integer path).
// The roundings of independent values add with random signs, so the error stays a few
// thousandths of the tolerance on every input measured.  A unit failing all three (one
// or two outliers far above everything near them, or a NaN / Inf) flags its CTA: the
// CTA's rows are then recomputed in fp32 from the weights in global memory before the
// tails (exact IEEE semantics for non-finite x).  That costs a second read of the
// CTA's weights, so the rule is no stricter than the tolerance needs.
struct XInt {
  uint32_t d2[4], d1[4], d0[4];  // digit bytes of the four element groups
  uint32_t c;                    // -8 * sum_j X_j (two's complement)
  float sc;                      // 2^-s
};

__device__ __forceinline__ uint32_t dp4a_us(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t dp4a_uu(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t dp4a_ss(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t dp4a_su(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Digit registers of four integers a..d (byte k of each register is element k).
__device__ __forceinline__ void pack_digits(uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t& d2,
                                            uint32_t& d1, uint32_t& d0) {
  const uint32_t ab = __byte_perm(a, b, 0x5140u), cd = __byte_perm(c, d, 0x5140u);  // bytes 0, 1 interleaved
  d0 = __byte_perm(ab, cd, 0x5410u);
  d1 = __byte_perm(ab, cd, 0x7632u);
  d2 = __byte_perm(__byte_perm(a, b, 0x0062u), __byte_perm(c, d, 0x6200u), 0x7610u);
}

// x of one unit (eight pairs in decode_unit()'s pair order: pairs 2g and 2g+1 form group
// g) -> XInt.  The exponent is kept in [-126, 126] so that 2^s and 2^-s are normal
// floats; below |x| = 2^-103 the integers get shorter (absolute error under 2^-126).
// Returns whether the unit's own values allow the integer path (the first two rules
// above); m gets the unit's largest |x| and rest the sum of |x| over its 14 smaller
// values (NaN when a value is not finite).
__device__ __forceinline__ bool x_to_int(const float2 (&xv)[8], XInt& xi, float& m_out, float& rest_out) {
  float m = 0.0f, m2 = 0.0f, sa = 0.0f;  // largest and second largest |x|, sum of |x|
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float a = fabsf(xv[k].x), b = fabsf(xv[k].y);
    const float hi = fmaxf(a, b), lo = fminf(a, b);
    sa += a + b;
    m2 = fmaxf(fmaxf(m2, lo), fminf(m, hi));
    m = fmaxf(m, hi);
  }
  // both false for NaN or Inf (sa is then NaN or Inf, and the rest NaN); true for zeros
  const float rest = sa - m - m2;  // |x| of the other 14 values (0 up to rounding: sparse)
  const bool dense = m * 14.0f <= 1024.0f * rest ||
                     (rest <= m * 0x1p-20f && (m2 == 0.0f || m <= 128.0f * m2));
  m_out = m;
  rest_out = rest;
  // m = f * 2^E with f in [0.5, 1): E = biased exponent - 126 (m = 0: any s works); one
  // less when f = 1 - 2^-24, whose m * 2^(23 - E) would round to 2^23
  const uint32_t mb = __float_as_uint(m);
  const int E = static_cast<int>((mb >> 23) & 0xFFu) - 126;
  const int s = max(-126, min(126, 23 - E - ((mb & 0x7FFFFFu) == 0x7FFFFFu ? 1 : 0)));
  const float up = __uint_as_float(static_cast<uint32_t>(s + 127) << 23);
  xi.sc = __uint_as_float(static_cast<uint32_t>(127 - s) << 23);
  int sum = 0;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const int X0 = __float2int_rn(xv[2 * g].x * up), X1 = __float2int_rn(xv[2 * g].y * up);
    const int X2 = __float2int_rn(xv[2 * g + 1].x * up), X3 = __float2int_rn(xv[2 * g + 1].y * up);
    sum += (X0 + X1) + (X2 + X3);
    pack_digits(static_cast<uint32_t>(X0), static_cast<uint32_t>(X1), static_cast<uint32_t>(X2),
                static_cast<uint32_t>(X3), xi.d2[g], xi.d1[g], xi.d0[g]);
  }
  xi.c = static_cast<uint32_t>(-8 * sum);
  return dense;
}

// Four registers of unsigned codes (byte k of n[g] is element 4g + k) against the XInt of
// each of NCT columns: t[c] = sum_j q_j X_j, minus 8 sum_j X_j with OFFSET (Q4_0's
// q - 8; |t| < 2^31 for codes below 16).
template <int NCT, bool OFFSET>
__device__ __forceinline__ void nibble_words_int(const uint32_t (&n)[4], const XInt (&xq)[NCT], int (&t)[NCT]) {
#pragma unroll
  for (int c = 0; c < NCT; ++c) {
    uint32_t s2 = 0u, s1 = 0u, s0 = OFFSET ? xq[c].c : 0u;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      s2 = dp4a_us(n[g], xq[c].d2[g], s2);
      s1 = dp4a_uu(n[g], xq[c].d1[g], s1);
      s0 = dp4a_uu(n[g], xq[c].d0[g], s0);
    }
    t[c] = static_cast<int>((s2 * 256u + s1) * 256u + s0);
  }
}

// A Q4_0 unit's two code words (code bytes 8h .. 8h+7 of its block) against the XInt of
// each of NCT columns: t[c] = sum_j (q_j - 8) X_j.
template <int NCT>
__device__ __forceinline__ void q4_0_words_int(uint32_t w0, uint32_t w1, const XInt (&xq)[NCT], int (&t)[NCT]) {
  const uint32_t n[4] = {w0 & 0x0F0F0F0Fu, w1 & 0x0F0F0F0Fu, (w0 >> 4) & 0x0F0F0F0Fu, (w1 >> 4) & 0x0F0F0F0Fu};
  nibble_words_int<NCT, true>(n, xq, t);
}

// A Q8_0 unit's four code words (16 signed codes, group g = word g) against the XInt of
// each of NCT columns: t[c] = sum_j q_j X_j.  |q_j| <= 128 and 24-bit X_j overflow 32
// bits in one sum, so the three digit sums (each exact, |.| < 2^19 * 2) are combined in
// float: t = S2 * 2^16 + S1 * 2^8 + S0, rounded once or twice to 24 bits.  (XInt.c, the
// Q4_0 offset term, is not used.)
template <int NCT>
__device__ __forceinline__ void q8_0_words_int(const uint32_t (&w)[4], const XInt (&xq)[NCT], float (&t)[NCT]) {
#pragma unroll
  for (int c = 0; c < NCT; ++c) {
    uint32_t s2 = 0u, s1 = 0u, s0 = 0u;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      s2 = dp4a_ss(w[g], xq[c].d2[g], s2);
      s1 = dp4a_su(w[g], xq[c].d1[g], s1);
      s0 = dp4a_su(w[g], xq[c].d0[g], s0);
    }
    t[c] = fmaf(static_cast<float>(static_cast<int>(s2)), 65536.0f,
                fmaf(static_cast<float>(static_cast<int>(s1)), 256.0f, static_cast<float>(static_cast<int>(s0))));
  }
}

// Quad rotation of a lane for the F32/F16 unit loads (0 for the block formats).
template <int WT>
__device__ __forceinline__ uint32_t lane_quad_rot(int lane) {
  return WT == WT_F32 ? ((lane >> 1) & 3u) : WT == WT_F16 ? (((lane >> 2) & 1u) << 1) : 0u;
}

// Element (within the row / chunk) of the first value of pair k of unit u.
template <int WT>
__device__ __forceinline__ uint32_t unit_pair_elem(uint32_t u, int k) {
  if constexpr (WT == WT_Q4_K) {
    const uint32_t p = u >> 1, pp = p & 7u;
    const uint32_t j = 2u * (pp >> 1) + (u & 1u);
    return (p >> 3) * 256u + 32u * j + 16u * (pp & 1u) + 2u * k;
  } else if constexpr (WT == WT_Q4_0) {
    const uint32_t b = u >> 1, h = u & 1u;
    return b * 32u + 8u * h + (k < 4 ? 2u * k : 16u + 2u * (k - 4));
  } else {
    return u * 16u + 2u * k;
  }
}

// Scalar decode of element k of a row in global memory (generic kernel).
template <int WT>
__device__ __forceinline__ float decode_elem(const uint8_t* row, int64_t k) {
  if constexpr (WT == WT_F32) {
    return reinterpret_cast<const float*>(row)[k];
  } else if constexpr (WT == WT_F16) {
    return __half2float(reinterpret_cast<const __half*>(row)[k]);
  } else if constexpr (WT == WT_Q8_0) {
    const int64_t b = k >> 5;
    const int j = static_cast<int>(k & 31);
    const uint8_t* blk = row + b * 34;
    const float d = h2f(*reinterpret_cast<const uint16_t*>(blk));
    return d * static_cast<float>(static_cast<int8_t>(blk[2 + j]));
  } else if constexpr (WT == WT_Q4_K) {
    const uint8_t* blk = row + (k >> 8) * kQ4kBytes;
    const int j = static_cast<int>((k & 255) >> 5), t = static_cast<int>(k & 31);
    const float d = h2f(*reinterpret_cast<const uint16_t*>(blk));
    const float dmin = h2f(*reinterpret_cast<const uint16_t*>(blk + 2));
    const uint8_t* sb = blk + 4;
    uint32_t sc, m;
    if (j < 4) {
      sc = sb[j] & 63u;
      m = sb[j + 4] & 63u;
    } else {
      sc = (sb[j + 4] & 15u) | ((sb[j - 4] >> 6) << 4);
      m = (sb[j + 4] >> 4) | ((sb[j] >> 6) << 4);
    }
    const uint32_t byte = blk[16 + 32 * (j >> 1) + t];
    const float q = static_cast<float>((j & 1) ? (byte >> 4) : (byte & 15u));
    return fmaf(d * static_cast<float>(sc), q, -(dmin * static_cast<float>(m)));
  } else {
    const int64_t b = k >> 5;
    const int j = static_cast<int>(k & 31);
    const uint8_t* blk = row + b * 18;
    const float d = h2f(*reinterpret_cast<const uint16_t*>(blk));
    const uint32_t byte = blk[2 + (j & 15)];
    const int q = static_cast<int>(j < 16 ? (byte & 15u) : (byte >> 4));
    return d * static_cast<float>(q - 8);
  }
}

// ------------------------------------------------------------------ fused tails
// One definition each, used by the fused epilogue and by the unfused element-wise
// control kernel so the two paths round identically.

__device__ __forceinline__ float tail_sigmoid(float y) { return 1.0f / (1.0f + expf(-y)); }
__device__ __forceinline__ float tail_silu(float y) { return y * tail_sigmoid(y); }

__device__ __forceinline__ float apply_tail(int epi, float y, float a) {
  switch (epi) {
    case EPI_SIGMOID: return tail_sigmoid(y);
    case EPI_SILU: return tail_silu(y);
    case EPI_SILU_MUL: return tail_silu(y) * a;
    case EPI_ADD: return y + a;
    default: return y;
  }
}

// ------------------------------------------------------------------ warp reduction
// Sums V per-lane values over the 32 lanes of a warp.  Lanes trade halves of their
// value vector (V - 1 shuffles in total for V <= 32) and finish with a butterfly.
// Afterwards lane l holds the total of value index (l >> (5 - log2 V)) & (V - 1) for
// V <= 32; red_owner() says which lane holds value j.
template <int V>
struct WarpVecReduce {
  static_assert(V >= 1 && V <= 32 && (V & (V - 1)) == 0, "V must be a power of two <= 32");
  static constexpr int kLog = (V >= 32) ? 5 : (V >= 16) ? 4 : (V >= 8) ? 3 : (V >= 4) ? 2 : (V >= 2) ? 1 : 0;
  __device__ __forceinline__ static float run(float (&v)[V], int lane) {
    int n = V;
#pragma unroll
    for (int step = 0; step < kLog; ++step) {
      const int off = 16 >> step;
      const bool upper = (lane & off) != 0;
      const int half = V >> (step + 1);
#pragma unroll
      for (int j = 0; j < half; ++j) {
        const float send = upper ? v[j] : v[j + half];
        const float keep = upper ? v[j + half] : v[j];
        v[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
      n >>= 1;
    }
    float s = v[0];
#pragma unroll
    for (int off = 16 >> kLog; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    return s;
  }
  __device__ __forceinline__ static int owner(int j) { return j << (5 - kLog); }
};

// ------------------------------------------------------------------ Walsh-Hadamard
// In-place transform of `total` floats in shared memory, laid out as segments of
// `seg_len` elements (one per column), each a whole number of blocks of B (a power of
// two).  Element e of a segment sits at column position koff + e.  The first pass
// multiplies by signs[(koff + e) % nsigns] while loading (signs may be null), the
// last multiplies by `scale` while storing.  Radix-4 passes (two butterfly stages
// (a, b) -> (a + b, a - b) at strides h and 2h), then one radix-2 pass if log2 B is
// odd.  `sync()` must be a barrier over the `nthr` participating threads; it is
// called after every pass.  Index arithmetic uses shifts and masks only, except the
// sign index when nsigns is not a power of two dividing B.
template <class Sync>
__device__ __forceinline__ void fwht_smem(float* buf, int total, int B, int seg_len, int64_t koff,
                                          const float* __restrict__ signs, int nsigns, float scale,
                                          int tid, int nthr, Sync sync) {
  int log2b = 0;
  while ((1 << log2b) < B) ++log2b;
  const int npass = (log2b >> 1) + (log2b & 1);
  // nsigns a power of two dividing B: koff and seg_len are multiples of B, so the sign
  // index of buffer position p is p & (nsigns - 1).
  const bool sign_mask = (nsigns & (nsigns - 1)) == 0 && nsigns <= B;
  const int koff32 = static_cast<int>(koff);
  auto sign_of = [&](int p) -> float {
    if (signs == nullptr) return 1.0f;
    if (sign_mask) return __ldg(signs + (p & (nsigns - 1)));
    const int pos = koff32 + (p % seg_len);
    return __ldg(signs + (pos % nsigns));
  };
  if (log2b == 0) {
    for (int p = tid; p < total; p += nthr) buf[p] = buf[p] * sign_of(p) * scale;
    sync();
    return;
  }
  int logh = 0;
  for (int pass = 0; pass < npass; ++pass) {
    const bool first = (pass == 0), last = (pass == npass - 1);
    const int h = 1 << logh;
    if (logh + 2 <= log2b) {
      // groups of 4 at strides h, 2h: B/4 groups per block
      const int lpb = log2b - 2;  // log2(groups per block)
      for (int g = tid; g < (total >> 2); g += nthr) {
        const int blk = g >> lpb, gi = g & ((1 << lpb) - 1);
        const int lo = gi & (h - 1), hi = gi >> logh;
        const int p0 = (blk << log2b) + (hi << (logh + 2)) + lo;
        float a0 = buf[p0], a1 = buf[p0 + h], a2 = buf[p0 + 2 * h], a3 = buf[p0 + 3 * h];
        if (first) {
          a0 *= sign_of(p0); a1 *= sign_of(p0 + h);
          a2 *= sign_of(p0 + 2 * h); a3 *= sign_of(p0 + 3 * h);
        }
        const float b0 = a0 + a1, b1 = a0 - a1, b2 = a2 + a3, b3 = a2 - a3;
        float c0 = b0 + b2, c1 = b1 + b3, c2 = b0 - b2, c3 = b1 - b3;
        if (last) { c0 *= scale; c1 *= scale; c2 *= scale; c3 *= scale; }
        buf[p0] = c0; buf[p0 + h] = c1; buf[p0 + 2 * h] = c2; buf[p0 + 3 * h] = c3;
      }
      logh += 2;
    } else {  // final radix-2 stage, h == B / 2
      const int lpb = log2b - 1;
      for (int g = tid; g < (total >> 1); g += nthr) {
        const int blk = g >> lpb, lo = g & ((1 << lpb) - 1);
        const int p0 = (blk << log2b) + lo;
        float a0 = buf[p0], a1 = buf[p0 + h];
        if (first) { a0 *= sign_of(p0); a1 *= sign_of(p0 + h); }
        float c0 = a0 + a1, c1 = a0 - a1;
        if (last) { c0 *= scale; c1 *= scale; }
        buf[p0] = c0; buf[p0 + h] = c1;
      }
      logh += 1;
    }
    sync();
  }
}

}  // namespace gf
