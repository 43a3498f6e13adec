// Device helpers of the moeq CUDA library (sm_103a): PTX wrappers for
// mbarriers, bulk async copies and ordered global accesses; codebook expansion
// of FP2/FP3/FP4 blocks with byte permutes and int8 dot products; the Q8
// activation quantizer; the H32 rotation. Layouts are those of include/moeq.h.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "moeq.h"

namespace moeq {

constexpr int kMaxK = 8;                 // top-k limit of the fused kernels
constexpr uint32_t kSpinLimit = 1u << 20;  // bounded waits: well under a second each

// ------------------------------------------------------------------ status
__device__ __forceinline__ void set_status(int32_t* st, int32_t code) {
  if (st) atomicCAS(st, 0, code);
}

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase; false when the limit ran out. Each try
// may suspend the thread in hardware (up to 0.5 us) until the phase completes.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 500;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}

// Bulk asynchronous copy global -> shared (size and both addresses multiples of 16).
__device__ __forceinline__ void bulk_g2s(void* sdst, const void* gsrc, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(sdst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_prefetch_l2(const void* gsrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gsrc), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded spin until *p >= target (acquire). false when the limit ran out.
__device__ __forceinline__ bool spin_until_geq(const uint32_t* p, uint32_t target,
                                               uint32_t limit = kSpinLimit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (ld_acquire(p) >= target) return true;
    __nanosleep(i < 4 ? 32 : 200);
  }
  return false;
}

// Store with release semantics at GPU scope.
__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Atomic add with acquire-release semantics at GPU scope; returns the old value.
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Reduction add with release semantics at GPU scope (no return value).
__device__ __forceinline__ void red_add_release(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Atomic add without ordering (work queues); returns the old value.
__device__ __forceinline__ uint32_t atom_add_relaxed(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.relaxed.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier that also returns the AND of pred over the participating threads.
__device__ __forceinline__ bool named_bar_and(int id, int threads, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(threads)
      : "memory");
  return out != 0;
}

// ------------------------------------------------------------------ small conversions
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float f16_bits_to_f32(uint16_t b) {
  return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ float e8m0_to_f32(uint8_t e) {
  // 2^(e-127); e = 0 gives 2^-127 (a subnormal float), e = 255 is rejected upstream
  return e == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(static_cast<uint32_t>(e) << 23);
}

__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
  uint32_t x = __float_as_uint(f);
  if ((x & 0x7fffffffu) > 0x7f800000u) return static_cast<uint16_t>((x >> 16) | 0x40u);
  x += 0x7fffu + ((x >> 16) & 1u);
  return static_cast<uint16_t>(x >> 16);
}

// ------------------------------------------------------------------ codebook expansion
// Block dot products S = sum_j cb[code_j] * q_j for one 32-weight block against
// 32 int8 activations packed little-endian in q[0..7] (q[i] = elements 4i..4i+3).
// The codebook sits in registers; byte permutes expand four codes per
// instruction, dp4a multiplies and accumulates four products.

// FP2: cb = entries 0..3 in one word; w0, w1 the block's words.
__device__ __forceinline__ int dot_fp2(uint32_t w0, uint32_t w1, uint32_t cb, const int* q) {
  uint32_t a = w0 & 0x33333333u, b = (w0 >> 2) & 0x33333333u;
  // two independent accumulation chains (exact integer sums; shorter dependency)
  int s = __dp4a(static_cast<int>(prmt(cb, cb, a)), q[0], 0);
  int s2 = __dp4a(static_cast<int>(prmt(cb, cb, a >> 16)), q[1], 0);
  s = __dp4a(static_cast<int>(prmt(cb, cb, b)), q[2], s);
  s2 = __dp4a(static_cast<int>(prmt(cb, cb, b >> 16)), q[3], s2);
  a = w1 & 0x33333333u;
  b = (w1 >> 2) & 0x33333333u;
  s = __dp4a(static_cast<int>(prmt(cb, cb, a)), q[4], s);
  s2 = __dp4a(static_cast<int>(prmt(cb, cb, a >> 16)), q[5], s2);
  s = __dp4a(static_cast<int>(prmt(cb, cb, b)), q[6], s);
  s2 = __dp4a(static_cast<int>(prmt(cb, cb, b >> 16)), q[7], s2);
  return s + s2;
}

// FP3 selectors for the four (w, h) groups of 8 elements: low two bits from
// w0/w1, bit 2 moved from w2 to nibble bit 2 by one shift.
struct Fp3Sel {
  uint32_t s00, s01, s10, s11;
};

__device__ __forceinline__ Fp3Sel fp3_selectors(uint32_t w0, uint32_t w1, uint32_t w2) {
  Fp3Sel s;
  s.s00 = (w0 & 0x33333333u) | (w2 & 0x44444444u);
  s.s01 = ((w0 >> 2) & 0x33333333u) | ((w2 >> 1) & 0x44444444u);
  s.s10 = (w1 & 0x33333333u) | ((w2 << 2) & 0x44444444u);
  s.s11 = ((w1 >> 2) & 0x33333333u) | ((w2 << 1) & 0x44444444u);
  return s;
}

// FP3: cb0 = entries 0..3, cb1 = entries 4..7.
__device__ __forceinline__ int dot_fp3(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t cb0,
                                       uint32_t cb1, const int* q) {
  Fp3Sel t = fp3_selectors(w0, w1, w2);
  int s = __dp4a(static_cast<int>(prmt(cb0, cb1, t.s00)), q[0], 0);
  int s2 = __dp4a(static_cast<int>(prmt(cb0, cb1, t.s00 >> 16)), q[1], 0);
  s = __dp4a(static_cast<int>(prmt(cb0, cb1, t.s01)), q[2], s);
  s2 = __dp4a(static_cast<int>(prmt(cb0, cb1, t.s01 >> 16)), q[3], s2);
  s = __dp4a(static_cast<int>(prmt(cb0, cb1, t.s10)), q[4], s);
  s2 = __dp4a(static_cast<int>(prmt(cb0, cb1, t.s10 >> 16)), q[5], s2);
  s = __dp4a(static_cast<int>(prmt(cb0, cb1, t.s11)), q[6], s);
  s2 = __dp4a(static_cast<int>(prmt(cb0, cb1, t.s11 >> 16)), q[7], s2);
  return s + s2;
}

// FP3 in the Packed24 layout: code j at bits 3j..3j+2 of the 12-byte block
// read as one 96-bit little-endian integer, 8 codes per 24 bits. Each 24-bit
// group is spread into 8 selector nibbles: 6-bit code pairs into bytes, then
// the two codes of each byte into its two nibbles.
__device__ __forceinline__ uint32_t p24_spread(uint32_t u) {
  const uint32_t t = (u & 0x3Fu) | ((u << 2) & 0x3F00u) | ((u << 4) & 0x3F0000u) | ((u << 6) & 0x3F000000u);
  return (t & 0x07070707u) | ((t << 1) & 0x70707070u);
}

__device__ __forceinline__ Fp3Sel p24_selectors(uint32_t w0, uint32_t w1, uint32_t w2) {
  Fp3Sel s;  // s00, s01, s10, s11 = codes 0..7, 8..15, 16..23, 24..31
  s.s00 = p24_spread(w0);
  s.s01 = p24_spread(__funnelshift_r(w0, w1, 24));
  s.s10 = p24_spread(__funnelshift_r(w1, w2, 16));
  s.s11 = p24_spread(w2 >> 8);
  return s;
}

__device__ __forceinline__ int dot_fp3_sel(const Fp3Sel& t, uint32_t cb0, uint32_t cb1, const int* q) {
  int s = __dp4a(static_cast<int>(prmt(cb0, cb1, t.s00)), q[0], 0);
  int s2 = __dp4a(static_cast<int>(prmt(cb0, cb1, t.s00 >> 16)), q[1], 0);
  s = __dp4a(static_cast<int>(prmt(cb0, cb1, t.s01)), q[2], s);
  s2 = __dp4a(static_cast<int>(prmt(cb0, cb1, t.s01 >> 16)), q[3], s2);
  s = __dp4a(static_cast<int>(prmt(cb0, cb1, t.s10)), q[4], s);
  s2 = __dp4a(static_cast<int>(prmt(cb0, cb1, t.s10 >> 16)), q[5], s2);
  s = __dp4a(static_cast<int>(prmt(cb0, cb1, t.s11)), q[6], s);
  s2 = __dp4a(static_cast<int>(prmt(cb0, cb1, t.s11 >> 16)), q[7], s2);
  return s + s2;
}

// FP4 expansion of one word (8 codes in nibbles) into two words of int8 values.
// Entries 0..7 and 8..15 are looked up with 3-bit selectors; bit 3 of each code
// becomes a 0x00/0xff byte mask by a sign-replicating permute (selector nibble
// 8 | byte) and blends the two lookups.
__device__ __forceinline__ void fp4_expand(uint32_t w, uint32_t c0, uint32_t c1, uint32_t c2,
                                           uint32_t c3, uint32_t& v0, uint32_t& v1) {
  const uint32_t s = w & 0x77777777u;
  const uint32_t t = w << 4;
  const uint32_t lo0 = prmt(c0, c1, s), hi0 = prmt(c2, c3, s);
  const uint32_t m0 = prmt(t, w, 0xD9C8u);  // bit 3 of codes 0..3
  const uint32_t s1 = s >> 16;
  const uint32_t lo1 = prmt(c0, c1, s1), hi1 = prmt(c2, c3, s1);
  const uint32_t m1 = prmt(t, w, 0xFBEAu);  // bit 3 of codes 4..7
  v0 = (hi0 & m0) | (lo0 & ~m0);
  v1 = (hi1 & m1) | (lo1 & ~m1);
}

__device__ __forceinline__ int dot_fp4(uint4 wd, const uint32_t* cb, const int* q) {
  uint32_t v0, v1;
  fp4_expand(wd.x, cb[0], cb[1], cb[2], cb[3], v0, v1);
  int s = __dp4a(static_cast<int>(v0), q[0], 0);
  int s2 = __dp4a(static_cast<int>(v1), q[1], 0);
  fp4_expand(wd.y, cb[0], cb[1], cb[2], cb[3], v0, v1);
  s = __dp4a(static_cast<int>(v0), q[2], s);
  s2 = __dp4a(static_cast<int>(v1), q[3], s2);
  fp4_expand(wd.z, cb[0], cb[1], cb[2], cb[3], v0, v1);
  s = __dp4a(static_cast<int>(v0), q[4], s);
  s2 = __dp4a(static_cast<int>(v1), q[5], s2);
  fp4_expand(wd.w, cb[0], cb[1], cb[2], cb[3], v0, v1);
  s = __dp4a(static_cast<int>(v0), q[6], s);
  s2 = __dp4a(static_cast<int>(v1), q[7], s2);
  return s + s2;
}

// Generic: block (codes at p, shared or global memory) dotted with q, for the
// compile-time format FMT. cb holds (1 << FMT) / 4 codebook words.
template <int FMT>
__device__ __forceinline__ int block_dot(const uint8_t* p, const uint32_t* cb, const int* q) {
  if constexpr (FMT == 2) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    return dot_fp2(w.x, w.y, cb[0], q);
  } else if constexpr (FMT == 3) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(p);
    return dot_fp3(w[0], w[1], w[2], cb[0], cb[1], q);
  } else if constexpr (FMT == MOEQ_FP3_PACKED24) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(p);
    return dot_fp3_sel(p24_selectors(w[0], w[1], w[2]), cb[0], cb[1], q);
  } else {
    return dot_fp4(*reinterpret_cast<const uint4*>(p), cb, q);
  }
}

// Expansion of one block into 8 words of int8 weights (v[i] = weights
// 4i..4i+3), for blocks dotted with several activation vectors.
template <int FMT>
__device__ __forceinline__ void block_expand(const uint8_t* p, const uint32_t* cb, uint32_t (&v)[8]) {
  if constexpr (FMT == 2) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    const uint32_t a0 = w.x & 0x33333333u, b0 = (w.x >> 2) & 0x33333333u;
    const uint32_t a1 = w.y & 0x33333333u, b1 = (w.y >> 2) & 0x33333333u;
    v[0] = prmt(cb[0], cb[0], a0); v[1] = prmt(cb[0], cb[0], a0 >> 16);
    v[2] = prmt(cb[0], cb[0], b0); v[3] = prmt(cb[0], cb[0], b0 >> 16);
    v[4] = prmt(cb[0], cb[0], a1); v[5] = prmt(cb[0], cb[0], a1 >> 16);
    v[6] = prmt(cb[0], cb[0], b1); v[7] = prmt(cb[0], cb[0], b1 >> 16);
  } else if constexpr (FMT == 3 || FMT == MOEQ_FP3_PACKED24) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(p);
    const Fp3Sel t = FMT == 3 ? fp3_selectors(w[0], w[1], w[2]) : p24_selectors(w[0], w[1], w[2]);
    v[0] = prmt(cb[0], cb[1], t.s00); v[1] = prmt(cb[0], cb[1], t.s00 >> 16);
    v[2] = prmt(cb[0], cb[1], t.s01); v[3] = prmt(cb[0], cb[1], t.s01 >> 16);
    v[4] = prmt(cb[0], cb[1], t.s10); v[5] = prmt(cb[0], cb[1], t.s10 >> 16);
    v[6] = prmt(cb[0], cb[1], t.s11); v[7] = prmt(cb[0], cb[1], t.s11 >> 16);
  } else {
    const uint4 wd = *reinterpret_cast<const uint4*>(p);
    fp4_expand(wd.x, cb[0], cb[1], cb[2], cb[3], v[0], v[1]);
    fp4_expand(wd.y, cb[0], cb[1], cb[2], cb[3], v[2], v[3]);
    fp4_expand(wd.z, cb[0], cb[1], cb[2], cb[3], v[4], v[5]);
    fp4_expand(wd.w, cb[0], cb[1], cb[2], cb[3], v[6], v[7]);
  }
}

// Dot product of an expanded block with 32 int8 activations (exact int32).
__device__ __forceinline__ int dot8(const uint32_t (&v)[8], const int* q) {
  int s = __dp4a(static_cast<int>(v[0]), q[0], 0);
  int s2 = __dp4a(static_cast<int>(v[1]), q[1], 0);
#pragma unroll
  for (int i = 2; i < 8; i += 2) {
    s = __dp4a(static_cast<int>(v[i]), q[i], s);
    s2 = __dp4a(static_cast<int>(v[i + 1]), q[i + 1], s2);
  }
  return s + s2;
}

template <int FMT>
__host__ __device__ constexpr int block_bytes() {
  return FMT == 2 ? 8 : FMT == 3 || FMT == MOEQ_FP3_PACKED24 ? 12 : 16;
}

template <int FMT>
__device__ __forceinline__ float block_scale(const uint8_t* scales, int i) {
  if constexpr (FMT == 4) {
    return e8m0_to_f32(scales[i]);
  } else {
    return f16_bits_to_f32(reinterpret_cast<const uint16_t*>(scales)[i]);
  }
}

// ------------------------------------------------------------------ Q8 and H32
// Q8 of one 32-block held by one thread (v[32] fp32): amax, d = fp16(amax/127)
// (IEEE division), r = 1/d (IEEE), q = clamp(rint(v*r), -127, 127).
__device__ __forceinline__ uint16_t q8_thread(const float* v, int* qw) {
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
  const __half dh = __float2half_rn(__fdiv_rn(amax, 127.0f));
  const float df = __half2float(dh);
  if (df == 0.0f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) qw[i] = 0;
  } else {
    const float r = __frcp_rn(df);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t w = 0;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        int qi = __float2int_rn(__fmul_rn(v[4 * i + t], r));
        qi = max(-127, min(127, qi));
        w |= (static_cast<uint32_t>(qi) & 0xffu) << (8 * t);
      }
      qw[i] = static_cast<int>(w);
    }
  }
  return __half_as_ushort(dh);
}

// Q8 of one 32-block spread over a warp (lane i holds element i).
__device__ __forceinline__ int8_t q8_warp(float v, uint16_t& dbits) {
  float amax = fabsf(v);
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
  const __half dh = __float2half_rn(__fdiv_rn(amax, 127.0f));
  dbits = __half_as_ushort(dh);
  const float df = __half2float(dh);
  if (df == 0.0f) return 0;
  int qi = __float2int_rn(__fmul_rn(v, __frcp_rn(df)));
  return static_cast<int8_t>(max(-127, min(127, qi)));
}

// H32 of one 32-block held by one thread: signs, then butterfly stages 0..4.
__device__ __forceinline__ void h32_thread(float* v, uint32_t signs) {
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if ((signs >> i) & 1u) v[i] = -v[i];
#pragma unroll
  for (int st = 0; st < 5; ++st) {
    const int bit = 1 << st;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (i & bit) continue;
      const float a = v[i], b = v[i | bit];
      v[i] = __fadd_rn(a, b);
      v[i | bit] = __fsub_rn(a, b);
    }
  }
}

// H32 of one 32-block spread over a warp (lane i holds element i).
__device__ __forceinline__ float h32_warp(float v, uint32_t signs, int lane) {
  if ((signs >> lane) & 1u) v = -v;
#pragma unroll
  for (int st = 0; st < 5; ++st) {
    const int bit = 1 << st;
    const float o = __shfl_xor_sync(0xffffffffu, v, bit);
    v = (lane & bit) ? __fsub_rn(o, v) : __fadd_rn(v, o);
  }
  return v;
}

// Canonical router-order warp sum: combining rounds 16, 8, 4, 2, 1.
__device__ __forceinline__ float warp_sum_canonical(float a) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, d));
  return a;
}

// Top-k selection ordering: larger value first, lower index on ties, NaN last,
// -0 equal to +0. ranks_key maps (value, index) to a 64-bit key whose unsigned
// order is that ordering (0 is below every real key and marks "no element").
__device__ __forceinline__ uint32_t ordered_bits(float v) {
  if (isnan(v)) return 0u;
  const uint32_t u = __float_as_uint(v == 0.0f ? 0.0f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float from_ordered_bits(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

__device__ __forceinline__ uint64_t ranks_key(float v, int index) {
  return (static_cast<uint64_t>(ordered_bits(v)) << 32) | (0xffffffffu - static_cast<uint32_t>(index));
}

// k rounds of a warp maximum over per-lane key lists: key[] of each lane is
// sorted in place (bitonic network, descending) and after the call lane s < k
// holds the s-th largest key of the warp (0 if fewer than s+1 keys exist).
template <int NPL>
__device__ __forceinline__ uint64_t warp_select_keys(uint64_t (&key)[NPL], int k, int lane) {
#pragma unroll
  for (int k2 = 2; k2 <= NPL; k2 <<= 1) {
#pragma unroll
    for (int j = k2 >> 1; j > 0; j >>= 1) {
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        const int l = i ^ j;
        if (l > i) {
          const bool desc = (i & k2) == 0;
          const uint64_t a = key[i], b = key[l];
          const bool swap = desc ? (a < b) : (a > b);
          key[i] = swap ? b : a;
          key[l] = swap ? a : b;
        }
      }
    }
  }
  uint64_t mine = 0ull;
  for (int s = 0; s < k; ++s) {
    uint64_t h = key[0];
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) {
      const uint64_t o = __shfl_xor_sync(0xffffffffu, h, d);
      h = o > h ? o : h;
    }
    if (lane == s) mine = h;
    if (h != 0ull && key[0] == h) {  // the lane that held the winner moves to its next key
#pragma unroll
      for (int i = 0; i + 1 < NPL; ++i) key[i] = key[i + 1];
      key[NPL - 1] = 0ull;
    }
  }
  return mine;
}

__device__ __forceinline__ int key_index(uint64_t key) {
  return static_cast<int>(0xffffffffu - static_cast<uint32_t>(key));
}
__device__ __forceinline__ float key_value(uint64_t key) {
  return from_ordered_bits(static_cast<uint32_t>(key >> 32));
}

// Top-k of E values held NPL per lane (lane l holds elements l + 32 i in v[i])
// and their softmax weights over all E: after the call lane s < k holds the
// s-th selected index in idx and its weight exp(l_s - max) / sum exp(l - max)
// in p.
template <int NPL>
__device__ __forceinline__ void warp_topk(const float (&v)[NPL], int E, int k, int lane, int& idx,
                                          float& p) {
  uint64_t key[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    key[i] = e < E ? ranks_key(v[i], e) : 0ull;
  }
  const uint64_t mine = warp_select_keys<NPL>(key, k, lane);
  const float m = key_value(__shfl_sync(0xffffffffu, mine, 0));
  float z = 0.0f;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E && !isnan(v[i])) z += expf(v[i] - m);
  }
  z = warp_sum_canonical(z);
  idx = key_index(mine);
  p = __fdiv_rn(expf(key_value(mine) - m), z);
}

}  // namespace moeq
