// Grouped GEMMs of the prefill on the 5th-generation tensor cores (tcgen05).
//
// One tile = 128 weight rows x up to 128 grouped rows (tokens of one expert),
// the whole contraction K. The block scales are folded into the operands and
// the operands split into bf16 parts:
//   weights  a = cb[code] * ws[r, b]   (<= 18 significant bits, exact in fp32)
//   activ.   x = q * d[t, b]            (<= 18 significant bits, exact in fp32)
//   a = a_hi + a_lo, x = x_hi + x_lo with a_hi = bf16(a), a_lo = bf16(a - a_hi)
//   (|lo| < 2^-8 |v|; what the two parts leave out is below 2^-17 of the value
//   over every int8 code and fp16 scale; for power-of-two (E8M0) weight scales
//   a is a bf16 value itself and a_lo = 0)
// and a . x ~ a_hi x_hi + a_hi x_lo + a_lo x_hi, each product exact in the fp32
// accumulator; with the term left out, a_lo x_lo (below 2^-16 of |a x|), the
// kept products differ from a x by less than 8 * 2^-18 (3.1e-5) of |a x|.
// tcgen05.mma kind::f16 accumulates the products and all 32-element blocks of
// K into one TMEM accumulator per tile, read out once per tile -- no per-block
// hand-off between the tensor cores and the CUDA cores. The only difference to
// the per-block formulation is the order of the fp32 sums and the parts' last
// bits, well inside the FFN output tolerance.
//
// The expanded weights (operand A) never touch shared memory: the expansion
// threads write them into TMEM (tcgen05.st, lane = weight row) and the MMA
// reads A from TMEM, so shared memory only carries the activation tiles (B).
// The MMA's N follows the rows a tile really has (a multiple of 16), so small
// expert groups do not pay for a full 128-row tile.
//
// Three GEMMs per expert kind: gate (epilogue: g to memory), up (epilogue:
// h = silu(g) u, H32 and Q8 of the 32-block of h, which is the 32 rows of one
// warp, and h's parts for the down GEMM), down (epilogue: the fp32 rows).
//
// Warp roles (18 warps):
//   0-7   expansion: warp w serves the rows of TMEM lane quarter w % 4 and
//         the 64-element stages of parity w / 4; the packed codes of its
//         stages, the chunk's block scales and the tile's codebook arrive by
//         cp.async into a per-thread ring of 3 chunk buffers (2 chunks ahead);
//         per block the codebook scaled by the block scale is split into bf16
//         parts, looked up with byte permutes and stored into the stage's
//         TMEM columns
//   8     activation producer: TMA (SWIZZLE_128B) of the tile's grouped rows,
//         parts hi and lo, 64 K-elements per stage, in 64-row boxes
//   9     MMA issuer (one thread) and TMEM owner
//   10-17 epilogue, two warps per TMEM lane quarter (64 columns each), once
//         per tile
// Rings (mbarriers, every wait bounded): 4 operand stages (B in shared memory,
// A in TMEM; a stage is full when both its barriers are: the producer's copies
// and the 4 expansion warps' stores), 2 TMEM tile accumulators (the epilogue
// of one tile overlaps the next tile's main loop). Before the CTA exits, the
// producer waits for the copies of its last stages, the MMA issuer for all of
// its MMAs and the expansion threads for their cp.async groups.
//
// Sources: "DeepSeek V4 Flash: 284B model, up to 32 tok/s on AMD Ryzen AI MAX+
// 395", section "ROCmFPX: fitting 284B weights into 128 GB" (small codebooks
// expanded on the fly); "deepseek-v4-flash-0731-evox3-rocm", section "The
// optimization ladder" (fused multi-token prefill with H32).
#include <cuda.h>
#include <cuda_runtime.h>

#include "moeq.h"
#include "moeq_device.cuh"
#include "moeq_host.h"
#include "moeq_layout.h"

namespace moeq {
namespace {

constexpr int kTM = 128;        // weight rows per tile = TMEM lanes
constexpr int kTN = 128;        // grouped rows per tile (largest MMA N)
constexpr int kBoxRows = 64;    // grouped rows per TMA box
constexpr int kKC = 8;          // 32-blocks per raw code chunk (4 stages)
constexpr int kStages = 4;      // operand stages (64 K-elements each)
constexpr int kAccBufs = 2;     // TMEM tile accumulators
constexpr int kRawBufs = 3;     // per-thread code chunk buffers (2 chunks prefetched)
constexpr int kTcThreads = 576;
constexpr int kExpWarps = 8;
constexpr int kBWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kEpiWarp0 = 10;
constexpr int kEpiWarps = 8;     // two per TMEM lane quarter, 64 columns each
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAcol0 = kAccBufs * kTN;  // first TMEM column of the weight ring

template <int FMT>
struct TcSmem {
  static constexpr int NA = FMT == 4 ? 1 : 2;  // weight parts
  static constexpr int BC = block_bytes<FMT>();
  // per-thread raw buffer: the codes of the thread's 4 blocks of a chunk, the
  // chunk's block scales (<= 16 B), the tile's codebook (<= 16 B)
  // (an odd number of 16-byte units, so that the threads of a quarter warp
  // start on different banks)
  static constexpr int RPT = ((kKC / 2) * BC + 32) / 16 % 2 ? (kKC / 2) * BC + 32 : (kKC / 2) * BC + 48;
  static constexpr int SCL = (kKC / 2) * BC;
  static constexpr int CBO = SCL + 16;
  uint8_t b[kStages][2][kTN * 128];   // activation parts: 128 rows x 64 bf16, SW128 K-major
  uint8_t raw[kRawBufs][kExpWarps * 32][RPT];
  uint64_t full_a[kStages];            // weight stage in TMEM: the 4 expansion warps of its parity
  uint64_t full_b[kStages];            // activation stage in shared memory: the producer + its bytes
  uint64_t empty[kStages];
  uint64_t acc_full[kAccBufs], acc_empty[kAccBufs];
  uint64_t drain;                     // completion of every MMA this CTA issued
  uint32_t nmma[kStages];             // MMA N of the stage (its tile's rows, rounded up to 16)
  uint32_t tmem_base;
  volatile int abort;
  volatile int drained;               // every MMA of this CTA has completed
};

// Waits with no dependency on another CTA (MMA completion, landing of this
// CTA's own copies) end unless the hardware is broken: they get a longer limit
// than the ring waits, so that a ring timeout never cuts them short.
constexpr uint32_t kDrainLimit = kSpinLimit * 16;
static_assert(kAcol0 + kStages * 2 * 32 <= kTmemCols, "TMEM: accumulators + weight ring");

enum EpiKind { EPI_G = 0, EPI_SWIGLU = 1, EPI_O = 2 };

struct TcArgs {
  DMat w;
  int shared, g0, g1;
  const int* toff;
  const int* offsets;
  int K, R, rows;
  float* g;          // EPI_G: written, EPI_SWIGLU: read; [rows x R]
  uint16_t* hhi;     // EPI_SWIGLU: h's parts for the down GEMM [rows x R]
  uint16_t* hlo;
  const uint32_t* signs_h;
  float* o;          // EPI_O [rows x R]
  const int* pid;
  int T, k, ns;
  moeq_debug dbg;
  int32_t* status;
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  uint64_t d = static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;                // leading byte offset (unused, K-major swizzled)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;        // stride byte offset: 8 rows x 128 B
  d |= 1ull << 46;                                     // descriptor version
  d |= 2ull << 61;                                     // 128-byte swizzle
  return d;
}

// kind::f16, bf16 A and B, fp32 D, both K-major, M = 128; N (a multiple of 16) at bits 17..22.
constexpr uint32_t kIdescM = (1u << 4) | (1u << 7) | (1u << 10) | ((kTM >> 4) << 24);

// D[tmem] (+)= A[TMEM, lane = row, bf16 pairs along the columns] x B[smem descriptor]^T
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bd, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
               :: "r"(d_tmem), "r"(a_tmem), "l"(bd), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                 "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 columns of this warp's lane quarter from 16 registers per thread.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
               :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
                  "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* bar) {
  asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
               :: "r"(smem_u32(dst)), "l"(tm), "r"(x), "r"(y), "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_u32(dst)), "l"(src) : "memory");
}
// 4- or 8-byte asynchronous copies (cache-all variant).
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" :: "r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

// mbarrier phase test that lets the hardware suspend the thread (for its own,
// system-dependent time limit) until the phase completes.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
               "selp.u32 %0, 1, 0, p;\n}"
               : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase by one lane, observing the abort flag
// (at most kSpinLimit suspensions of at most 1 us).
template <int FMT>
__device__ __forceinline__ bool ring_wait(TcSmem<FMT>& sm, uint64_t* bar, uint32_t parity, int32_t* status) {
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (sm.abort) return false;
  }
  sm.abort = 1;
  set_status(status, MOEQ_ERR_DEVICE_TIMEOUT);
  return false;
}

// Warp-wide form: every lane polls the barrier (one broadcast read), the
// decision is made uniform across the warp.
template <int FMT>
__device__ __forceinline__ bool warp_wait(TcSmem<FMT>& sm, uint64_t* bar, uint32_t parity, int32_t* status) {
  return __all_sync(0xffffffffu, ring_wait<FMT>(sm, bar, parity, status) ? 1 : 0) != 0;
}

// ---------------------------------------------------------------- operand parts
// Two fp32 values -> bf16 pair (round to nearest even), lower half = x.
__device__ __forceinline__ uint32_t bf16x2_rn(float x, float y) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(y), "f"(x));
  return r;
}
__device__ __forceinline__ float bf16_lo_f(uint32_t p) { return __uint_as_float(p << 16); }
__device__ __forceinline__ float bf16_hi_f(uint32_t p) { return __uint_as_float(p & 0xffff0000u); }

// hi/lo bf16 parts of four fp32 values (v = hi + lo up to the bits below 2^-16
// of v): hi pairs and lo pairs, elements (0, 1) and (2, 3).
__device__ __forceinline__ void split4(const float* v, uint32_t* hi, uint32_t* lo) {
  hi[0] = bf16x2_rn(v[0], v[1]);
  hi[1] = bf16x2_rn(v[2], v[3]);
  lo[0] = bf16x2_rn(__fsub_rn(v[0], bf16_lo_f(hi[0])), __fsub_rn(v[1], bf16_hi_f(hi[0])));
  lo[1] = bf16x2_rn(__fsub_rn(v[2], bf16_lo_f(hi[1])), __fsub_rn(v[3], bf16_hi_f(hi[1])));
}

// Byte planes (low bytes, high bytes) of four bf16 values given as two pairs.
__device__ __forceinline__ void planes(uint32_t p01, uint32_t p23, uint32_t& lo, uint32_t& hi) {
  lo = prmt(p01, p23, 0x6420u);
  hi = prmt(p01, p23, 0x7531u);
}

// The codebook scaled by one block scale, split into bf16 parts, as byte
// planes for the permute lookups: tl/th of the hi part, ul/uh of the lo part
// (1 << FMT entries, 4 per word). cbf: the codebook as fp32.
template <int FMT>
__device__ __forceinline__ void scaled_tables(const float* cbf, float ws, uint32_t* tl, uint32_t* th,
                                              uint32_t* ul, uint32_t* uh) {
  constexpr int NV = 1 << FMT;
#pragma unroll
  for (int w = 0; w < NV / 4; ++w) {
    float t[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) t[j] = __fmul_rn(cbf[4 * w + j], ws);  // exact: <= 18 significant bits
    uint32_t hp[2], lp[2];
    split4(t, hp, lp);
    planes(hp[0], hp[1], tl[w], th[w]);
    if constexpr (FMT != 4) planes(lp[0], lp[1], ul[w], uh[w]);
  }
}

// bf16 pairs of 4 elements from their low and high bytes.
__device__ __forceinline__ void interleave4(uint32_t lo, uint32_t hi, uint32_t* out) {
  out[0] = prmt(lo, hi, 0x5140u);
  out[1] = prmt(lo, hi, 0x7362u);
}

// The packed codes of one block (BC bytes at p, 8- or 16-byte aligned for
// FP2 / FP4, 4-byte for FP3) into registers.
template <int FMT>
__device__ __forceinline__ void load_codes(const uint8_t* p, uint32_t (&w)[4]) {
  if constexpr (FMT == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    w[0] = v.x; w[1] = v.y; w[2] = 0; w[3] = 0;
  } else if constexpr (FMT == 3) {
    const uint32_t* q = reinterpret_cast<const uint32_t*>(p);
    w[0] = q[0]; w[1] = q[1]; w[2] = q[2]; w[3] = 0;
  } else {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  }
}

// One block (its code words w) -> 16 words of bf16 pairs (elements 2i, 2i+1 in
// word i), values from the byte planes tl (low bytes) and th (high bytes).
template <int FMT>
__device__ __forceinline__ void expand_bf16(const uint32_t (&w)[4], const uint32_t* tl, const uint32_t* th,
                                            uint32_t* out) {
  if constexpr (FMT == 2) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t sa = w[q] & 0x33333333u, sb = (w[q] >> 2) & 0x33333333u;
      const uint32_t sel[4] = {sa, sa >> 16, sb, sb >> 16};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        interleave4(prmt(tl[0], tl[0], sel[i]), prmt(th[0], th[0], sel[i]), out + 8 * q + 2 * i);
    }
  } else if constexpr (FMT == 3) {
    const Fp3Sel s = fp3_selectors(w[0], w[1], w[2]);
    const uint32_t sel[8] = {s.s00, s.s00 >> 16, s.s01, s.s01 >> 16, s.s10, s.s10 >> 16, s.s11, s.s11 >> 16};
#pragma unroll
    for (int i = 0; i < 8; ++i)
      interleave4(prmt(tl[0], tl[1], sel[i]), prmt(th[0], th[1], sel[i]), out + 2 * i);
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t l0, l1, h0, h1;
      fp4_expand(w[q], tl[0], tl[1], tl[2], tl[3], l0, l1);
      fp4_expand(w[q], th[0], th[1], th[2], th[3], h0, h1);
      interleave4(l0, h0, out + 4 * q);
      interleave4(l1, h1, out + 4 * q + 2);
    }
  }
}

struct TileInfo {
  int g, e, m0, tt, off, n;
};

// Group of `tile`, scanning forward from group g, the group of an earlier tile
// of this CTA (tiles are numbered group by group; toff[c] = first tile of group
// c, non-decreasing, so the groups with toff[c] <= tile form a prefix). All 32
// lanes call it; one load per lane and step of 32 groups.
__device__ __forceinline__ int group_from(const TcArgs& a, int tile, int g, int lane) {
  for (;;) {
    const int c = g + 1 + lane;
    const bool le = c < a.g1 && __ldg(&a.toff[c]) <= tile;
    const unsigned m = __ballot_sync(0xffffffffu, le);
    g += __popc(m);
    if (m != 0xffffffffu) return g;
  }
}

__device__ __forceinline__ TileInfo tile_at(const TcArgs& a, int tile, int g) {
  TileInfo t;
  t.g = g;
  const int local = tile - __ldg(&a.toff[g]);
  const int rtiles = a.R / kTM;
  t.tt = local / rtiles;
  t.m0 = (local % rtiles) * kTM;
  t.e = a.shared ? 0 : g;
  t.off = __ldg(&a.offsets[g]);
  t.n = __ldg(&a.offsets[g + 1]) - t.off;
  return t;
}

__device__ __forceinline__ void pid_split(const TcArgs& a, int pid, int& t, int& s) {
  const int Tk = a.T * a.k;
  if (pid >= Tk) {
    t = pid - Tk;
    s = a.k;
  } else {
    t = pid / a.k;
    s = pid - t * a.k;
  }
}

// TMEM column of the weight ring: stage slot, part pa.
template <int NA>
__device__ __forceinline__ uint32_t a_col(int slot, int pa) {
  return kAcol0 + static_cast<uint32_t>((slot * NA + pa) * 32);
}

// ---------------------------------------------------------------- kernel
template <int FMT, int EPI>
__global__ void __launch_bounds__(kTcThreads, 1) tc_gemm_kernel(const __grid_constant__ CUtensorMap tm_hi,
                                                                const __grid_constant__ CUtensorMap tm_lo,
                                                                const TcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  TcSmem<FMT>& sm = *reinterpret_cast<TcSmem<FMT>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  using SM = TcSmem<FMT>;
  constexpr int BC = SM::BC;
  constexpr int NA = SM::NA;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = a.K / 32;
  const int nstages = a.K / 64;
  const int t_begin = __ldg(&a.toff[a.g0]);
  const int ntiles = __ldg(&a.toff[a.g1]) - t_begin;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm.full_a[i], 4);
      mbar_init(&sm.full_b[i], 1);
      mbar_init(&sm.empty[i], 1);             // MMA commit
    }
    for (int i = 0; i < kAccBufs; ++i) {
      mbar_init(&sm.acc_full[i], 1);  // MMA commit
      mbar_init(&sm.acc_empty[i], kEpiWarps);
    }
    mbar_init(&sm.drain, 1);
    sm.abort = 0;
    sm.drained = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(&sm.tmem_base)), "n"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp < kExpWarps) {
    // ------------------------------------------------------------ expansion
    // warp (q, hb): rows 32q .. 32q + 31 of the tile, the stages of parity hb
    // (every tile has an even number of stages, so the parity is the same in
    // the tile and in the ring); both 32-blocks of each of its stages
    const int q = warp & 3, hb = warp >> 2;
    const int r = 32 * q + lane;                       // weight row in the tile = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q) << 16);
    constexpr int NV = 1 << FMT;
    constexpr int SB = FMT == 4 ? 1 : 2;
    const int nchunks = (nstages + 3) / 4;             // chunks of 4 stages = kKC blocks
    // chunk c of tile t into raw buffer `buf`: the block pairs of this warp's
    // stages (hb and hb + 2 of the chunk), the chunk's scales, for c = 0 the
    // tile's codebook; the caller commits the group
    auto issue_chunk = [&](const TileInfo& t, int c, int buf) {
      const size_t row = static_cast<size_t>(t.m0 + r);
      const int kc = c * kKC, kb = min(kKC, nb - kc);
      uint8_t* dst = sm.raw[buf][tid];
      const uint8_t* src = a.w.codes + static_cast<size_t>(t.e) * a.w.stride_codes + (row * nb + kc) * BC;
      for (int pp = 0; pp < 2; ++pp) {
        const int sl = hb + 2 * pp;                    // stage in the chunk
        if (2 * sl >= kb) break;
        const uint8_t* ps = src + 2 * sl * BC;         // blocks 2 sl, 2 sl + 1: 2 BC contiguous bytes
        uint8_t* pd = dst + 2 * pp * BC;
        if constexpr (FMT == 3) {
          cp_async8(pd, ps);
          cp_async8(pd + 8, ps + 8);
          cp_async8(pd + 16, ps + 16);
        } else {
#pragma unroll
          for (int i = 0; i < 2 * BC; i += 16) cp_async16(pd + i, ps + i);
        }
      }
      const size_t soff = (row * nb + kc) * SB;
      const uint8_t* ssrc = a.w.scales + static_cast<size_t>(t.e) * a.w.stride_scales + soff;
      uint8_t* sdst = dst + SM::SCL;
      const int sbytes = kb * SB;  // 4, 8 or 16; soff is aligned to the piece used
      if (sbytes % 16 == 0 && soff % 16 == 0) {
        for (int i = 0; i < sbytes; i += 16) cp_async16(sdst + i, ssrc + i);
      } else if (sbytes % 8 == 0 && soff % 8 == 0) {
        for (int i = 0; i < sbytes; i += 8) cp_async8(sdst + i, ssrc + i);
      } else {
        for (int i = 0; i < sbytes; i += 4) cp_async4(sdst + i, ssrc + i);
      }
      if (c == 0) {  // codebook record: 16-byte aligned, NV bytes
        const int8_t* cb = a.w.cb + static_cast<size_t>(t.e) * a.w.cb_stride;
        if constexpr (NV == 16) cp_async16(dst + SM::CBO, cb);
        else if constexpr (NV == 8) cp_async8(dst + SM::CBO, cb);
        else cp_async4(dst + SM::CBO, cb);
      }
    };
    // prefetch cursor: kRawBufs - 1 chunks ahead of the one expanded, across
    // tile boundaries; one commit group per chunk (an empty one past the end)
    int p_ti = blockIdx.x, p_c = 0, p_g = a.g0, p_buf = 0;
    TileInfo p_t{};
    if (p_ti < ntiles) {
      p_g = group_from(a, t_begin + p_ti, p_g, lane);
      p_t = tile_at(a, t_begin + p_ti, p_g);
    }
    auto prefetch = [&]() {
      if (p_ti < ntiles) {
        issue_chunk(p_t, p_c, p_buf);
        if (++p_c == nchunks) {
          p_c = 0;
          p_ti += gridDim.x;
          if (p_ti < ntiles) {
            p_g = group_from(a, t_begin + p_ti, p_g, lane);
            p_t = tile_at(a, t_begin + p_ti, p_g);
          }
        }
      }
      cp_async_commit();
      p_buf = p_buf + 1 == kRawBufs ? 0 : p_buf + 1;
    };
    for (int i = 0; i < kRawBufs - 1; ++i) prefetch();
    float cbf[NV];
    int cbuf = 0, ks = 0;
    for (int ti = blockIdx.x; ti < ntiles && !sm.abort; ti += gridDim.x) {
      for (int c = 0; c < nchunks; ++c) {
        prefetch();
        cp_async_wait<kRawBufs - 1>();  // this chunk's group is complete
        const uint8_t* rawr = sm.raw[cbuf][tid];
        cbuf = cbuf + 1 == kRawBufs ? 0 : cbuf + 1;
        if (c == 0) {
#pragma unroll
          for (int v = 0; v < NV; ++v) cbf[v] = static_cast<float>(reinterpret_cast<const int8_t*>(rawr + SM::CBO)[v]);
        }
        const int nsc = min(4, nstages - 4 * c);
        for (int sl = hb; sl < nsc; sl += 2) {
          const int kg = ks + sl;  // stage in the ring's sequence
          const int slot = kg % kStages;
          if (kg >= kStages && !warp_wait<FMT>(sm, &sm.empty[slot], ((kg / kStages) - 1) & 1, a.status)) break;
          const uint8_t* pair = rawr + 2 * (sl >> 1) * BC;
#pragma unroll
          for (int bb = 0; bb < 2; ++bb) {
            const int jb = 2 * sl + bb;  // block in the chunk
            float ws;
            if constexpr (FMT == 4) ws = e8m0_to_f32(rawr[SM::SCL + jb]);
            else ws = f16_bits_to_f32(reinterpret_cast<const uint16_t*>(rawr + SM::SCL)[jb]);
            uint32_t cw[4];
            load_codes<FMT>(pair + bb * BC, cw);
            uint32_t tl[4], th[4], ul[4], uh[4];
            scaled_tables<FMT>(cbf, ws, tl, th, ul, uh);
            uint32_t vh[16], vl[16];
            expand_bf16<FMT>(cw, tl, th, vh);
            if constexpr (NA == 2) expand_bf16<FMT>(cw, ul, uh, vl);
            tmem_st16(lane_base + a_col<NA>(slot, 0) + 16 * bb, vh);
            if constexpr (NA == 2) tmem_st16(lane_base + a_col<NA>(slot, 1) + 16 * bb, vl);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.full_a[slot]);
        }
        ks += nsc;
        if (sm.abort) break;
      }
    }
    cp_async_wait<0>();
  } else if (warp == kBWarp) {
    // ------------------------------------------------------------ activation producer
    int ks = 0, g = a.g0;  // ks: stages issued
    for (int ti = blockIdx.x; ti < ntiles && !sm.abort; ti += gridDim.x) {
      g = group_from(a, t_begin + ti, g, lane);
      const TileInfo t = tile_at(a, t_begin + ti, g);
      const int y0 = t.off + t.tt * kTN;
      const int nv = min(kTN, t.n - t.tt * kTN);          // >= 1
      const int nbox = (nv + kBoxRows - 1) / kBoxRows;
      const uint32_t nm = static_cast<uint32_t>(min(kTN, (nv + 15) & ~15));
      for (int p = 0; p < nstages; ++p, ++ks) {
        const int slot = ks % kStages;
        if (ks >= kStages && !warp_wait<FMT>(sm, &sm.empty[slot], ((ks / kStages) - 1) & 1, a.status)) break;
        if (lane == 0) {
          sm.nmma[slot] = nm;
          mbar_arrive_expect_tx(&sm.full_b[slot], static_cast<uint32_t>(2 * nbox * kBoxRows * 128));
          for (int bx = 0; bx < nbox; ++bx) {
            tma_load_2d(sm.b[slot][0] + bx * kBoxRows * 128, &tm_hi, 64 * p, y0 + bx * kBoxRows, &sm.full_b[slot]);
            tma_load_2d(sm.b[slot][1] + bx * kBoxRows * 128, &tm_lo, 64 * p, y0 + bx * kBoxRows, &sm.full_b[slot]);
          }
        }
        __syncwarp();
      }
    }
    // the copies of the last use of each slot have landed before the CTA may
    // exit (they have, unless a wait ran out and the MMA stopped consuming)
    if (lane == 0) {
      for (int j = max(0, ks - kStages); j < ks; ++j) {
        bool done = false;
        for (uint32_t i = 0; i < kDrainLimit && !done; ++i)
          done = mbar_try_wait_sleep(&sm.full_b[j % kStages], (j / kStages) & 1);
        if (!done) {
          set_status(a.status, MOEQ_ERR_DEVICE_TIMEOUT);
          break;
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue (one thread)
    if (lane == 0) {
      // descriptor of b[slot][pb]: the parts are 16 KB apart, 1024 in the address field (addr >> 4)
      const uint64_t bdesc0 = sw128_desc(smem_u32(sm.b[0][0]));
      static_assert(sizeof(sm.b[0][0]) == 16384, "B part size");
      int ks = 0, kt = 0;
      bool ok = true;
      for (int ti = blockIdx.x; ti < ntiles && ok; ti += gridDim.x, ++kt) {
        const int tb = kt % kAccBufs;
        if (kt >= kAccBufs && !(ok = ring_wait<FMT>(sm, &sm.acc_empty[tb], ((kt / kAccBufs) - 1) & 1, a.status)))
          break;
        tc_fence_after();
        const uint32_t dcol = tmem + static_cast<uint32_t>(tb * kTN);
        for (int p = 0; p < nstages && ok; ++p, ++ks) {
          const int slot = ks % kStages;
          if (!(ok = ring_wait<FMT>(sm, &sm.full_b[slot], (ks / kStages) & 1, a.status))) break;
          if (!(ok = ring_wait<FMT>(sm, &sm.full_a[slot], (ks / kStages) & 1, a.status))) break;
          tc_fence_after();
          const uint32_t idesc = kIdescM | ((sm.nmma[slot] >> 3) << 17);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // products a_hi x_hi, a_hi x_lo (and a_lo x_hi for two weight parts)
#pragma unroll
            for (int pr = 0; pr < NA + 1; ++pr) {
              const int pa = pr == 2 ? 1 : 0, pb = pr == 1 ? 1 : 0;
              const uint64_t bd = bdesc0 + static_cast<uint64_t>((2 * slot + pb) * 1024 + 2 * kk);
              mma_bf16_ts(dcol, tmem + a_col<NA>(slot, pa) + 8 * kk, bd, idesc,
                          (p > 0 || kk > 0 || pr > 0) ? 1u : 0u);
            }
          }
          mma_commit(&sm.empty[slot]);
        }
        if (ok) mma_commit(&sm.acc_full[tb]);
      }
      // TMEM is released only after every MMA this thread issued has completed
      // (also when a wait above ran out and the loops were left early)
      mma_commit(&sm.drain);
      bool drained = false;
      for (uint32_t i = 0; i < kDrainLimit && !drained; ++i) drained = mbar_try_wait_sleep(&sm.drain, 0);
      if (!drained) set_status(a.status, MOEQ_ERR_DEVICE_TIMEOUT);
      sm.drained = drained ? 1 : 0;
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue (once per tile)
    const int q = warp & 3;                // TMEM lane quarter = rows 32q .. 32q + 31
    const int half = (warp - kEpiWarp0) >> 2;  // columns 64 half .. 64 half + 63
    const int r = 32 * q + lane;
    int kt = 0, g = a.g0;
    for (int ti = blockIdx.x; ti < ntiles; ti += gridDim.x, ++kt) {
      g = group_from(a, t_begin + ti, g, lane);
      const TileInfo t = tile_at(a, t_begin + ti, g);
      const int tb = kt % kAccBufs;
      if (!warp_wait<FMT>(sm, &sm.acc_full[tb], (kt / kAccBufs) & 1, a.status)) break;
      tc_fence_after();
      const int nv = min(kTN, t.n - t.tt * kTN);
      const size_t rowcol = static_cast<size_t>(t.m0 + r);
      constexpr int CW = EPI == EPI_SWIGLU ? 16 : 32;  // columns per TMEM read
      for (int c0 = 64 * half; c0 < min(nv, 64 * half + 64); c0 += CW) {
        float acc[CW];
        const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(tb * kTN + c0);
#pragma unroll
        for (int i = 0; i < CW; i += 16) tmem_ld16(taddr + i, acc + i);
        tmem_wait_ld();
        float gpre[EPI == EPI_SWIGLU ? CW : 1];
        if constexpr (EPI == EPI_SWIGLU) {  // the chunk's g values first: independent loads in flight
#pragma unroll
          for (int j = 0; j < CW; ++j) {
            const int jr = t.tt * kTN + c0 + j;
            gpre[j] = jr < t.n ? __ldcg(&a.g[static_cast<size_t>(t.off + jr) * a.R + rowcol]) : 0.0f;
          }
        }
#pragma unroll
        for (int j = 0; j < CW; ++j) {
          const int jr = t.tt * kTN + c0 + j;
          if (jr >= t.n) continue;  // warp-uniform
          const size_t grow = static_cast<size_t>(t.off + jr);
          const size_t at = grow * a.R + rowcol;
          if constexpr (EPI == EPI_G) {
            a.g[at] = acc[j];
          } else if constexpr (EPI == EPI_O) {
            a.o[at] = acc[j];
            if (a.dbg.o) {
              int tk, s;
              pid_split(a, a.pid[grow], tk, s);
              a.dbg.o[(static_cast<size_t>(tk) * a.ns + s) * a.R + rowcol] = acc[j];
            }
          } else {
            const float gv = gpre[j], u = acc[j];
            const float h = gv * u / (1.0f + expf(-gv));
            const int blk = (t.m0 + 32 * q) / 32;
            float vv = h;
            if (a.signs_h) vv = h32_warp(vv, __ldg(&a.signs_h[blk]), lane);
            uint16_t db;
            const int8_t qv = q8_warp(vv, db);
            // h's parts for the down GEMM: q * d (exact in fp32) as bf16 hi + lo
            const float pv = __fmul_rn(static_cast<float>(qv), f16_bits_to_f32(db));
            const uint32_t hp = bf16x2_rn(pv, 0.0f);
            a.hhi[at] = static_cast<uint16_t>(hp & 0xffffu);
            a.hlo[at] = static_cast<uint16_t>(bf16x2_rn(__fsub_rn(pv, bf16_lo_f(hp)), 0.0f) & 0xffffu);
            if (a.dbg.h || a.dbg.hq || a.dbg.hd) {
              int tk, s;
              pid_split(a, a.pid[grow], tk, s);
              const size_t vec = static_cast<size_t>(tk) * a.ns + s;
              if (a.dbg.h) a.dbg.h[vec * a.R + rowcol] = h;
              if (a.dbg.hq) a.dbg.hq[vec * a.R + rowcol] = qv;
              if (a.dbg.hd && lane == 0) a.dbg.hd[vec * (a.R / 32) + blk] = db;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.acc_empty[tb]);
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  // TMEM is released only once no MMA of this CTA can still write it; if the
  // drain wait itself ran out (broken hardware, reported in the status), the
  // CTA exits holding it rather than free columns under an MMA in flight
  if (warp == kMmaWarp && sm.drained) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "n"(kTmemCols));
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// bf16 [rows x K] activation parts, boxes of 64 K-elements x 64 rows, 128-byte swizzle.
int act_map(EncodeTiledFn enc, CUtensorMap* tm, const uint16_t* base, int K, int rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {64, kBoxRows};
  const cuuint32_t es[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? MOEQ_OK
             : MOEQ_ERR_CUDA;
}

template <int FMT, int EPI>
int launch_tc(const CUtensorMap& th, const CUtensorMap& tl, const TcArgs& a, int grid, cudaStream_t s) {
  const size_t smem = sizeof(TcSmem<FMT>) + 1024;
  if (smem > device_info().max_smem_optin) return MOEQ_ERR_SHAPE;
  if (cudaFuncSetAttribute(tc_gemm_kernel<FMT, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MOEQ_ERR_CUDA;
  tc_gemm_kernel<FMT, EPI><<<grid, kTcThreads, smem, s>>>(th, tl, a);
  return cuda_status(cudaGetLastError());
}

template <int EPI>
int launch_fmt(int fmt, const CUtensorMap& th, const CUtensorMap& tl, const TcArgs& a, int grid, cudaStream_t s) {
  if (fmt == 2) return launch_tc<2, EPI>(th, tl, a, grid, s);
  if (fmt == 3) return launch_tc<3, EPI>(th, tl, a, grid, s);
  return launch_tc<4, EPI>(th, tl, a, grid, s);
}

}  // namespace

int tc_grouped_gemm(const TcGemm& g, cudaStream_t s) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return MOEQ_ERR_CUDA;
  if (g.K % 128 || g.R % kTM) return MOEQ_ERR_SHAPE;  // an even number of 64-element stages
  CUtensorMap th, tl;
  int rc = act_map(enc, &th, g.act_hi, g.K, g.rows);
  if (!rc) rc = act_map(enc, &tl, g.act_lo, g.K, g.rows);
  if (rc) return rc;
  TcArgs a{};
  a.w = g.w;
  a.shared = g.shared;
  a.g0 = g.g0;
  a.g1 = g.g1;
  a.toff = g.toff;
  a.offsets = g.offsets;
  a.K = g.K;
  a.R = g.R;
  a.rows = g.rows;
  a.g = g.g;
  a.hhi = g.hhi;
  a.hlo = g.hlo;
  a.signs_h = g.signs_h;
  a.o = g.o;
  a.pid = g.pid;
  a.T = g.T;
  a.k = g.k;
  a.ns = g.ns;
  a.dbg = g.dbg;
  a.status = g.status;
  const int grid = device_info().sm_count;
  if (g.epi == EPI_G) return launch_fmt<EPI_G>(g.w.fmt, th, tl, a, grid, s);
  if (g.epi == EPI_SWIGLU) return launch_fmt<EPI_SWIGLU>(g.w.fmt, th, tl, a, grid, s);
  return launch_fmt<EPI_O>(g.w.fmt, th, tl, a, grid, s);
}

}  // namespace moeq
