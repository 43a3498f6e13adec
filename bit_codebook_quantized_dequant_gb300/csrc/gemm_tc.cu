// Grouped GEMMs of the prefill on the 5th-generation tensor cores (tcgen05).
//
// One tile = 128 weight rows x 64 grouped rows (tokens of one expert), the
// whole contraction K in 32-element blocks. Per block the exact integer dot
// products S[r, t] = sum_j cb[code] q are formed by tcgen05.mma kind::f16 on
// bf16 operands (|cb|, |q| <= 127: every product and every 32-term sum is
// exact in the fp32 accumulator), and the epilogue warps promote them with
// the block scales in fp32, acc = fma(ws[r,b] * xd[t,b], S, acc), in block
// order -- the same operations as the CUDA-core formulation, so the results
// are those of the decode's arithmetic up to the order of the final sums.
//
// Warp roles (16 warps):
//   0-3   expansion: thread = weight row; packed codes arrive by cp.async into
//         a per-row shared buffer, are expanded to bf16 with byte-permute
//         lookups in the codebook (low and high bytes of the bf16 values) and
//         written in the 128-byte-swizzled K-major layout of the MMA operand;
//         the row's block scales go to the scale ring
//   4     activation producer: one TMA (cp.async.bulk.tensor, SWIZZLE_128B)
//         per 2 blocks of the tile's 64 grouped bf16 rows; their block scales
//         go to the scale ring
//   5     MMA issuer (one thread) and TMEM owner (512 columns)
//   8-15  epilogue: two warpgroups, each the 128 rows x 32 columns of the
//         accumulators (gate and up for the gate/up GEMM); tcgen05.ld per
//         block, promotion, then SwiGLU + H32 + Q8 of h (a 32-block of h is
//         the 32 rows of one warp) or the fp32 output rows.
// Rings (mbarriers, every wait bounded): operand slots (2 blocks each), TMEM
// accumulator buffers (1 block each), scale slots (2 blocks each).
//
// Sources: "DeepSeek V4 Flash: 284B model, up to 32 tok/s on AMD Ryzen AI MAX+
// 395", section "ROCmFPX: fitting 284B weights into 128 GB" (small codebooks
// expanded on the fly, integer dot products); "deepseek-v4-flash-0731-evox3-
// rocm", section "The optimization ladder" (fused multi-token prefill with H32).
#include <cuda.h>
#include <cuda_runtime.h>

#include "moeq.h"
#include "moeq_device.cuh"
#include "moeq_host.h"
#include "moeq_layout.h"

namespace moeq {
namespace {

constexpr int kTM = 128;       // weight rows per tile
constexpr int kTN = 64;        // grouped rows per tile
constexpr int kKC = 8;         // 32-blocks per raw code chunk
constexpr int kSlots = 3;      // operand slots (2 blocks each)
constexpr int kBufs = 4;       // TMEM accumulator buffers (1 block each)
constexpr int kScs = 6;        // scale slots (2 blocks each)
constexpr int kXd = 4;         // pairs the activation scales are fetched ahead
constexpr int kXr = 8;         // their staging ring (> kXd)
constexpr int kTcThreads = 512;
constexpr int kBWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kEpiWarp0 = 8;
constexpr uint32_t kTmemCols = 512;

template <int FMT>
struct TcSmem {
  static constexpr int BC = block_bytes<FMT>();
  // raw row: the chunk's codes, then its block scales (<= 16 B); the pitch
  // also keeps the rows of a warp on different banks
  static constexpr int RP = kKC * BC + 16;
  uint8_t a[kSlots][2][kTM * 128];          // A operand: 128 rows x 64 bf16, SW128 K-major
  uint8_t b[kSlots][kTN * 128];             // B operand: 64 rows x 64 bf16, SW128 K-major
  uint8_t raw[2][2][kTM][RP];               // packed code chunks [stage][matrix][row]
  float ws[kScs][2][2][kTM];                // weight block scales [slot][block][matrix][row]
  float xd[kScs][2][kTN];                   // activation block scales [slot][block][row]
  uint32_t xraw[kXr][kTN];                  // fp16 pairs of activation scales, kXd pairs ahead
  uint64_t ab_full[kSlots], ab_empty[kSlots];
  uint64_t acc_full[kBufs], acc_empty[kBufs];
  uint64_t sc_full[kScs], sc_empty[kScs];
  uint64_t drain;                           // completion of every MMA this CTA issued
  uint32_t tmem_base;
  volatile int abort;
};

struct TcArgs {
  int gu;
  DMat wa, wb;
  int shared, g0, g1;
  const int* toff;
  const int* offsets;
  int K, R, rows;
  const uint16_t* act_scale;  // fp16 [rows x K/32]
  int8_t* hq;
  uint16_t* hd;
  uint16_t* hbf;
  const uint32_t* signs_h;
  float* o;
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

// kind::f16, bf16 A and B, fp32 D, both K-major, M = 128, N = kTN.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((kTN >> 3) << 17) | ((kTM >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t ad, uint64_t bd, uint32_t accumulate) {
  asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
               :: "r"(d_tmem), "l"(ad), "l"(bd), "r"(kIdesc), "r"(accumulate));
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

// Packed fp32 pairs (each lane an IEEE fp32 operation, round to nearest).
__device__ __forceinline__ uint64_t pack2(float x, float y) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& x, float& y) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(v));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

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
// 4- or 8-byte asynchronous copies (cache-all variant); src_bytes 0 fills zeros.
__device__ __forceinline__ void cp_async4(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" :: "r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" :: "r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

// mbarrier phase test that lets the hardware suspend the thread (up to 1 us)
// until the phase completes, instead of spinning on issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 1000;\n"
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

// Warp-wide form: lane 0 waits, the result is broadcast.
template <int FMT>
__device__ __forceinline__ bool warp_wait(TcSmem<FMT>& sm, uint64_t* bar, uint32_t parity, int32_t* status,
                                          int lane) {
  bool ok = true;
  if (lane == 0) ok = ring_wait<FMT>(sm, bar, parity, status);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// ---------------------------------------------------------------- codebook expansion to bf16
__device__ __forceinline__ uint32_t bf16_bits_of_int(int v) {
  return __float_as_uint(static_cast<float>(v)) >> 16;  // exact for |v| < 256
}

// Low and high bytes of the bf16 values of a codebook of n entries, 4 per word.
__device__ __forceinline__ void cb_tables(const int8_t* cb, int n, uint32_t* lo, uint32_t* hi) {
  for (int w = 0; w < n / 4; ++w) {
    uint32_t l = 0, h = 0;
    for (int j = 0; j < 4; ++j) {
      const uint32_t b = bf16_bits_of_int(cb[4 * w + j]);
      l |= (b & 0xffu) << (8 * j);
      h |= (b >> 8) << (8 * j);
    }
    lo[w] = l;
    hi[w] = h;
  }
}

// bf16 pairs of 4 elements from their low and high bytes.
__device__ __forceinline__ void interleave4(uint32_t lo, uint32_t hi, uint32_t* out) {
  out[0] = prmt(lo, hi, 0x5140u);
  out[1] = prmt(lo, hi, 0x7362u);
}

// One block (32 codes at p) -> 16 words of bf16 pairs (elements 2i, 2i+1 in word i).
template <int FMT>
__device__ __forceinline__ void expand_bf16(const uint8_t* p, const uint32_t* tl, const uint32_t* th,
                                            uint32_t* out) {
  if constexpr (FMT == 2) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    const uint32_t ws[2] = {w.x, w.y};
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t sa = ws[q] & 0x33333333u, sb = (ws[q] >> 2) & 0x33333333u;
      const uint32_t sel[4] = {sa, sa >> 16, sb, sb >> 16};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        interleave4(prmt(tl[0], tl[0], sel[i]), prmt(th[0], th[0], sel[i]), out + 8 * q + 2 * i);
    }
  } else if constexpr (FMT == 3) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(p);
    const Fp3Sel s = fp3_selectors(w[0], w[1], w[2]);
    const uint32_t sel[8] = {s.s00, s.s00 >> 16, s.s01, s.s01 >> 16, s.s10, s.s10 >> 16, s.s11, s.s11 >> 16};
#pragma unroll
    for (int i = 0; i < 8; ++i)
      interleave4(prmt(tl[0], tl[1], sel[i]), prmt(th[0], th[1], sel[i]), out + 2 * i);
  } else {
    const uint4 wd = *reinterpret_cast<const uint4*>(p);
    const uint32_t ws[4] = {wd.x, wd.y, wd.z, wd.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t l0, l1, h0, h1;
      fp4_expand(ws[q], tl[0], tl[1], tl[2], tl[3], l0, l1);
      fp4_expand(ws[q], th[0], th[1], th[2], th[3], h0, h1);
      interleave4(l0, h0, out + 4 * q);
      interleave4(l1, h1, out + 4 * q + 2);
    }
  }
}

struct TileInfo {
  int g, e, m0, tt, off, n;
};

__device__ __forceinline__ TileInfo tile_info(const TcArgs& a, int tile) {
  int lo = a.g0, hi = a.g1 - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(&a.toff[mid]) <= tile) lo = mid;
    else hi = mid - 1;
  }
  TileInfo t;
  t.g = lo;
  const int local = tile - __ldg(&a.toff[lo]);
  const int rtiles = a.R / kTM;
  t.tt = local / rtiles;
  t.m0 = (local % rtiles) * kTM;
  t.e = a.shared ? 0 : lo;
  t.off = __ldg(&a.offsets[lo]);
  t.n = __ldg(&a.offsets[lo + 1]) - t.off;
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

// Timeline event of CTA 0 (debug only): role 0 expansion, 1 producer, 2 MMA,
// 3 epilogue; (globaltimer ns, event << 32 | counter).
__device__ __forceinline__ void tc_trace(const TcArgs& a, int role, int& n, uint32_t ev, int ctr) {
  if (a.dbg.trace && blockIdx.x == 0 && n < a.dbg.trace_cap) {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    uint64_t* p = a.dbg.trace + 2 * (static_cast<size_t>(role) * a.dbg.trace_cap + n);
    p[0] = t;
    p[1] = (static_cast<uint64_t>(ev) << 32) | static_cast<uint32_t>(ctr);
  }
  ++n;
}

// ---------------------------------------------------------------- kernel
template <int FMT, bool GU>
__global__ void __launch_bounds__(kTcThreads, 1) tc_gemm_kernel(const __grid_constant__ CUtensorMap tm_act,
                                                                const TcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  TcSmem<FMT>& sm = *reinterpret_cast<TcSmem<FMT>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr int BC = block_bytes<FMT>();
  constexpr int NM = GU ? 2 : 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = a.K / 32;
  const int npairs = nb / 2;
  const int t_begin = __ldg(&a.toff[a.g0]);
  const int ntiles = __ldg(&a.toff[a.g1]) - t_begin;

  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&sm.ab_full[i], 5);   // 4 expansion warps + the activation producer (+ its bytes)
      mbar_init(&sm.ab_empty[i], 1);  // MMA commit
    }
    for (int i = 0; i < kBufs; ++i) {
      mbar_init(&sm.acc_full[i], 1);  // MMA commit
      mbar_init(&sm.acc_empty[i], 8); // epilogue warps
    }
    for (int i = 0; i < kScs; ++i) {
      mbar_init(&sm.sc_full[i], 5);
      mbar_init(&sm.sc_empty[i], 8);
    }
    mbar_init(&sm.drain, 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(&sm.tmem_base)), "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp < 4) {
    // ------------------------------------------------------------ expansion (thread = row)
    const int r = tid;
    int ks = 0, ntr = 0;
    for (int ti = blockIdx.x; ti < ntiles && !sm.abort; ti += gridDim.x) {
      const TileInfo t = tile_info(a, t_begin + ti);
      uint32_t tl[2][4], th[2][4];
#pragma unroll
      for (int m = 0; m < NM; ++m) {
        const DMat& M = m == 0 ? a.wa : a.wb;
        cb_tables(M.cb + static_cast<size_t>(t.e) * M.cb_stride, 1 << FMT, tl[m], th[m]);
      }
      const size_t row = static_cast<size_t>(t.m0 + r);
      // one chunk of the row: its codes and its block scales, by asynchronous copies
      auto issue_chunk = [&](int c) {
        constexpr int SB = FMT == 4 ? 1 : 2;
        const int kc = c * kKC, kb = min(kKC, nb - kc);
        const int pieces = kb * BC / 16;
#pragma unroll
        for (int m = 0; m < NM; ++m) {
          const DMat& M = m == 0 ? a.wa : a.wb;
          const uint8_t* src = M.codes + static_cast<size_t>(t.e) * M.stride_codes + (row * nb + kc) * BC;
          uint8_t* dst = sm.raw[c & 1][m][r];
          for (int i = 0; i < pieces; ++i) cp_async16(dst + 16 * i, src + 16 * i);
          const size_t soff = (row * nb + kc) * SB;
          const uint8_t* ssrc = M.scales + static_cast<size_t>(t.e) * M.stride_scales + soff;
          uint8_t* sdst = dst + kKC * BC;
          const int sbytes = kb * SB;  // 4, 8 or 16; soff is aligned to the piece used
          if (sbytes % 16 == 0 && soff % 16 == 0) {
            for (int i = 0; i < sbytes; i += 16) cp_async16(sdst + i, ssrc + i);
          } else if (sbytes % 8 == 0 && soff % 8 == 0) {
            for (int i = 0; i < sbytes; i += 8) cp_async8(sdst + i, ssrc + i);
          } else {
            for (int i = 0; i < sbytes; i += 4) cp_async4(sdst + i, ssrc + i, 4);
          }
        }
        cp_async_commit();
      };
      const int nchunks = (nb + kKC - 1) / kKC;
      issue_chunk(0);
      for (int c = 0; c < nchunks; ++c) {
        if (c + 1 < nchunks) {
          issue_chunk(c + 1);
          cp_async_wait<1>();
        } else {
          cp_async_wait<0>();
        }
        if (tid == 0) tc_trace(a, 0, ntr, 4, c);
        const int kc = c * kKC, kb = min(kKC, nb - kc);
        for (int jp = 0; jp < kb / 2; ++jp, ++ks) {
          const int slot = ks % kSlots, scs = ks % kScs;
          if (tid == 0) tc_trace(a, 0, ntr, 1, ks);
          if (ks >= kSlots && !warp_wait<FMT>(sm, &sm.ab_empty[slot], ((ks / kSlots) - 1) & 1, a.status, lane)) break;
          if (tid == 0) tc_trace(a, 0, ntr, 2, ks);
          float wsr[NM][2];
#pragma unroll
          for (int m = 0; m < NM; ++m)
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
              const uint8_t* sp = &sm.raw[c & 1][m][r][kKC * BC];
              if constexpr (FMT == 4) wsr[m][hb] = e8m0_to_f32(sp[2 * jp + hb]);
              else wsr[m][hb] = f16_bits_to_f32(reinterpret_cast<const uint16_t*>(sp)[2 * jp + hb]);
            }
#pragma unroll
          for (int m = 0; m < NM; ++m) {
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
              uint32_t v[16];
              expand_bf16<FMT>(&sm.raw[c & 1][m][r][(2 * jp + hb) * BC], tl[m], th[m], v);
              uint8_t* rowp = sm.a[slot][m] + r * 128;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int ch = (4 * hb + i) ^ (r & 7);
                *reinterpret_cast<uint4*>(rowp + 16 * ch) = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
              }
            }
          }
          if (tid == 0) tc_trace(a, 0, ntr, 3, ks);
          if (ks >= kScs && !warp_wait<FMT>(sm, &sm.sc_empty[scs], ((ks / kScs) - 1) & 1, a.status, lane)) break;
#pragma unroll
          for (int m = 0; m < NM; ++m)
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) sm.ws[scs][hb][m][r] = wsr[m][hb];
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&sm.ab_full[slot]);
            mbar_arrive(&sm.sc_full[scs]);
          }
        }
        if (sm.abort) break;
      }
    }
    cp_async_wait<0>();
  } else if (warp == kBWarp) {
    // ------------------------------------------------------------ activation producer
    int ks = 0, ntr = 0;
    for (int ti = blockIdx.x; ti < ntiles && !sm.abort; ti += gridDim.x) {
      const TileInfo t = tile_info(a, t_begin + ti);
      const int y0 = t.off + t.tt * kTN;
      // the 2 fp16 scales of a pair for rows lane and lane + 32, kXd pairs ahead
      // (one copy group per pair; a lane only reads what it copied)
      auto fetch_xd = [&](int p) {
        if (p < npairs) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int j = lane + 32 * h, jr = t.tt * kTN + j;
            const uint16_t* src = a.act_scale + static_cast<size_t>(t.off + (jr < t.n ? jr : 0)) * nb + 2 * p;
            cp_async4(&sm.xraw[p % kXr][j], src, jr < t.n ? 4u : 0u);
          }
        }
        cp_async_commit();
      };
      for (int p = 0; p < kXd; ++p) fetch_xd(p);
      for (int p = 0; p < npairs; ++p, ++ks) {
        const int slot = ks % kSlots, scs = ks % kScs;
        if (ks >= kSlots && !warp_wait<FMT>(sm, &sm.ab_empty[slot], ((ks / kSlots) - 1) & 1, a.status, lane)) break;
        if (lane == 0) tc_trace(a, 1, ntr, 2, ks);
        if (lane == 0) {
          mbar_arrive_expect_tx(&sm.ab_full[slot], kTN * 128);
          tma_load_2d(sm.b[slot], &tm_act, 64 * p, y0, &sm.ab_full[slot]);
        }
        if (ks >= kScs && !warp_wait<FMT>(sm, &sm.sc_empty[scs], ((ks / kScs) - 1) & 1, a.status, lane)) break;
        fetch_xd(p + kXd);
        cp_async_wait<kXd>();  // this pair's group has landed
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t v = sm.xraw[p % kXr][lane + 32 * h];
          sm.xd[scs][0][lane + 32 * h] = f16_bits_to_f32(static_cast<uint16_t>(v & 0xffffu));
          sm.xd[scs][1][lane + 32 * h] = f16_bits_to_f32(static_cast<uint16_t>(v >> 16));
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sm.sc_full[scs]);
          tc_trace(a, 1, ntr, 5, ks);
        }
      }
      cp_async_wait<0>();
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue (one thread)
    if (lane == 0) {
      int ks = 0, kg = 0, ntr = 0;
      bool ok = true;
      for (int ti = blockIdx.x; ti < ntiles && ok; ti += gridDim.x) {
        for (int p = 0; p < npairs && ok; ++p, ++ks) {
          const int slot = ks % kSlots;
          if (!(ok = ring_wait<FMT>(sm, &sm.ab_full[slot], (ks / kSlots) & 1, a.status))) break;
          tc_trace(a, 2, ntr, 2, ks);
          tc_fence_after();
          const uint32_t abase[2] = {smem_u32(sm.a[slot][0]), smem_u32(sm.a[slot][1])};
          const uint32_t bbase = smem_u32(sm.b[slot]);
#pragma unroll 1
          for (int hb = 0; hb < 2; ++hb, ++kg) {
            const int buf = kg % kBufs;
            if (kg >= kBufs && !(ok = ring_wait<FMT>(sm, &sm.acc_empty[buf], ((kg / kBufs) - 1) & 1, a.status)))
              break;
            tc_trace(a, 2, ntr, 6, kg);
            tc_fence_after();
            const uint32_t dcol = tmem + static_cast<uint32_t>(buf * (GU ? 2 * kTN : kTN));
#pragma unroll
            for (int m = 0; m < NM; ++m) {
#pragma unroll
              for (int s = 0; s < 2; ++s) {
                const uint32_t koff = static_cast<uint32_t>((2 * hb + s) * 32);
                mma_bf16(dcol + static_cast<uint32_t>(m * kTN), sw128_desc(abase[m] + koff),
                         sw128_desc(bbase + koff), s);
              }
            }
            mma_commit(&sm.acc_full[buf]);
          }
          if (ok) mma_commit(&sm.ab_empty[slot]);
        }
      }
      // TMEM is released only after every MMA this thread issued has completed
      // (also when a wait above ran out and the loops were left early)
      mma_commit(&sm.drain);
      bool drained = false;
      for (uint32_t i = 0; i < kSpinLimit && !drained; ++i) drained = mbar_try_wait_sleep(&sm.drain, 0);
      if (!drained) set_status(a.status, MOEQ_ERR_DEVICE_TIMEOUT);
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;           // TMEM lane quarter = rows 32q .. 32q + 31
    const int half = (warp - kEpiWarp0) >> 2;
    const int c0 = 32 * half;         // this warpgroup's 32 columns
    const int r = 32 * q + lane;
    int ks = 0, kg = 0, ntr = 0;
    bool ok = true;
    for (int ti = blockIdx.x; ti < ntiles && ok; ti += gridDim.x) {
      const TileInfo t = tile_info(a, t_begin + ti);
      uint64_t acc[NM][16];  // column pairs (2j, 2j + 1) of this warpgroup's 32 columns
#pragma unroll
      for (int m = 0; m < NM; ++m)
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[m][j] = 0ull;
      for (int p = 0; p < npairs && ok; ++p, ++ks) {
        const int scs = ks % kScs;
        if (!(ok = warp_wait<FMT>(sm, &sm.sc_full[scs], (ks / kScs) & 1, a.status, lane))) break;
#pragma unroll 1
        for (int hb = 0; hb < 2; ++hb, ++kg) {
          const int buf = kg % kBufs;
          if (!(ok = warp_wait<FMT>(sm, &sm.acc_full[buf], (kg / kBufs) & 1, a.status, lane))) break;
          if (tid == 32 * kEpiWarp0) tc_trace(a, 3, ntr, 6, kg);
          tc_fence_after();
          const float4* xdv = reinterpret_cast<const float4*>(&sm.xd[scs][hb][c0]);
#pragma unroll
          for (int m = 0; m < NM; ++m) {
            const float wsv = sm.ws[scs][hb][m][r];
            const uint64_t ws2 = pack2(wsv, wsv);
            const uint32_t col = static_cast<uint32_t>(buf * (GU ? 2 * kTN : kTN) + m * kTN + c0);
            const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + col;
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
              float S[16];
              tmem_ld16(taddr + 16 * ch, S);
              tmem_wait_ld();
              // acc = fma(ws * xd, S, acc) per column, two columns per instruction
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float4 x4 = xdv[4 * ch + i];
                const uint64_t sc0 = mul2(ws2, pack2(x4.x, x4.y));
                const uint64_t sc1 = mul2(ws2, pack2(x4.z, x4.w));
                acc[m][8 * ch + 2 * i] = fma2(sc0, pack2(S[4 * i], S[4 * i + 1]), acc[m][8 * ch + 2 * i]);
                acc[m][8 * ch + 2 * i + 1] = fma2(sc1, pack2(S[4 * i + 2], S[4 * i + 3]), acc[m][8 * ch + 2 * i + 1]);
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.acc_empty[buf]);
          if (tid == 32 * kEpiWarp0) tc_trace(a, 3, ntr, 7, kg);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.sc_empty[scs]);
      }
      if (!ok) break;
      if (tid == 32 * kEpiWarp0) tc_trace(a, 3, ntr, 8, ti);
      // tile epilogue: 32 columns of this warpgroup; row m0 + r (unrolled:
      // the accumulators stay in registers)
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int jr = t.tt * kTN + c0 + j;
        if (jr >= t.n) continue;  // warp-uniform
        const size_t grow = static_cast<size_t>(t.off + jr);
        float av[NM];
#pragma unroll
        for (int m = 0; m < NM; ++m) {
          float lo, hi;
          unpack2(acc[m][j / 2], lo, hi);
          av[m] = (j & 1) ? hi : lo;
        }
        if constexpr (GU) {
          const float g = av[0], u = av[NM - 1];
          const float h = g * u / (1.0f + expf(-g));
          const int blk = (t.m0 + 32 * q) / 32;
          float v = h;
          if (a.signs_h) v = h32_warp(v, __ldg(&a.signs_h[blk]), lane);
          uint16_t db;
          const int8_t qv = q8_warp(v, db);
          const size_t at = grow * a.R + t.m0 + r;
          a.hq[at] = qv;
          a.hbf[at] = static_cast<uint16_t>(bf16_bits_of_int(qv));
          if (lane == 0) a.hd[grow * (a.R / 32) + blk] = db;
          if (a.dbg.h || a.dbg.hq || a.dbg.hd) {
            int tk, s;
            pid_split(a, a.pid[grow], tk, s);
            const size_t vec = static_cast<size_t>(tk) * a.ns + s;
            if (a.dbg.h) a.dbg.h[vec * a.R + t.m0 + r] = h;
            if (a.dbg.hq) a.dbg.hq[vec * a.R + t.m0 + r] = qv;
            if (a.dbg.hd && lane == 0) a.dbg.hd[vec * (a.R / 32) + blk] = db;
          }
        } else {
          a.o[grow * a.R + t.m0 + r] = av[0];
          if (a.dbg.o) {
            int tk, s;
            pid_split(a, a.pid[grow], tk, s);
            a.dbg.o[(static_cast<size_t>(tk) * a.ns + s) * a.R + t.m0 + r] = av[0];
          }
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(kTmemCols));
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

template <int FMT, bool GU>
int launch_tc(const CUtensorMap& tm, const TcArgs& a, int grid, cudaStream_t s) {
  const size_t smem = sizeof(TcSmem<FMT>) + 1024;
  if (smem > device_info().max_smem_optin) return MOEQ_ERR_SHAPE;
  if (cudaFuncSetAttribute(tc_gemm_kernel<FMT, GU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MOEQ_ERR_CUDA;
  tc_gemm_kernel<FMT, GU><<<grid, kTcThreads, smem, s>>>(tm, a);
  return cuda_status(cudaGetLastError());
}

}  // namespace

int tc_grouped_gemm(const TcGemm& g, cudaStream_t s) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return MOEQ_ERR_CUDA;
  if (g.K % 64 || g.R % kTM) return MOEQ_ERR_SHAPE;
  // activations [rows x K] bf16, boxes of 64 K-elements x 64 rows, 128-byte swizzle
  CUtensorMap tm;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(g.K), static_cast<cuuint64_t>(g.rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(g.K) * 2};
  const cuuint32_t box[2] = {64, kTN};
  const cuuint32_t es[2] = {1, 1};
  if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(g.act), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return MOEQ_ERR_CUDA;
  TcArgs a{};
  a.gu = g.gu;
  a.wa = g.wa;
  a.wb = g.wb;
  a.shared = g.shared;
  a.g0 = g.g0;
  a.g1 = g.g1;
  a.toff = g.toff;
  a.offsets = g.offsets;
  a.K = g.K;
  a.R = g.R;
  a.rows = g.rows;
  a.act_scale = g.act_scale;
  a.hq = g.hq;
  a.hd = g.hd;
  a.hbf = g.hbf;
  a.signs_h = g.signs_h;
  a.o = g.o;
  a.pid = g.pid;
  a.T = g.T;
  a.k = g.k;
  a.ns = g.ns;
  a.dbg = g.dbg;
  a.status = g.status;
  const int grid = device_info().sm_count;
  const int fmt = g.wa.fmt;
  if (g.gu) {
    if (fmt == 2) return launch_tc<2, true>(tm, a, grid, s);
    if (fmt == 3) return launch_tc<3, true>(tm, a, grid, s);
    return launch_tc<4, true>(tm, a, grid, s);
  }
  if (fmt == 2) return launch_tc<2, false>(tm, a, grid, s);
  if (fmt == 3) return launch_tc<3, false>(tm, a, grid, s);
  return launch_tc<4, false>(tm, a, grid, s);
}

}  // namespace moeq
