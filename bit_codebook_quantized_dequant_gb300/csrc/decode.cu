// Batch-1 decode of one codebook-quantized MoE FFN layer in one persistent,
// cooperative, warp-specialized kernel.
//
// Work is cut into units taken from a global queue in dependency order:
//   router rows (8 per unit) -> shared-expert gate/up rows (16) -> routed
//   gate/up rows (16 per unit, slot-major) -> shared down rows (32) -> routed
//   down rows (32, slot-major).
// A unit only waits on units with a smaller queue index, and every CTA is
// resident (cooperative launch), so the waits always end; each is bounded
// anyway and reports MOEQ_ERR_DEVICE_TIMEOUT into the status word if it runs out.
//
// Per CTA: one producer warp takes units from the queue and streams their
// packed rows (codes plane and scale plane, contiguous per row range) from HBM
// into a 3-stage shared-memory ring with bulk asynchronous copies; it also
// computes the top-k once the router rows are done. Sixteen compute warps
// expand codes in registers (byte permutes), take int8 dot products per
// 32-block (dp4a) and apply the block scales in fp32:
//   * router unit : canonical-order bf16 logits, one warp per row;
//   * gate/up unit: one warp per row computes g and u, then h = silu(g) u;
//                   the CTA that finishes the second half of a 32-row block
//                   rotates (H32) and quantizes (Q8) that block of h;
//   * down unit   : one warp per two rows computes o; the CTA that writes the
//                   last slot of a 32-row chunk of y combines the slots in
//                   order: y = sum_s p_s o_s (+ o_shared).
// Sources: "DeepSeek V4 Flash: 284B model, up to 32 tok/s on AMD Ryzen AI MAX+
// 395", section "ROCmFPX: fitting 284B weights into 128 GB" (read packed blocks
// directly, expand small codebooks in registers, integer dot products, decode
// bound by weight traffic); "Lucebox x Geometric ...", section "Lucebox Engine
// integration with Geometric" (fused matvec, sync-free MoE decode).
#include <cuda_runtime.h>

#include "moeq.h"
#include "moeq_device.cuh"
#include "moeq_host.h"
#include "moeq_layout.h"

namespace moeq {
namespace {

constexpr int kComputeWarps = 16;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kThreads = kComputeThreads + 32;
constexpr int kStages = 3;
constexpr int kStageBytes = 68 * 1024;
constexpr int kRouterRows = 8;
constexpr int kGuRows = 16;
constexpr int kDownRows = 32;
constexpr int kMaxH = 4096;
constexpr int kMaxB = kMaxH / 32 / 32;  // 32-blocks per lane along K
constexpr int kMaxE = 512;
constexpr int kMaxEPerLane = kMaxE / 32;
constexpr int kBarCompute = 1;  // named barrier of the compute warps

enum UnitKind { U_ROUTER = 0, U_SGU, U_GU, U_SDOWN, U_DOWN, U_END };

struct Unit {
  int kind, slot, chunk;
};

struct DecodeArgs {
  int H, I, E, k, nslots, has_shared;
  const uint16_t* x;
  const uint16_t* router;
  DMat gate, up, down, sgate, sup, sdown;
  const uint32_t* signs_x;
  const uint32_t* signs_h;
  float* y;
  uint32_t* ctr;
  float* logits;
  float* hbuf;
  int8_t* hq;
  uint16_t* hd;
  float* obuf;
  int32_t* status;
  moeq_debug dbg;
  int nR, nSG, nGU, nSD, nD, total;
};

struct alignas(128) DecodeSmem {
  uint8_t stage[kStages][kStageBytes];
  uint16_t xb[kMaxH];
  int8_t xq[kMaxH];
  float xd[kMaxH / 32];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int unit[kStages];
  int idx[kMaxK];
  float p[kMaxK];
  int last_cta;
  int issued;    // stage fills issued by the producer
  int consumed;  // stage fills waited for by the compute warps
};

__device__ __forceinline__ Unit unit_of(const DecodeArgs& a, int u) {
  Unit r{U_END, 0, 0};
  if (u < 0) return r;
  if (u < a.nR) return Unit{U_ROUTER, 0, u};
  u -= a.nR;
  if (u < a.nSG) return Unit{U_SGU, a.k, u};
  u -= a.nSG;
  const int gu_per_slot = a.I / kGuRows;
  if (u < a.nGU) return Unit{U_GU, u / gu_per_slot, u % gu_per_slot};
  u -= a.nGU;
  if (u < a.nSD) return Unit{U_SDOWN, a.k, u};
  u -= a.nSD;
  const int d_per_slot = a.H / kDownRows;
  if (u < a.nD) return Unit{U_DOWN, u / d_per_slot, u % d_per_slot};
  return r;
}

// Byte offsets inside a stage: [codes A][scales A][codes B][scales B].
struct StageMap {
  uint32_t ca, sa, cb, sb, total;
};

__host__ __device__ __forceinline__ uint32_t al16(uint32_t x) { return (x + 15u) & ~15u; }

__host__ __device__ __forceinline__ StageMap gu_map(int fmt, int K) {
  const int nb = K / 32;
  const uint32_t c = kGuRows * nb * (fmt == 2 ? 8 : fmt == 3 ? 12 : 16);
  const uint32_t s = al16(kGuRows * nb * (fmt == 4 ? 1 : 2));
  return StageMap{0, c, c + s, c + s + c, 2 * (c + s)};
}

__host__ __device__ __forceinline__ StageMap down_map(int fmt, int K) {
  const int nb = K / 32;
  const uint32_t c = kDownRows * nb * (fmt == 2 ? 8 : fmt == 3 ? 12 : 16);
  const uint32_t s = al16(kDownRows * nb * (fmt == 4 ? 1 : 2));
  return StageMap{0, c, 0, 0, c + s};
}

// ------------------------------------------------------------------ producer side
__device__ void producer_topk(const DecodeArgs& a, DecodeSmem& sm, int lane) {
  if (lane == 0 && !spin_until_geq(&a.ctr[1], static_cast<uint32_t>(a.nR)))
    set_status(a.status, MOEQ_ERR_DEVICE_TIMEOUT);
  __syncwarp();
  const int nper = (a.E + 31) / 32;
  float v[kMaxEPerLane];
  uint32_t valid = 0;
#pragma unroll
  for (int i = 0; i < kMaxEPerLane; ++i) {
    const bool ok = i < nper && lane + 32 * i < a.E;
    v[i] = ok ? __ldcg(&a.logits[lane + 32 * i]) : 0.0f;
    valid |= (ok ? 1u : 0u) << i;
  }
  uint32_t taken = 0;
  int sel[kMaxK];
  float selv[kMaxK];
#pragma unroll
  for (int s = 0; s < kMaxK; ++s) {
    sel[s] = 0;
    selv[s] = 0.0f;
    if (s >= a.k) continue;
    float bv = 0.0f;
    int bi = -1;
#pragma unroll
    for (int i = 0; i < kMaxEPerLane; ++i) {
      if (!((valid >> i) & 1u) || ((taken >> i) & 1u)) continue;
      const int e = lane + 32 * i;
      if (bi < 0 || ranks_before(v[i], e, bv, bi)) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, d);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, d);
      if (oi >= 0 && (bi < 0 || ranks_before(ov, oi, bv, bi))) {
        bv = ov;
        bi = oi;
      }
    }
    if (bi >= 0 && (bi & 31) == lane) taken |= 1u << (bi >> 5);
    sel[s] = bi;
    selv[s] = bv;
  }
  // softmax over all E logits at the selected indices (max = the first selected)
  const float m = selv[0];
  float z = 0.0f;
#pragma unroll
  for (int i = 0; i < kMaxEPerLane; ++i)
    if (((valid >> i) & 1u) && !isnan(v[i])) z += expf(v[i] - m);
  z = warp_sum_canonical(z);
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kMaxK; ++s) {
      if (s >= a.k) continue;
      const float ps = __fdiv_rn(expf(selv[s] - m), z);
      sm.idx[s] = sel[s];
      sm.p[s] = ps;
      if (blockIdx.x == 0) {
        if (a.dbg.idx) a.dbg.idx[s] = sel[s];
        if (a.dbg.p) a.dbg.p[s] = ps;
      }
    }
  }
  __syncwarp();
}

__device__ __forceinline__ const DMat& gu_mat(const DecodeArgs& a, bool shared, bool up) {
  return shared ? (up ? a.sup : a.sgate) : (up ? a.up : a.gate);
}

// Issues the copies of unit un into stage s (lane 0 of the producer warp).
__device__ void issue_unit(const DecodeArgs& a, DecodeSmem& sm, int s, const Unit& un) {
  uint8_t* st = sm.stage[s];
  uint64_t* bar = &sm.full[s];
  if (un.kind == U_ROUTER) {
    const uint32_t bytes = kRouterRows * a.H * 2;
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(st, a.router + static_cast<size_t>(un.chunk) * kRouterRows * a.H, bytes, bar);
    return;
  }
  if (un.kind == U_SGU || un.kind == U_GU) {
    const bool shared = un.kind == U_SGU;
    const DMat& G = gu_mat(a, shared, false);
    const DMat& U = gu_mat(a, shared, true);
    const int e = shared ? 0 : sm.idx[un.slot];
    const int nb = a.H / 32;
    const size_t pc = static_cast<size_t>(nb) * (G.fmt == 2 ? 8 : G.fmt == 3 ? 12 : 16);
    const size_t ps = static_cast<size_t>(nb) * (G.fmt == 4 ? 1 : 2);
    const StageMap mp = gu_map(G.fmt, a.H);
    const size_t r0 = static_cast<size_t>(un.chunk) * kGuRows;
    const uint32_t cbytes = static_cast<uint32_t>(kGuRows * pc), sbytes = static_cast<uint32_t>(kGuRows * ps);
    mbar_arrive_expect_tx(bar, 2 * (cbytes + sbytes));
    bulk_g2s(st + mp.ca, G.codes + e * G.stride_codes + r0 * pc, cbytes, bar);
    bulk_g2s(st + mp.sa, G.scales + e * G.stride_scales + r0 * ps, sbytes, bar);
    bulk_g2s(st + mp.cb, U.codes + e * U.stride_codes + r0 * pc, cbytes, bar);
    bulk_g2s(st + mp.sb, U.scales + e * U.stride_scales + r0 * ps, sbytes, bar);
    return;
  }
  if (un.kind == U_SDOWN || un.kind == U_DOWN) {
    const bool shared = un.kind == U_SDOWN;
    const DMat& D = shared ? a.sdown : a.down;
    const int e = shared ? 0 : sm.idx[un.slot];
    const int nb = a.I / 32;
    const size_t pc = static_cast<size_t>(nb) * (D.fmt == 2 ? 8 : D.fmt == 3 ? 12 : 16);
    const size_t ps = static_cast<size_t>(nb) * (D.fmt == 4 ? 1 : 2);
    const StageMap mp = down_map(D.fmt, a.I);
    const size_t r0 = static_cast<size_t>(un.chunk) * kDownRows;
    const uint32_t cbytes = static_cast<uint32_t>(kDownRows * pc), sbytes = static_cast<uint32_t>(kDownRows * ps);
    mbar_arrive_expect_tx(bar, cbytes + sbytes);
    bulk_g2s(st + mp.ca, D.codes + e * D.stride_codes + r0 * pc, cbytes, bar);
    bulk_g2s(st + mp.sa, D.scales + e * D.stride_scales + r0 * ps, sbytes, bar);
    return;
  }
}

// ------------------------------------------------------------------ compute side
__device__ __forceinline__ void load_cb(const DMat& m, int e, uint32_t* cb) {
  const uint32_t* p = reinterpret_cast<const uint32_t*>(m.cb + static_cast<size_t>(e) * m.cb_stride);
  const int n = (1 << m.fmt) / 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) cb[i] = i < n ? __ldg(p + i) : 0u;
}

// One row of gate and up (same row index) against the quantized x in smem.
template <int FMT>
__device__ void gu_row(const DecodeArgs& a, const DecodeSmem& sm, const uint8_t* st,
                       const StageMap& mp, const uint32_t* cbg, const uint32_t* cbu, int r,
                       int grow, int slot, int lane, float& g, float& u) {
  constexpr int BC = block_bytes<FMT>();
  const int nb = a.H / 32;
  const uint8_t* gc = st + mp.ca + r * nb * BC;
  const uint8_t* uc = st + mp.cb + r * nb * BC;
  const uint8_t* gs = st + mp.sa + r * nb * (FMT == 4 ? 1 : 2);
  const uint8_t* us = st + mp.sb + r * nb * (FMT == 4 ? 1 : 2);
  float ag = 0.0f, au = 0.0f;
#pragma unroll
  for (int i = 0; i < kMaxB; ++i) {
    const int b = lane + 32 * i;
    if (b < nb) {
      int q[8];
      const int4 q0 = *reinterpret_cast<const int4*>(sm.xq + 32 * b);
      const int4 q1 = *reinterpret_cast<const int4*>(sm.xq + 32 * b + 16);
      q[0] = q0.x; q[1] = q0.y; q[2] = q0.z; q[3] = q0.w;
      q[4] = q1.x; q[5] = q1.y; q[6] = q1.z; q[7] = q1.w;
      const float xd = sm.xd[b];
      const int sg = block_dot<FMT>(gc + b * BC, cbg, q);
      const int su = block_dot<FMT>(uc + b * BC, cbu, q);
      ag = fmaf(block_scale<FMT>(gs, b) * xd, static_cast<float>(sg), ag);
      au = fmaf(block_scale<FMT>(us, b) * xd, static_cast<float>(su), au);
      if (a.dbg.S_gate) a.dbg.S_gate[(static_cast<size_t>(slot) * a.I + grow) * nb + b] = sg;
      if (a.dbg.S_up) a.dbg.S_up[(static_cast<size_t>(slot) * a.I + grow) * nb + b] = su;
    }
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) {
    ag += __shfl_xor_sync(0xffffffffu, ag, d);
    au += __shfl_xor_sync(0xffffffffu, au, d);
  }
  g = ag;
  u = au;
}

// Two rows (r, r + 16) of a down matrix against the quantized h of one slot.
template <int FMT>
__device__ void down_rows(const DecodeArgs& a, const uint8_t* st, const StageMap& mp,
                          const uint32_t* cb, const int (*q)[8], const float* hdf, int warp,
                          int lane, int chunk, int slot, float* o) {
  constexpr int BC = block_bytes<FMT>();
  const int nb = a.I / 32;
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int r = warp + 16 * rr;
    const uint8_t* c = st + mp.ca + r * nb * BC;
    const uint8_t* sc = st + mp.sa + r * nb * (FMT == 4 ? 1 : 2);
    float acc = 0.0f;
#pragma unroll
    for (int i = 0; i < kMaxB; ++i) {
      const int b = lane + 32 * i;
      if (b < nb) {
        const int sd = block_dot<FMT>(c + b * BC, cb, q[i]);
        acc = fmaf(block_scale<FMT>(sc, b) * hdf[i], static_cast<float>(sd), acc);
        if (a.dbg.S_down)
          a.dbg.S_down[(static_cast<size_t>(slot) * a.H + chunk * kDownRows + r) * nb + b] = sd;
      }
    }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, d);
    o[rr] = acc;
  }
}

__device__ void router_unit(const DecodeArgs& a, const DecodeSmem& sm, const uint8_t* st,
                            int chunk, int warp, int lane) {
  if (warp < kRouterRows) {
    const int e = chunk * kRouterRows + warp;
    const uint8_t* wrow = st + static_cast<size_t>(warp) * a.H * 2;
    float acc = 0.0f;
    for (int i = 0; i < a.H / 256; ++i) {
      const int k0 = 256 * i + 8 * lane;
      const uint4 w = *reinterpret_cast<const uint4*>(wrow + 2 * k0);
      const uint4 x = *reinterpret_cast<const uint4*>(sm.xb + k0);
      acc = fmaf(bf16_lo(x.x), bf16_lo(w.x), acc);
      acc = fmaf(bf16_hi(x.x), bf16_hi(w.x), acc);
      acc = fmaf(bf16_lo(x.y), bf16_lo(w.y), acc);
      acc = fmaf(bf16_hi(x.y), bf16_hi(w.y), acc);
      acc = fmaf(bf16_lo(x.z), bf16_lo(w.z), acc);
      acc = fmaf(bf16_hi(x.z), bf16_hi(w.z), acc);
      acc = fmaf(bf16_lo(x.w), bf16_lo(w.w), acc);
      acc = fmaf(bf16_hi(x.w), bf16_hi(w.w), acc);
    }
    acc = warp_sum_canonical(acc);
    if (lane == 0) {
      a.logits[e] = acc;
      if (a.dbg.logits) a.dbg.logits[e] = acc;
    }
  }
  named_bar(kBarCompute, kComputeThreads);
  if (warp == 0 && lane == 0) {
    __threadfence();
    atomicAdd(&a.ctr[1], 1u);
  }
}

template <int FMT>
__device__ void gu_unit(const DecodeArgs& a, DecodeSmem& sm, const uint8_t* st, const Unit& un,
                        int warp, int lane) {
  const bool shared = un.kind == U_SGU;
  const DMat& G = gu_mat(a, shared, false);
  const DMat& U = gu_mat(a, shared, true);
  const int e = shared ? 0 : sm.idx[un.slot];
  uint32_t cbg[4], cbu[4];
  load_cb(G, e, cbg);
  load_cb(U, e, cbu);
  const StageMap mp = gu_map(FMT, a.H);
  const int grow = un.chunk * kGuRows + warp;
  float g, u;
  gu_row<FMT>(a, sm, st, mp, cbg, cbu, warp, grow, un.slot, lane, g, u);
  if (lane == 0) {
    const float h = g * u / (1.0f + expf(-g));
    a.hbuf[static_cast<size_t>(un.slot) * a.I + grow] = h;
    if (a.dbg.h) a.dbg.h[static_cast<size_t>(un.slot) * a.I + grow] = h;
  }
  named_bar(kBarCompute, kComputeThreads);
  if (warp == 0) {
    // the second CTA to finish a half of this 32-row block quantizes the block
    const int nbI = a.I / 32, blk = un.chunk / 2;
    uint32_t old = 0;
    if (lane == 0) {
      __threadfence();
      old = atomicAdd(&a.ctr[kPairBase + un.slot * nbI + blk], 1u);
    }
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old == 1) {
      __threadfence();
      const size_t base = static_cast<size_t>(un.slot) * a.I + 32 * blk;
      float v = __ldcg(&a.hbuf[base + lane]);
      if (a.signs_h) v = h32_warp(v, __ldg(&a.signs_h[blk]), lane);
      uint16_t db;
      const int8_t q = q8_warp(v, db);
      a.hq[base + lane] = q;
      if (lane == 0) a.hd[static_cast<size_t>(un.slot) * nbI + blk] = db;
      if (a.dbg.hq) a.dbg.hq[base + lane] = q;
      if (a.dbg.hd && lane == 0) a.dbg.hd[static_cast<size_t>(un.slot) * nbI + blk] = db;
      __syncwarp();
      if (lane == 0) {
        __threadfence();
        atomicAdd(&a.ctr[kCtrHqDone + un.slot], 1u);
      }
    }
  }
}

template <int FMT>
__device__ void down_unit(const DecodeArgs& a, DecodeSmem& sm, const uint8_t* st, const Unit& un,
                          int warp, int lane) {
  const bool shared = un.kind == U_SDOWN;
  const DMat& D = shared ? a.sdown : a.down;
  const int e = shared ? 0 : sm.idx[un.slot];
  const int nbI = a.I / 32;
  if (warp == 0 && lane == 0 &&
      !spin_until_geq(&a.ctr[kCtrHqDone + un.slot], static_cast<uint32_t>(nbI)))
    set_status(a.status, MOEQ_ERR_DEVICE_TIMEOUT);
  named_bar(kBarCompute, kComputeThreads);
  __threadfence();
  uint32_t cb[4];
  load_cb(D, e, cb);
  int q[kMaxB][8];
  float hdf[kMaxB];
#pragma unroll
  for (int i = 0; i < kMaxB; ++i) {
    const int b = lane + 32 * i;
    if (b < nbI) {
      const size_t base = static_cast<size_t>(un.slot) * a.I + 32 * b;
      const int4 q0 = __ldcg(reinterpret_cast<const int4*>(a.hq + base));
      const int4 q1 = __ldcg(reinterpret_cast<const int4*>(a.hq + base + 16));
      q[i][0] = q0.x; q[i][1] = q0.y; q[i][2] = q0.z; q[i][3] = q0.w;
      q[i][4] = q1.x; q[i][5] = q1.y; q[i][6] = q1.z; q[i][7] = q1.w;
      hdf[i] = f16_bits_to_f32(__ldcg(a.hd + static_cast<size_t>(un.slot) * nbI + b));
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) q[i][j] = 0;
      hdf[i] = 0.0f;
    }
  }
  const StageMap mp = down_map(FMT, a.I);
  float o[2];
  down_rows<FMT>(a, st, mp, cb, q, hdf, warp, lane, un.chunk, un.slot, o);
  if (lane == 0) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const size_t at = static_cast<size_t>(un.slot) * a.H + un.chunk * kDownRows + warp + 16 * rr;
      a.obuf[at] = o[rr];
      if (a.dbg.o) a.dbg.o[at] = o[rr];
    }
  }
  named_bar(kBarCompute, kComputeThreads);
  if (warp == 0) {
    const int nchunks = a.H / kDownRows;
    uint32_t old = 0;
    if (lane == 0) {
      __threadfence();
      old = atomicAdd(&a.ctr[kPairBase + a.nslots * nbI + un.chunk], 1u);
    }
    old = __shfl_sync(0xffffffffu, old, 0);
    (void)nchunks;
    if (old == static_cast<uint32_t>(a.nslots - 1)) {
      __threadfence();
      const int row = un.chunk * kDownRows + lane;
      float acc = 0.0f;
      for (int s = 0; s < a.k; ++s) acc = fmaf(sm.p[s], __ldcg(&a.obuf[static_cast<size_t>(s) * a.H + row]), acc);
      if (a.has_shared) acc += __ldcg(&a.obuf[static_cast<size_t>(a.k) * a.H + row]);
      a.y[row] = acc;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  DecodeSmem& sm = *reinterpret_cast<DecodeSmem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kComputeWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kComputeWarps) {
    // ---------------------------------------------------------------- producer warp
    bool have_topk = false;
    int it = 0;
    for (;; ++it) {
      const int s = it % kStages;
      if (it >= kStages) {
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&sm.empty[s], ((it / kStages) - 1) & 1);
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
          set_status(a.status, MOEQ_ERR_DEVICE_TIMEOUT);
          break;
        }
      }
      int u = 0;
      if (lane == 0) u = static_cast<int>(atomicAdd(&a.ctr[0], 1u));
      u = __shfl_sync(0xffffffffu, u, 0);
      const Unit un = unit_of(a, u);
      if (un.kind == U_END) {
        if (lane == 0) {
          sm.unit[s] = -1;
          mbar_arrive(&sm.full[s]);
        }
        ++it;
        break;
      }
      if (!have_topk && un.kind != U_ROUTER && un.kind != U_SGU) {
        producer_topk(a, sm, lane);
        have_topk = true;
      }
      if (lane == 0) {
        sm.unit[s] = u;
        issue_unit(a, sm, s, un);
      }
      __syncwarp();
    }
    if (lane == 0) sm.issued = it;
  } else {
    // ---------------------------------------------------------------- compute warps
    const int nbH = a.H / 32;
    for (int i = tid; i < a.H / 8; i += kComputeThreads)
      reinterpret_cast<uint4*>(sm.xb)[i] = __ldg(reinterpret_cast<const uint4*>(a.x) + i);
    named_bar(kBarCompute, kComputeThreads);
    if (tid < nbH) {
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(static_cast<uint32_t>(sm.xb[32 * tid + j]) << 16);
      if (a.signs_x) h32_thread(v, __ldg(&a.signs_x[tid]));
      int qw[8];
      const uint16_t db = q8_thread(v, qw);
      reinterpret_cast<int4*>(sm.xq + 32 * tid)[0] = make_int4(qw[0], qw[1], qw[2], qw[3]);
      reinterpret_cast<int4*>(sm.xq + 32 * tid)[1] = make_int4(qw[4], qw[5], qw[6], qw[7]);
      sm.xd[tid] = f16_bits_to_f32(db);
      if (blockIdx.x == 0) {
        if (a.dbg.xq) {
          reinterpret_cast<int4*>(a.dbg.xq + 32 * tid)[0] = make_int4(qw[0], qw[1], qw[2], qw[3]);
          reinterpret_cast<int4*>(a.dbg.xq + 32 * tid)[1] = make_int4(qw[4], qw[5], qw[6], qw[7]);
        }
        if (a.dbg.xd) a.dbg.xd[tid] = db;
      }
    }
    named_bar(kBarCompute, kComputeThreads);

    int it = 0;
    bool aborted = false;
    for (;; ++it) {
      const int s = it % kStages;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&sm.full[s], (it / kStages) & 1);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      // one decision for all compute warps, so that a timeout never splits them
      if (!named_bar_and(kBarCompute, kComputeThreads, ok)) {
        if (tid == 0) set_status(a.status, MOEQ_ERR_DEVICE_TIMEOUT);
        aborted = true;
        break;
      }
      const int u = sm.unit[s];
      const Unit un = unit_of(a, u);
      if (un.kind == U_END) break;
      const uint8_t* st = sm.stage[s];
      if (un.kind == U_ROUTER) {
        router_unit(a, sm, st, un.chunk, warp, lane);
      } else if (un.kind == U_SGU || un.kind == U_GU) {
        const int fmt = un.kind == U_SGU ? a.sgate.fmt : a.gate.fmt;
        if (fmt == 2) gu_unit<2>(a, sm, st, un, warp, lane);
        else if (fmt == 3) gu_unit<3>(a, sm, st, un, warp, lane);
        else gu_unit<4>(a, sm, st, un, warp, lane);
      } else {
        const int fmt = un.kind == U_SDOWN ? a.sdown.fmt : a.down.fmt;
        if (fmt == 2) down_unit<2>(a, sm, st, un, warp, lane);
        else if (fmt == 3) down_unit<3>(a, sm, st, un, warp, lane);
        else down_unit<4>(a, sm, st, un, warp, lane);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[s]);
    }
    if (tid == 0) sm.consumed = aborted ? it - 1 : it;  // last fill waited for
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (warp == kComputeWarps && lane == 0) {
    // copies issued but never waited for (only after a timeout): let them land
    for (int j = sm.consumed + 1; j < sm.issued; ++j)
      if (!mbar_wait(&sm.full[j % kStages], (j / kStages) & 1)) break;
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const uint32_t old = atomicAdd(&a.ctr[2], 1u);
    sm.last_cta = old == gridDim.x - 1;
    if (sm.last_cta) __threadfence();
  }
  __syncthreads();
  if (sm.last_cta) {
    const int n = kPairBase + a.nslots * (a.I / 32) + a.H / kDownRows;
    for (int i = tid; i < n; i += kThreads)
      if (i != 2) a.ctr[i] = 0u;
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      a.ctr[2] = 0u;
    }
  }
}

}  // namespace

bool decode_supported(const moeq_layer* L) {
  if (L->H > kMaxH || L->I > kMaxH || L->E > kMaxE || L->E % kRouterRows || L->k > kMaxK) return false;
  if (static_cast<long>(kRouterRows) * L->H * 2 > kStageBytes) return false;
  if (gu_map(L->gate.fmt, L->H).total > static_cast<uint32_t>(kStageBytes)) return false;
  if (down_map(L->down.fmt, L->I).total > static_cast<uint32_t>(kStageBytes)) return false;
  if (L->has_shared) {
    if (gu_map(L->sgate.fmt, L->H).total > static_cast<uint32_t>(kStageBytes)) return false;
    if (down_map(L->sdown.fmt, L->I).total > static_cast<uint32_t>(kStageBytes)) return false;
  }
  return true;
}

}  // namespace moeq

using namespace moeq;

extern "C" int moe_ffn_decode(const moeq_layer* L, const uint16_t* x, float* y, void* ws,
                              size_t ws_bytes, int32_t* dev_status, const moeq_debug* dbg,
                              moeq_stream stream) {
  int rc = validate_layer(L);
  if (rc) return rc;
  if (!x || !y) return MOEQ_ERR_ARG;
  if (!aligned16(x) || !aligned16(y)) return MOEQ_ERR_ALIGN;
  if (!decode_supported(L)) return MOEQ_ERR_SHAPE;
  const DecodeWs wl = decode_ws_layout(L->H, L->I, L->E, L->k, L->has_shared);
  if (!ws || ws_bytes < wl.total || !aligned16(ws)) return MOEQ_ERR_WORKSPACE;

  DecodeArgs a{};
  a.H = L->H; a.I = L->I; a.E = L->E; a.k = L->k;
  a.has_shared = L->has_shared ? 1 : 0;
  a.nslots = wl.nslots;
  a.x = x;
  a.router = L->router;
  a.gate = to_dmat(L->gate); a.up = to_dmat(L->up); a.down = to_dmat(L->down);
  if (a.has_shared) {
    a.sgate = to_dmat(L->sgate); a.sup = to_dmat(L->sup); a.sdown = to_dmat(L->sdown);
  }
  a.signs_x = L->h32_signs_x;
  a.signs_h = L->h32_signs_h;
  a.y = y;
  uint8_t* w = static_cast<uint8_t*>(ws);
  a.ctr = reinterpret_cast<uint32_t*>(w + wl.ctr);
  a.logits = reinterpret_cast<float*>(w + wl.logits);
  a.hbuf = reinterpret_cast<float*>(w + wl.hbuf);
  a.hq = reinterpret_cast<int8_t*>(w + wl.hq);
  a.hd = reinterpret_cast<uint16_t*>(w + wl.hd);
  a.obuf = reinterpret_cast<float*>(w + wl.obuf);
  a.status = dev_status;
  if (dbg) a.dbg = *dbg;
  a.nR = L->E / kRouterRows;
  a.nSG = a.has_shared ? L->I / kGuRows : 0;
  a.nGU = L->k * (L->I / kGuRows);
  a.nSD = a.has_shared ? L->H / kDownRows : 0;
  a.nD = L->k * (L->H / kDownRows);
  a.total = a.nR + a.nSG + a.nGU + a.nSD + a.nD;

  const DeviceInfo& di = device_info();
  const size_t smem = sizeof(DecodeSmem);
  if (smem > di.max_smem_optin) return MOEQ_ERR_CUDA;
  static thread_local int configured_dev = -1;
  if (configured_dev != di.device) {
    if (cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return MOEQ_ERR_CUDA;
    configured_dev = di.device;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(di.sm_count);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, decode_kernel, a));
}
