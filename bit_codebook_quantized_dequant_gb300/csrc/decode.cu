// Batch-1 decode of one codebook-quantized MoE FFN layer in one persistent,
// cooperative, warp-specialized kernel.
//
// Work items are taken from a global queue in dependency order:
//   router rows (4 per item)
//   -> shared-expert gate/up (32 rows per item, as two 16-row fills)
//   -> routing (one item: top-k and softmax weights of the router logits)
//   -> routed gate/up (32 rows per item, slot-major)
//   -> shared-expert down rows (32 per item)
//   -> routed down rows (32 per item, slot-major)
// (item_fills can also place a slot's down rows a fixed number of slots after
// its gate/up rows; measured slower, since a producer that waits for one slot's
// h holds back the fills queued behind it.)
//   -> (after every down item) the combine of y.
// An item only waits on items with a smaller queue index, and every CTA is
// resident (cooperative launch), so every wait ends; each is bounded anyway and
// reports MOEQ_ERR_DEVICE_TIMEOUT into the status word if it runs out.
//
// Per CTA (17 warps):
//   * producer warp: takes items, streams their packed rows (code plane and
//     scale plane, contiguous per row range) from HBM into a 3-stage shared
//     memory ring with bulk asynchronous copies; once the routing record is
//     published it stages the selected experts' codebooks and prefetches their
//     down rows into L2; for a down item it waits until that slot's quantized h
//     is complete and copies it into the stage next to the weights;
//   * two compute groups of 8 warps, on alternate stage fills: expand codes in
//     registers (byte permutes), take int8 dot products per 32-block (dp4a),
//     apply the block scales in fp32, and release the stage as soon as it is
//     read. They also do all of the kernel's control work, because they own the
//     issue slots (a separate control warp, sharing a scheduler with busy
//     compute warps, ran an order of magnitude slower): the two halves of a
//     gate/up item meet through shared memory and the second group rotates
//     (H32) and quantizes (Q8) the 32-block of h; results are published with
//     release reductions; the routing item is a rank-based top-k over 256
//     threads.
// After its last item every CTA with a share of y waits for all down items and
// combines its rows in slot order: y = sum_s p_s o_s (+ o_shared).
//
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
constexpr int kGroups = 2;  // compute groups on alternate stage fills
constexpr int kGroupWarps = kComputeWarps / kGroups;
constexpr int kGroupThreads = kGroupWarps * 32;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kProducerWarp = kComputeWarps;
constexpr int kThreads = kComputeThreads + 32;
constexpr int kStages = 3;
constexpr int kStageBytes = 68 * 1024;
constexpr int kRouterRows = 4;
constexpr int kGuRows = 16;  // rows per gate/up fill; an item is two fills (one 32-block of h)
constexpr int kDownRows = 32;
constexpr int kMaxH = 4096;
constexpr int kMaxE = 512;
constexpr int kBarCompute = 1;  // named barrier of all compute warps
constexpr int kBarGroup = 2;    // named barriers 2, 3: one per compute group
constexpr int kDownLag = kMaxK;  // slots between a slot's gate/up items and its down items

enum UnitKind { U_ROUTER = 0, U_SGU, U_GU, U_SDOWN, U_DOWN, U_ROUTE, U_END };

// One stage fill: kind, slot (0..k-1 routed, k shared), row chunk of its size.
struct Unit {
  int kind, slot, chunk;
};

__device__ __forceinline__ int pack_unit(const Unit& u) { return (u.kind << 28) | (u.slot << 20) | u.chunk; }
__device__ __forceinline__ Unit unpack_unit(int v) {
  if (v < 0) return Unit{U_END, 0, 0};
  return Unit{(v >> 28) & 15, (v >> 20) & 255, v & 0xfffff};
}

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
  int8_t* hq;
  uint8_t* hd;  // per slot, hd_stride bytes of fp16
  int hd_stride;
  float* obuf;
  int32_t* status;
  moeq_debug dbg;
  int nR, nSG, nSD, nGU, nD, items;  // item counts per kind (plus one routing item)
  int route_base, n_ctr;             // counter word offsets (moeq_layout.h)
};

struct alignas(128) DecodeSmem {
  uint8_t stage[kStages][kStageBytes];
  uint16_t xb[kMaxH];
  int8_t xq[kMaxH];
  float xd[kMaxH / 32];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int unit[kStages];
  uint64_t rkey[kGroupWarps * kMaxK];  // routing item: per-warp candidate keys
  uint32_t stage_cb[kStages][8];       // codebook records of the fill in each stage
  float rwarp[kGroupWarps];         // routing item: per-warp softmax partial sums
  float hs_first[kGroups][kGuRows];   // h of a first-half gate/up fill, by group
  float hs_second[kGroups][kGuRows];  // h of a second-half gate/up fill, by group
  volatile int hs_seq[kGroups];       // fill index of the first half in hs_first[g]
  volatile int hs_ack[kGroups];       // fill index of the first half last consumed from it
  int idx[kMaxK];
  float p[kMaxK];
  int have_route;
  int last_cta;
  int issued;             // stage fills issued by the producer
  int consumed[kGroups];  // last stage fill waited for by each compute group
};

// Item -> its first fill and number of fills.
__device__ __forceinline__ int item_fills(const DecodeArgs& a, int i, Unit& first) {
  if (i < 0 || i >= a.items) return 0;
  if (i < a.nR) { first = Unit{U_ROUTER, 0, i}; return 1; }
  i -= a.nR;
  if (i < a.nSG) { first = Unit{U_SGU, a.k, 2 * i}; return 2; }
  i -= a.nSG;
  if (i == 0) { first = Unit{U_ROUTE, 0, 0}; return 1; }
  i -= 1;
  // routed work, with the down rows of slot s placed after the gate/up rows of
  // slot s + kDownLag so that a slot's h is complete before its down items come:
  //   GU(0) .. GU(lag-1), then for s >= lag: GU(s) D(s-lag), then SD, D(k-lag) ..
  const int pairs = a.I / (2 * kGuRows);
  const int per = a.H / kDownRows;
  const int lag = a.k < kDownLag ? a.k : kDownLag;
  if (i < lag * pairs) { first = Unit{U_GU, i / pairs, 2 * (i % pairs)}; return 2; }
  i -= lag * pairs;
  const int round = pairs + per;
  if (i < (a.k - lag) * round) {
    const int s = lag + i / round, j = i % round;
    if (j < pairs) { first = Unit{U_GU, s, 2 * j}; return 2; }
    first = Unit{U_DOWN, s - lag, j - pairs};
    return 1;
  }
  i -= (a.k - lag) * round;
  if (i < a.nSD) { first = Unit{U_SDOWN, a.k, i}; return 1; }
  i -= a.nSD;
  first = Unit{U_DOWN, a.k - lag + i / per, i % per};
  return 1;
}

// Byte offsets inside a stage. Gate/up: [codes G][scales G][codes U][scales U].
// Down: [codes][scales][hq of the slot][hd of the slot].
struct StageMap {
  uint32_t ca, sa, cb, sb, total;
};

__host__ __device__ __forceinline__ uint32_t al16(uint32_t x) { return (x + 15u) & ~15u; }

__host__ __device__ __forceinline__ uint32_t code_pitch(int fmt, int K) {
  return static_cast<uint32_t>(K / 32) * (fmt == 2 ? 8 : fmt == 3 ? 12 : 16);
}
__host__ __device__ __forceinline__ uint32_t scale_pitch(int fmt, int K) {
  return static_cast<uint32_t>(K / 32) * (fmt == 4 ? 1 : 2);
}

__host__ __device__ __forceinline__ StageMap gu_map(int fmt, int K) {
  const uint32_t c = kGuRows * code_pitch(fmt, K);
  const uint32_t s = al16(kGuRows * scale_pitch(fmt, K));
  return StageMap{0, c, c + s, c + s + c, 2 * (c + s)};
}

__host__ __device__ __forceinline__ StageMap down_map(int fmt, int K) {
  const uint32_t c = kDownRows * code_pitch(fmt, K);
  const uint32_t s = al16(kDownRows * scale_pitch(fmt, K));
  const uint32_t hq = static_cast<uint32_t>(K);
  const uint32_t hd = al16(2 * static_cast<uint32_t>(K / 32));
  return StageMap{0, c, c + s, c + s + hq, c + s + hq + hd};
}

__device__ __forceinline__ const DMat& gu_mat(const DecodeArgs& a, bool shared, bool up) {
  return shared ? (up ? a.sup : a.sgate) : (up ? a.up : a.gate);
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Appends one timeline event of a role of this CTA (debug only).
__device__ __forceinline__ void trace_ev(const DecodeArgs& a, int role, int& n, uint32_t ev, int unit) {
  if (a.dbg.trace && n < a.dbg.trace_cap) {
    uint64_t* p = a.dbg.trace + 2 * ((static_cast<size_t>(blockIdx.x) * 4 + role) * a.dbg.trace_cap + n);
    p[0] = global_ns();
    p[1] = (static_cast<uint64_t>(ev) << 32) | static_cast<uint32_t>(unit);
  }
  ++n;
}

// Bounded spin on a shared-memory word until it equals want.
__device__ __forceinline__ bool smem_wait_eq(const volatile int* w, int want) {
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (*w == want) return true;
    __nanosleep(i < 8 ? 20 : 100);
  }
  return false;
}

// ------------------------------------------------------------------ routing
// Waits for this CTA's copy of the routing record and loads it (one warp).
__device__ void fetch_route(const DecodeArgs& a, DecodeSmem& sm, int lane) {
  const uint32_t* rec = a.ctr + a.route_base + kCtrLine * (blockIdx.x % kRouteCopies);
  if (lane == 0 && !spin_until_geq(rec + kRouteFlag, 1u)) set_status(a.status, MOEQ_ERR_DEVICE_TIMEOUT);
  __syncwarp();
  if (lane < a.k) {
    sm.idx[lane] = static_cast<int>(__ldcg(rec + lane));
    sm.p[lane] = __uint_as_float(__ldcg(rec + 8 + lane));
  }
  __syncwarp();
}

// The routing item, run by one compute group (256 threads, named barrier bar):
// every warp selects the top k of its logits, one warp selects the top k of
// those candidates (key order: larger value, then lower index, NaN last), the
// softmax weights are taken over all E, and the routing record goes to
// kRouteCopies lines, each published by its own release store.
__device__ void route_item(const DecodeArgs& a, DecodeSmem& sm, int bar, int t) {
  constexpr int NPL = kMaxE / kGroupThreads;  // logits per thread
  const int warp = t >> 5, lane = t & 31;
  if (t == 0 && !spin_until_geq(&a.ctr[kCtrRouter], static_cast<uint32_t>(a.nR)))
    set_status(a.status, MOEQ_ERR_DEVICE_TIMEOUT);
  named_bar(bar, kGroupThreads);
  float l[NPL];
  uint64_t key[NPL];
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    const int e = warp * 32 * NPL + 32 * j + lane;  // a warp owns a contiguous range
    l[j] = e < a.E ? __ldcg(&a.logits[e]) : 0.0f;
    key[j] = e < a.E ? ranks_key(l[j], e) : 0ull;
  }
  const uint64_t cand = warp_select_keys<NPL>(key, a.k, lane);
  if (lane < a.k) sm.rkey[warp * kMaxK + lane] = cand;
  named_bar(bar, kGroupThreads);
  if (warp == 0) {
    uint64_t k2[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int c = lane + 32 * j;  // candidates: kGroupWarps x kMaxK = 64
      k2[j] = (c % kMaxK) < a.k ? sm.rkey[c] : 0ull;
    }
    const uint64_t top = warp_select_keys<2>(k2, a.k, lane);
    if (lane < a.k) {
      sm.idx[lane] = key_index(top);
      sm.p[lane] = key_value(top);  // the logit for now
    }
  }
  named_bar(bar, kGroupThreads);
  const float m = sm.p[0];
  float z = 0.0f;
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    const int e = warp * 32 * NPL + 32 * j + lane;
    if (e < a.E && !isnan(l[j])) z += expf(l[j] - m);
  }
  z = warp_sum_canonical(z);
  if (lane == 0) sm.rwarp[warp] = z;
  named_bar(bar, kGroupThreads);
  if (t < a.k) {
    float zt = 0.0f;
    for (int w = 0; w < kGroupWarps; ++w) zt += sm.rwarp[w];
    const float ps = __fdiv_rn(expf(sm.p[t] - m), zt);
    if (a.dbg.idx) a.dbg.idx[t] = sm.idx[t];
    if (a.dbg.p) a.dbg.p[t] = ps;
    sm.p[t] = ps;  // each thread reads and writes only its own entry here
  }
  named_bar(bar, kGroupThreads);
  if (t < kRouteCopies) {
    uint32_t* rec = a.ctr + a.route_base + kCtrLine * t;
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      w[i] = i < a.k ? static_cast<uint32_t>(sm.idx[i]) : 0u;
      w[8 + i] = i < a.k ? __float_as_uint(sm.p[i]) : 0u;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
      reinterpret_cast<uint4*>(rec)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    st_release(rec + kRouteFlag, 1u);
  }
}

// ------------------------------------------------------------------ producer side
// Source ranges of the down rows of (slot, chunk).
__device__ __forceinline__ void down_src(const DecodeArgs& a, const DecodeSmem& sm, int slot,
                                         int chunk, const uint8_t*& c, uint32_t& cbytes,
                                         const uint8_t*& s, uint32_t& sbytes) {
  const bool shared = slot == a.k;
  const DMat& D = shared ? a.sdown : a.down;
  const int e = shared ? 0 : sm.idx[slot];
  const size_t pc = code_pitch(D.fmt, a.I), ps = scale_pitch(D.fmt, a.I);
  const size_t r0 = static_cast<size_t>(chunk) * kDownRows;
  c = D.codes + e * D.stride_codes + r0 * pc;
  s = D.scales + e * D.stride_scales + r0 * ps;
  cbytes = static_cast<uint32_t>(kDownRows * pc);
  sbytes = static_cast<uint32_t>(kDownRows * ps);
}

// L2 prefetch of this CTA's share of the down rows of slots [slot_lo, slot_hi).
__device__ void prefetch_down(const DecodeArgs& a, const DecodeSmem& sm, int slot_lo, int slot_hi) {
  const int per = a.H / kDownRows;
  for (int j = blockIdx.x; j < (slot_hi - slot_lo) * per; j += gridDim.x) {
    const uint8_t *c, *s;
    uint32_t cb, sb;
    down_src(a, sm, slot_lo + j / per, j % per, c, cb, s, sb);
    bulk_prefetch_l2(c, cb);
    bulk_prefetch_l2(s, sb);
  }
}

// Issues the copies of fill un into stage s (lane 0 of the producer warp).
__device__ void issue_unit(const DecodeArgs& a, DecodeSmem& sm, int s, const Unit& un) {
  uint8_t* st = sm.stage[s];
  uint64_t* bar = &sm.full[s];
  if (un.kind == U_ROUTE) {
    mbar_arrive(bar);  // no data
    return;
  }
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
    const size_t pc = code_pitch(G.fmt, a.H), ps = scale_pitch(G.fmt, a.H);
    const StageMap mp = gu_map(G.fmt, a.H);
    const size_t r0 = static_cast<size_t>(un.chunk) * kGuRows;
    const uint32_t cbytes = static_cast<uint32_t>(kGuRows * pc);
    const uint32_t sbytes = static_cast<uint32_t>(kGuRows * ps);
    mbar_arrive_expect_tx(bar, 2 * (cbytes + sbytes) + 32);
    bulk_g2s(st + mp.ca, G.codes + e * G.stride_codes + r0 * pc, cbytes, bar);
    bulk_g2s(st + mp.sa, G.scales + e * G.stride_scales + r0 * ps, sbytes, bar);
    bulk_g2s(st + mp.cb, U.codes + e * U.stride_codes + r0 * pc, cbytes, bar);
    bulk_g2s(st + mp.sb, U.scales + e * U.stride_scales + r0 * ps, sbytes, bar);
    bulk_g2s(sm.stage_cb[s], G.cb + static_cast<size_t>(e) * G.cb_stride, 16, bar);
    bulk_g2s(sm.stage_cb[s] + 4, U.cb + static_cast<size_t>(e) * U.cb_stride, 16, bar);
    return;
  }
  // down fill: weights now, this slot's quantized h once it is complete
  const DMat& D = un.kind == U_SDOWN ? a.sdown : a.down;
  const StageMap mp = down_map(D.fmt, a.I);
  const uint8_t *c, *sc;
  uint32_t cbytes, sbytes;
  down_src(a, sm, un.slot, un.chunk, c, cbytes, sc, sbytes);
  const uint32_t hqb = static_cast<uint32_t>(a.I), hdb = static_cast<uint32_t>(a.hd_stride);
  mbar_arrive_expect_tx(bar, cbytes + sbytes + hqb + hdb + 16);
  bulk_g2s(st + mp.ca, c, cbytes, bar);
  bulk_g2s(st + mp.sa, sc, sbytes, bar);
  const int e = un.kind == U_SDOWN ? 0 : sm.idx[un.slot];
  bulk_g2s(sm.stage_cb[s], D.cb + static_cast<size_t>(e) * D.cb_stride, 16, bar);
  if (!spin_until_geq(&a.ctr[kCtrHqDone + kCtrLine * un.slot], static_cast<uint32_t>(a.I / 32)))
    set_status(a.status, MOEQ_ERR_DEVICE_TIMEOUT);
  asm volatile("fence.proxy.async.global;" ::: "memory");
  bulk_g2s(st + mp.cb, a.hq + static_cast<size_t>(un.slot) * a.I, hqb, bar);
  bulk_g2s(st + mp.sb, a.hd + static_cast<size_t>(un.slot) * a.hd_stride, hdb, bar);
}

// ------------------------------------------------------------------ compute side
__device__ __forceinline__ void load_q(const int8_t* p, int* q) {
  const int4 q0 = *reinterpret_cast<const int4*>(p);
  const int4 q1 = *reinterpret_cast<const int4*>(p + 16);
  q[0] = q0.x; q[1] = q0.y; q[2] = q0.z; q[3] = q0.w;
  q[4] = q1.x; q[5] = q1.y; q[6] = q1.z; q[7] = q1.w;
}

// Rows r0 and r1 of the gate and up tiles in the stage against the quantized x
// in shared memory: g[0], u[0] for r0 and g[1], u[1] for r1.
template <int FMT, bool DBG>
__device__ void gu_rows(const DecodeArgs& a, const DecodeSmem& sm, const uint8_t* st,
                        const uint32_t* cbg, const uint32_t* cbu, int r0, int r1, int row_base,
                        int slot, int lane, float* g, float* u) {
  constexpr int BC = block_bytes<FMT>();
  constexpr int SB = FMT == 4 ? 1 : 2;
  const StageMap mp = gu_map(FMT, a.H);
  const int nb = a.H / 32;
  const uint8_t* gc0 = st + mp.ca + r0 * nb * BC;
  const uint8_t* gc1 = st + mp.ca + r1 * nb * BC;
  const uint8_t* uc0 = st + mp.cb + r0 * nb * BC;
  const uint8_t* uc1 = st + mp.cb + r1 * nb * BC;
  const uint8_t* gs0 = st + mp.sa + r0 * nb * SB;
  const uint8_t* gs1 = st + mp.sa + r1 * nb * SB;
  const uint8_t* us0 = st + mp.sb + r0 * nb * SB;
  const uint8_t* us1 = st + mp.sb + r1 * nb * SB;
  float ag0 = 0.0f, au0 = 0.0f, ag1 = 0.0f, au1 = 0.0f;
#pragma unroll 1
  for (int b = lane; b < nb; b += 32) {
    {
      int q[8];
      load_q(sm.xq + 32 * b, q);
      const float xd = sm.xd[b];
      const int sg0 = block_dot<FMT>(gc0 + b * BC, cbg, q);
      const int su0 = block_dot<FMT>(uc0 + b * BC, cbu, q);
      const int sg1 = block_dot<FMT>(gc1 + b * BC, cbg, q);
      const int su1 = block_dot<FMT>(uc1 + b * BC, cbu, q);
      ag0 = fmaf(block_scale<FMT>(gs0, b) * xd, static_cast<float>(sg0), ag0);
      au0 = fmaf(block_scale<FMT>(us0, b) * xd, static_cast<float>(su0), au0);
      ag1 = fmaf(block_scale<FMT>(gs1, b) * xd, static_cast<float>(sg1), ag1);
      au1 = fmaf(block_scale<FMT>(us1, b) * xd, static_cast<float>(su1), au1);
      if (DBG && a.dbg.S_gate) {
        a.dbg.S_gate[(static_cast<size_t>(slot) * a.I + row_base + r0) * nb + b] = sg0;
        a.dbg.S_gate[(static_cast<size_t>(slot) * a.I + row_base + r1) * nb + b] = sg1;
      }
      if (DBG && a.dbg.S_up) {
        a.dbg.S_up[(static_cast<size_t>(slot) * a.I + row_base + r0) * nb + b] = su0;
        a.dbg.S_up[(static_cast<size_t>(slot) * a.I + row_base + r1) * nb + b] = su1;
      }
    }
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) {
    ag0 += __shfl_xor_sync(0xffffffffu, ag0, d);
    au0 += __shfl_xor_sync(0xffffffffu, au0, d);
    ag1 += __shfl_xor_sync(0xffffffffu, ag1, d);
    au1 += __shfl_xor_sync(0xffffffffu, au1, d);
  }
  g[0] = ag0; u[0] = au0; g[1] = ag1; u[1] = au1;
}

// Rows wg, wg + 8, wg + 16, wg + 24 of the down tile in the stage against the
// slot's quantized h, which the producer placed in the same stage.
template <int FMT, bool DBG>
__device__ void down_rows(const DecodeArgs& a, const uint8_t* st, const uint32_t* cb, int wg,
                          int lane, int chunk, int slot, float* o) {
  constexpr int BC = block_bytes<FMT>();
  constexpr int SB = FMT == 4 ? 1 : 2;
  constexpr int R = kDownRows / kGroupWarps;
  const StageMap mp = down_map(FMT, a.I);
  const int nb = a.I / 32;
  const int8_t* hq = reinterpret_cast<const int8_t*>(st + mp.cb);
  const uint16_t* hd = reinterpret_cast<const uint16_t*>(st + mp.sb);
  float acc[R];
#pragma unroll
  for (int j = 0; j < R; ++j) acc[j] = 0.0f;
#pragma unroll 1
  for (int b = lane; b < nb; b += 32) {
    {
      int q[8];
      load_q(hq + 32 * b, q);
      const float hdf = f16_bits_to_f32(hd[b]);
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int r = wg + kGroupWarps * j;
        const int d = block_dot<FMT>(st + mp.ca + r * nb * BC + b * BC, cb, q);
        acc[j] = fmaf(block_scale<FMT>(st + mp.sa + r * nb * SB, b) * hdf, static_cast<float>(d), acc[j]);
        if (DBG && a.dbg.S_down)
          a.dbg.S_down[(static_cast<size_t>(slot) * a.H + chunk * kDownRows + r) * nb + b] = d;
      }
    }
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) {
#pragma unroll
    for (int j = 0; j < R; ++j) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], d);
  }
#pragma unroll
  for (int j = 0; j < R; ++j) o[j] = acc[j];
}

__device__ float router_row(const DecodeArgs& a, const DecodeSmem& sm, const uint8_t* st, int r,
                            int lane) {
  const uint8_t* wrow = st + static_cast<size_t>(r) * a.H * 2;
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
  return warp_sum_canonical(acc);
}

// Rotates (H32) and quantizes (Q8) one 32-block of h of slot by one warp;
// lane i holds element i. Publishes the block.
__device__ void quantize_h_block(const DecodeArgs& a, float v, int slot, int blk, int lane) {
  if (a.signs_h) v = h32_warp(v, __ldg(&a.signs_h[blk]), lane);
  uint16_t db;
  const int8_t q = q8_warp(v, db);
  const size_t base = static_cast<size_t>(slot) * a.I + 32 * blk;
  a.hq[base + lane] = q;
  if (lane == 0) reinterpret_cast<uint16_t*>(a.hd + static_cast<size_t>(slot) * a.hd_stride)[blk] = db;
  if (a.dbg.hq) a.dbg.hq[base + lane] = q;
  if (a.dbg.hd && lane == 0) a.dbg.hd[static_cast<size_t>(slot) * (a.I / 32) + blk] = db;
  __syncwarp();
  if (lane == 0) red_add_release(&a.ctr[kCtrHqDone + kCtrLine * slot], 1u);
}

// Computes fill n (unit un) from stage s with the 8 warps of compute group grp
// (wg = warp in group), releasing the stage as soon as it is read, then does
// the fill's share of publishing. first_prev: this group's previous first-half
// gate/up fill (-1 if none).
template <bool DBG>
__device__ void compute_unit(const DecodeArgs& a, DecodeSmem& sm, int s, int n, const Unit& un,
                             int grp, int wg, int lane, int& first_prev) {
  const uint8_t* st = sm.stage[s];
  const int bar = kBarGroup + grp;
  const int t = wg * 32 + lane;
  if (un.kind == U_ROUTE) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[s]);
    route_item(a, sm, bar, t);
    return;
  }
  if (un.kind == U_ROUTER) {
    float l = 0.0f;
    if (wg < kRouterRows) l = router_row(a, sm, st, wg, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[s]);
    if (wg < kRouterRows && lane == 0) {
      const int ex = un.chunk * kRouterRows + wg;
      a.logits[ex] = l;
      if (DBG && a.dbg.logits) a.dbg.logits[ex] = l;
    }
    named_bar(bar, kGroupThreads);
    if (t == 0) red_add_release(&a.ctr[kCtrRouter], 1u);
    return;
  }
  if (un.kind == U_SGU || un.kind == U_GU) {
    const int fmt = un.kind == U_SGU ? a.sgate.fmt : a.gate.fmt;
    uint32_t cbg[4], cbu[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      cbg[i] = sm.stage_cb[s][i];
      cbu[i] = sm.stage_cb[s][4 + i];
    }
    const int base = un.chunk * kGuRows;
    float g[2], u[2];
    if (fmt == 2) gu_rows<2, DBG>(a, sm, st, cbg, cbu, wg, wg + kGroupWarps, base, un.slot, lane, g, u);
    else if (fmt == 3) gu_rows<3, DBG>(a, sm, st, cbg, cbu, wg, wg + kGroupWarps, base, un.slot, lane, g, u);
    else gu_rows<4, DBG>(a, sm, st, cbg, cbu, wg, wg + kGroupWarps, base, un.slot, lane, g, u);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[s]);
    const bool first_half = (un.chunk & 1) == 0;
    if (first_half && first_prev >= 0) {
      // the other group must have consumed this group's previous first half
      if (t == 0 && !smem_wait_eq(&sm.hs_ack[grp], first_prev)) set_status(a.status, MOEQ_ERR_DEVICE_TIMEOUT);
      named_bar(bar, kGroupThreads);
    }
    float* hs = first_half ? sm.hs_first[grp] : sm.hs_second[grp];
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r = wg + kGroupWarps * j;
        const float h = g[j] * u[j] / (1.0f + expf(-g[j]));
        hs[r] = h;
        if (DBG && a.dbg.h) a.dbg.h[static_cast<size_t>(un.slot) * a.I + base + r] = h;
      }
    }
    named_bar(bar, kGroupThreads);
    if (first_half) {
      if (t == 0) {
        __threadfence_block();
        sm.hs_seq[grp] = n;
      }
      first_prev = n;
      return;
    }
    // second half: the first half was fill n - 1, computed by the other group
    if (wg == 0) {
      const int other = grp ^ 1;
      if (lane == 0 && !smem_wait_eq(&sm.hs_seq[other], n - 1)) set_status(a.status, MOEQ_ERR_DEVICE_TIMEOUT);
      __syncwarp();
      __threadfence_block();
      const float v = lane < kGuRows ? sm.hs_first[other][lane] : sm.hs_second[grp][lane - kGuRows];
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        sm.hs_ack[other] = n - 1;
      }
      quantize_h_block(a, v, un.slot, un.chunk / 2, lane);
    }
    return;
  }
  const int fmt = un.kind == U_SDOWN ? a.sdown.fmt : a.down.fmt;
  uint32_t cb[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) cb[i] = sm.stage_cb[s][i];
  constexpr int R = kDownRows / kGroupWarps;
  float o[R];
  if (fmt == 2) down_rows<2, DBG>(a, st, cb, wg, lane, un.chunk, un.slot, o);
  else if (fmt == 3) down_rows<3, DBG>(a, st, cb, wg, lane, un.chunk, un.slot, o);
  else down_rows<4, DBG>(a, st, cb, wg, lane, un.chunk, un.slot, o);
  __syncwarp();
  if (lane == 0) {
    mbar_arrive(&sm.empty[s]);
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const size_t at = static_cast<size_t>(un.slot) * a.H + un.chunk * kDownRows + wg + kGroupWarps * j;
      a.obuf[at] = o[j];
      if (DBG && a.dbg.o) a.dbg.o[at] = o[j];
    }
  }
  named_bar(bar, kGroupThreads);
  if (t == 0) red_add_release(&a.ctr[kCtrDownDone], 1u);
}

template <bool DBG>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  DecodeSmem& sm = *reinterpret_cast<DecodeSmem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kGroupWarps);
    }
    sm.issued = 0;
    sm.have_route = 0;
    for (int g = 0; g < kGroups; ++g) {
      sm.consumed[g] = g - kGroups;
      sm.hs_seq[g] = -1;
      sm.hs_ack[g] = -1;
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- producer warp
    if (lane == 0 && a.has_shared) prefetch_down(a, sm, a.k, a.k + 1);
    __syncwarp();
    int it = 0, ntr = 0;
    bool aborted = false;
    for (;;) {
      int item = 0;
      if (lane == 0) {
        item = static_cast<int>(atom_add_relaxed(&a.ctr[kCtrQueue], 1u));
        trace_ev(a, 1, ntr, MOEQ_TRACE_TAKE, item);
      }
      item = __shfl_sync(0xffffffffu, item, 0);
      Unit first{U_END, 0, 0};
      const int nf = item_fills(a, item, first);
      if (nf > 0 && (first.kind == U_GU || first.kind == U_DOWN) && !sm.have_route) {
        fetch_route(a, sm, lane);
        if (lane == 0) {
          sm.have_route = 1;
          trace_ev(a, 1, ntr, MOEQ_TRACE_TOPK, item);
        }
        __syncwarp();
      }
      // nf == 0: one end marker per compute group, on consecutive fills
      const int fills = nf > 0 ? nf : kGroups;
      for (int f = 0; f < fills; ++f, ++it) {
        const int s = it % kStages;
        if (it >= kStages) {
          bool ok = true;
          if (lane == 0) ok = mbar_wait(&sm.empty[s], ((it / kStages) - 1) & 1);
          if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
            set_status(a.status, MOEQ_ERR_DEVICE_TIMEOUT);
            aborted = true;
            break;
          }
        }
        if (lane == 0) {
          if (nf == 0) {
            sm.unit[s] = -1;
            mbar_arrive(&sm.full[s]);
          } else {
            Unit un = first;
            un.chunk += f;
            sm.unit[s] = pack_unit(un);
            issue_unit(a, sm, s, un);
            trace_ev(a, 1, ntr, MOEQ_TRACE_ISSUED, item);
          }
        }
        __syncwarp();
      }
      if (aborted || nf == 0) break;
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
    const int grp = warp / kGroupWarps, wg = warp % kGroupWarps;
    const int role = grp == 0 ? 0 : 3;
    int ntr = 0, first_prev = -1;
    if (wg == 0 && lane == 0) trace_ev(a, role, ntr, MOEQ_TRACE_START, 0);

    for (int it = grp;; it += kGroups) {
      const int s = it % kStages;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&sm.full[s], (it / kStages) & 1);
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
        set_status(a.status, MOEQ_ERR_DEVICE_TIMEOUT);
        break;
      }
      const int u = sm.unit[s];
      if (wg == 0 && lane == 0) {
        sm.consumed[grp] = it;
        trace_ev(a, role, ntr, MOEQ_TRACE_READY, u);
      }
      const Unit un = unpack_unit(u);
      if (un.kind == U_END) break;
      compute_unit<DBG>(a, sm, s, it, un, grp, wg, lane, first_prev);
      if (wg == 0 && lane == 0) trace_ev(a, role, ntr, MOEQ_TRACE_DONE, u);
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (warp == kProducerWarp && lane == 0) {
    // fills issued but never waited for (only after a timeout): let them land
    for (int g = 0; g < kGroups; ++g)
      for (int j = sm.consumed[g] + kGroups; j < sm.issued; j += kGroups)
        if (!mbar_wait(&sm.full[j % kStages], (j / kStages) & 1)) break;
  }
  // combine y in slot order once every down item is done; 32 rows per warp
  const int nchunks = a.H / kDownRows;
  constexpr int kWarps = kThreads / 32;
  if (static_cast<int>(blockIdx.x) * kWarps < nchunks) {
    if (warp == 0) {
      if (lane == 0 && !spin_until_geq(&a.ctr[kCtrDownDone], static_cast<uint32_t>(a.nSD + a.nD)))
        set_status(a.status, MOEQ_ERR_DEVICE_TIMEOUT);
      __syncwarp();
      if (!sm.have_route) fetch_route(a, sm, lane);
    }
    __syncthreads();
    const int c = static_cast<int>(blockIdx.x) * kWarps + warp;
    if (c < nchunks) {
      const int row = c * kDownRows + lane;
      float acc = 0.0f;
      for (int s = 0; s < a.k; ++s)
        acc = fmaf(sm.p[s], __ldcg(&a.obuf[static_cast<size_t>(s) * a.H + row]), acc);
      if (a.has_shared) acc += __ldcg(&a.obuf[static_cast<size_t>(a.k) * a.H + row]);
      a.y[row] = acc;
    }
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const uint32_t old = atomicAdd(&a.ctr[kCtrDone], 1u);
    sm.last_cta = old == gridDim.x - 1;
    if (sm.last_cta) __threadfence();
  }
  __syncthreads();
  if (sm.last_cta) {
    for (int i = tid; i < a.n_ctr; i += kThreads)
      if (i != kCtrDone) a.ctr[i] = 0u;
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      a.ctr[kCtrDone] = 0u;
    }
  }
}

}  // namespace

bool decode_supported(const moeq_layer* L) {
  if (L->H > kMaxH || L->I > kMaxH || L->E > kMaxE || L->E % kRouterRows || L->k > kMaxK)
    return false;
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
  a.hq = reinterpret_cast<int8_t*>(w + wl.hq);
  a.hd = w + wl.hd;
  a.hd_stride = static_cast<int>(hd_stride(L->I));
  a.obuf = reinterpret_cast<float*>(w + wl.obuf);
  a.status = dev_status;
  if (dbg) a.dbg = *dbg;
  a.nR = L->E / kRouterRows;
  a.nSG = a.has_shared ? L->I / (2 * kGuRows) : 0;
  a.nSD = a.has_shared ? L->H / kDownRows : 0;
  a.nGU = L->k * (L->I / (2 * kGuRows));
  a.nD = L->k * (L->H / kDownRows);
  a.items = a.nR + a.nSG + 1 + a.nSD + a.nGU + a.nD;
  a.route_base = route_base(a.nslots);
  a.n_ctr = static_cast<int>(wl.n_ctr);

  const DeviceInfo& di = device_info();
  const size_t smem = sizeof(DecodeSmem);
  if (smem > di.max_smem_optin) return MOEQ_ERR_CUDA;
  // the debug instantiation carries the stores of intermediates and the timeline
  const bool want_dbg = dbg != nullptr;
  void (*kern)(const DecodeArgs) = want_dbg ? decode_kernel<true> : decode_kernel<false>;
  static thread_local int configured_dev = -1;
  if (configured_dev != di.device) {
    if (cudaFuncSetAttribute(decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess ||
        cudaFuncSetAttribute(decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, a));
}
