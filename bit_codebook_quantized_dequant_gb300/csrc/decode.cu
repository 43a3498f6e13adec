// Batch-1 decode (one column) and q=4 verification (four columns) of one
// codebook-quantized MoE FFN layer, each in one persistent, cooperative,
// warp-specialized kernel, templated on the number of columns.
//
// A "unit" is one expert whose weights are read once per call: for one
// column the k selected experts; for four columns the distinct experts of the
// union of their selections (in order of first appearance, column-major), each
// applied to every column that selected it; then the shared expert.
//
// Work items are taken from a global queue in dependency order:
//   router rows (4 per item; every column's logits from one read of a row)
//   -> shared-expert gate/up (32 rows per item, as two 16-row fills)
//   -> dense projection rows (32 per item; four columns only)
//   -> routing (one item: top-k and softmax weights per column, the units)
//   -> routed gate/up (32 rows per item, unit-major)
//   -> shared-expert down rows (32 per item)
//   -> routed down rows (32 per item, unit-major)
//   -> (after every down item) the combine of y.
// (Placing a unit's down rows a few units after its gate/up rows, to start
// down work earlier, measured slower: a producer that waits for one unit's h
// holds back the fills queued behind it.)
// An item only waits on items with a smaller queue index, and every CTA is
// resident (cooperative launch), so every wait ends; each is bounded anyway and
// reports MOEQ_ERR_DEVICE_TIMEOUT into the status word if it runs out.
//
// Per CTA (17 warps):
//   * producer warp: takes items, streams their packed rows (code plane and
//     scale plane, contiguous per row range) and codebook records from HBM
//     into a 3-stage shared memory ring with bulk asynchronous copies; for a
//     down item it waits until that unit's quantized h is complete and copies
//     it into the stage next to the weights;
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
// combines its rows in slot order: y_c = sum_s p_{c,s} o_{c,s} (+ o_shared,c).
//
// Sources: "DeepSeek V4 Flash: 284B model, up to 32 tok/s on AMD Ryzen AI MAX+
// 395", section "ROCmFPX: fitting 284B weights into 128 GB" (read packed blocks
// directly, expand small codebooks in registers, integer dot products, decode
// bound by weight traffic) and section "Decode: up to 32 tok/s" (q=4
// verification that decodes each packed weight once for all four columns);
// "Lucebox x Geometric ...", section "Lucebox Engine integration with
// Geometric" (fused matvec, sync-free MoE decode).
#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>

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
constexpr int kMaxCols = 4;
constexpr int kBarCompute = 1;  // named barrier of all compute warps
constexpr int kBarGroup = 2;    // named barriers 2, 3: one per compute group
static_assert(kMaxCols * kMaxK <= 32, "one lane per (column, slot) in the unit builder");
static_assert(kMaxE / 64 == kGroupWarps, "softmax partial sums: one 64-logit range per group warp");

enum UnitKind { U_ROUTER = 0, U_SGU, U_GU, U_SDOWN, U_DOWN, U_ROUTE, U_DENSE, U_END };

// One stage fill: kind, unit (routed 0..nu-1, shared cols*k), row chunk of its size.
struct Unit {
  int kind, slot, chunk;
};

__device__ __forceinline__ int pack_unit(const Unit& u) { return (u.kind << 28) | (u.slot << 20) | u.chunk; }
__device__ __forceinline__ Unit unpack_unit(int v) {
  if (v < 0) return Unit{U_END, 0, 0};
  return Unit{(v >> 28) & 15, (v >> 20) & 255, v & 0xfffff};
}

// Unit word: expert (bits 0..9), column mask (bits 10..13), and for every
// column c in the mask the slot (rank in that column's top-k, k for the shared
// expert) at bits 16 + 4c.
__device__ __forceinline__ int uw_expert(uint32_t w) { return static_cast<int>(w & 0x3ffu); }
__device__ __forceinline__ uint32_t uw_mask(uint32_t w) { return (w >> 10) & 0xfu; }
__device__ __forceinline__ int uw_slot(uint32_t w, int c) { return static_cast<int>((w >> (16 + 4 * c)) & 0xfu); }

struct DecodeArgs {
  int H, I, E, k, has_shared;
  int su;  // index of the shared unit (cols * k)
  const uint16_t* x;  // [cols][H] bf16
  const uint16_t* router;
  DMat gate, up, down, sgate, sup, sdown, dense;
  const uint32_t* signs_x;
  const uint32_t* signs_h;
  float* y;        // [cols][H]
  float* y_dense;  // [cols][dense rows]
  uint32_t* ctr;
  float* logits;   // [cols][E]
  int8_t* hq;      // vector v = unit * cols + column: I bytes each
  uint8_t* hd;     // vector v: hd_stride bytes of fp16 each
  int hd_stride;
  float* obuf;     // vector v: H fp32 each
  int32_t* status;
  moeq_debug dbg;
  int nR, nSG, nDN, nSD;  // item counts that do not depend on the routing
  int route_idx;          // queue index of the routing item
  int route_base, n_ctr;  // counter word offsets (moeq_layout.h)
  uint32_t spin;          // polls of each wait on another CTA before it gives up
};

template <int COLS>
struct alignas(128) DecodeSmem {
  uint8_t stage[kStages][kStageBytes];
  uint16_t xb[COLS == 1 ? kMaxH : 8];  // bf16 x for the router rows (one column only)
  int8_t xq[COLS][kMaxH];
  float xd[COLS][kMaxH / 32];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int unit[kStages];
  uint64_t rkey[kGroupWarps * kMaxK];  // routing item: per-warp candidate keys
  alignas(16) uint32_t stage_cb[kStages][8];  // codebook records of the fill in each stage (bulk-copy target)
  float rwarp[kMaxCols * kGroupWarps];  // routing item: softmax partial sums per 64 logits
  float hs_first[kGroups][COLS][kGuRows];   // h of a first-half gate/up fill, by group
  float hs_second[kGroups][COLS][kGuRows];  // h of a second-half gate/up fill, by group
  volatile int hs_seq[kGroups];  // fill index of the first half in hs_first[g]
  volatile int hs_ack[kGroups];  // fill index of the first half last consumed from it
  int idx[COLS][kMaxK];
  float p[COLS][kMaxK];
  uint32_t uw[COLS * kMaxK + 1];  // unit words: routed units, then the shared unit
  int uof[COLS][kMaxK];           // unit of (column, slot)
  int nu;                         // routed units
  int have_route;
  int last_cta;
  int issued;             // stage fills issued by the producer
  int consumed[kGroups];  // last stage fill waited for by each compute group
};

// Bulk asynchronous copies land in stage[] and stage_cb[]: both 16-byte aligned.
static_assert(offsetof(DecodeSmem<1>, stage_cb) % 16 == 0 && offsetof(DecodeSmem<4>, stage_cb) % 16 == 0,
              "bulk-copy targets must be 16-byte aligned");
static_assert(offsetof(DecodeSmem<1>, stage) % 128 == 0 && offsetof(DecodeSmem<4>, stage) % 128 == 0,
              "bulk-copy targets must be 16-byte aligned");

// Item -> its first fill and number of fills (nu: routed units, needed only
// past the routing item).
__device__ __forceinline__ int item_fills(const DecodeArgs& a, int nu, int i, Unit& first) {
  if (i < 0) return 0;
  if (i < a.nR) { first = Unit{U_ROUTER, 0, i}; return 1; }
  i -= a.nR;
  if (i < a.nSG) { first = Unit{U_SGU, a.su, 2 * i}; return 2; }
  i -= a.nSG;
  if (i < a.nDN) { first = Unit{U_DENSE, 0, i}; return 1; }
  i -= a.nDN;
  if (i == 0) { first = Unit{U_ROUTE, 0, 0}; return 1; }
  i -= 1;
  const int pairs = a.I / (2 * kGuRows);
  if (i < nu * pairs) { first = Unit{U_GU, i / pairs, 2 * (i % pairs)}; return 2; }
  i -= nu * pairs;
  if (i < a.nSD) { first = Unit{U_SDOWN, a.su, i}; return 1; }
  i -= a.nSD;
  const int per = a.H / kDownRows;
  if (i < nu * per) { first = Unit{U_DOWN, i / per, i % per}; return 1; }
  return 0;
}

// Byte offsets inside a stage. Gate/up: [codes G][scales G][codes U][scales U].
// Down: [codes][scales][hq of the unit's columns][hd of the unit's columns].
// Dense: [codes][scales].
struct StageMap {
  uint32_t ca, sa, cb, sb, total;
};

__host__ __device__ __forceinline__ uint32_t al16(uint32_t x) { return (x + 15u) & ~15u; }

__host__ __device__ __forceinline__ uint32_t code_pitch(int fmt, int K) {
  return static_cast<uint32_t>(K / 32) * (fmt == 2 ? 8 : fmt == 3 || fmt == MOEQ_FP3_PACKED24 ? 12 : 16);
}
__host__ __device__ __forceinline__ uint32_t scale_pitch(int fmt, int K) {
  return static_cast<uint32_t>(K / 32) * (fmt == 4 ? 1 : 2);
}
__host__ __device__ __forceinline__ uint32_t hd_pitch(int K) {
  return al16(2 * static_cast<uint32_t>(K / 32));
}

__host__ __device__ __forceinline__ StageMap gu_map(int fmt, int K) {
  const uint32_t c = kGuRows * code_pitch(fmt, K);
  const uint32_t s = al16(kGuRows * scale_pitch(fmt, K));
  return StageMap{0, c, c + s, c + s + c, 2 * (c + s)};
}

__host__ __device__ __forceinline__ StageMap down_map(int fmt, int K, int cols) {
  const uint32_t c = kDownRows * code_pitch(fmt, K);
  const uint32_t s = al16(kDownRows * scale_pitch(fmt, K));
  const uint32_t hq = static_cast<uint32_t>(cols) * static_cast<uint32_t>(K);
  const uint32_t hd = static_cast<uint32_t>(cols) * hd_pitch(K);
  return StageMap{0, c, c + s, c + s + hq, c + s + hq + hd};
}

__host__ __device__ __forceinline__ StageMap dense_map(int fmt, int K) {
  const uint32_t c = kDownRows * code_pitch(fmt, K);
  const uint32_t s = al16(kDownRows * scale_pitch(fmt, K));
  return StageMap{0, c, 0, 0, c + s};
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

// Debug vector of (column c, slot s): c * (k + shared) + s.
__device__ __forceinline__ int dbg_vec(const DecodeArgs& a, int c, int s) {
  return c * (a.k + a.has_shared) + s;
}

// ------------------------------------------------------------------ routing
// Waits for this CTA's copy of the routing record and loads it (one warp).
template <int COLS>
__device__ void fetch_route(const DecodeArgs& a, DecodeSmem<COLS>& sm, int lane) {
  constexpr int RL = route_lines(COLS);
  const uint32_t* rec = a.ctr + a.route_base + kCtrLine * RL * (blockIdx.x % kRouteCopies);
  if (lane == 0 && !spin_until_geq(rec + kCtrLine * (RL - 1) + kRouteFlag, 1u, a.spin))
    set_status(a.status, MOEQ_ERR_DEVICE_TIMEOUT);
  __syncwarp();
  if constexpr (COLS == 1) {
    if (lane < a.k) {
      const int e = static_cast<int>(__ldcg(rec + lane));
      sm.idx[0][lane] = e;
      sm.p[0][lane] = __uint_as_float(__ldcg(rec + 8 + lane));
      sm.uw[lane] = static_cast<uint32_t>(e) | (1u << 10) | (static_cast<uint32_t>(lane) << 16);
      sm.uof[0][lane] = lane;
    }
    if (lane == 0) sm.nu = a.k;
  } else {
    const int c = lane / kMaxK, j = lane % kMaxK;
    if (c < COLS) {
      sm.idx[c][j] = static_cast<int>(__ldcg(rec + lane));
      sm.p[c][j] = __uint_as_float(__ldcg(rec + kCtrLine + lane));
    }
    const uint32_t w = __ldcg(rec + 2 * kCtrLine + lane);
    const int nu = static_cast<int>(__ldcg(rec + 3 * kCtrLine));
    if (lane < nu) {
      sm.uw[lane] = w;
      for (int cc = 0; cc < COLS; ++cc)
        if ((uw_mask(w) >> cc) & 1u) sm.uof[cc][uw_slot(w, cc)] = lane;
    }
    if (lane == 0) sm.nu = nu;
  }
  __syncwarp();
}

// The routing item, run by one compute group (256 threads, named barrier bar):
// per column, every warp selects the top k of its share of the logits, one warp
// selects the top k of those candidates (key order: larger value, then lower
// index, NaN last), and the softmax weights are taken over all E. With several
// columns the distinct selected experts become the units. The record goes to
// kRouteCopies places, each published by its own release store.
template <int COLS>
__device__ void route_item(const DecodeArgs& a, DecodeSmem<COLS>& sm, int bar, int t) {
  constexpr int WPC = kGroupWarps / COLS;   // warps per column
  constexpr int NPL = kMaxE / (32 * WPC);   // logits per lane
  const int warp = t >> 5, lane = t & 31;
  const int col = warp / WPC, sub = warp % WPC;
  if (t == 0 && !spin_until_geq(&a.ctr[kCtrRouter], static_cast<uint32_t>(a.nR), a.spin))
    set_status(a.status, MOEQ_ERR_DEVICE_TIMEOUT);
  named_bar(bar, kGroupThreads);
  float l[NPL];
  uint64_t key[NPL];
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    const int e = sub * 32 * NPL + 32 * j + lane;  // a warp owns a contiguous range
    l[j] = e < a.E ? __ldcg(&a.logits[col * a.E + e]) : 0.0f;
    key[j] = e < a.E ? ranks_key(l[j], e) : 0ull;
  }
  const uint64_t cand = warp_select_keys<NPL>(key, a.k, lane);
  if (lane < a.k) sm.rkey[warp * kMaxK + lane] = cand;
  named_bar(bar, kGroupThreads);
  if (warp < COLS) {
    uint64_t k2[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int c = lane + 32 * j;  // candidates of the column: WPC x kMaxK <= 64
      k2[j] = (c < WPC * kMaxK && (c % kMaxK) < a.k) ? sm.rkey[warp * WPC * kMaxK + c] : 0ull;
    }
    const uint64_t top = warp_select_keys<2>(k2, a.k, lane);
    if (lane < a.k) {
      sm.idx[warp][lane] = key_index(top);
      sm.p[warp][lane] = key_value(top);  // the logit for now
    }
  }
  named_bar(bar, kGroupThreads);
  // softmax denominator in one fixed order for any column count: partial sums
  // over ranges of 64 logits (two per lane, then the combining rounds), then
  // the 8 range sums in order
  const float m = sm.p[col][0];
  const float mt = t < COLS * a.k ? sm.p[t / a.k][0] : 0.0f;
  constexpr int RPW = NPL / 2;  // ranges per warp
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    float z = 0.0f;
#pragma unroll
    for (int j = 2 * r; j < 2 * r + 2; ++j) {
      const int e = sub * 32 * NPL + 32 * j + lane;
      if (e < a.E && !isnan(l[j])) z += expf(l[j] - m);
    }
    z = warp_sum_canonical(z);
    if (lane == 0) sm.rwarp[warp * RPW + r] = z;
  }
  named_bar(bar, kGroupThreads);
  if (t < COLS * a.k) {
    const int c = t / a.k, j = t % a.k;
    float zt = 0.0f;
    for (int w = 0; w < kGroupWarps; ++w) zt += sm.rwarp[c * kGroupWarps + w];
    const float ps = __fdiv_rn(expf(sm.p[c][j] - mt), zt);
    if (a.dbg.idx) a.dbg.idx[t] = sm.idx[c][j];
    if (a.dbg.p) a.dbg.p[t] = ps;
    sm.p[c][j] = ps;  // each thread reads and writes only its own entry here
  }
  if constexpr (COLS > 1) {
    // units: lane i < COLS*k stands for (column i / k, slot i % k); lanes with
    // equal experts form one unit, numbered by its first lane
    named_bar(bar, kGroupThreads);
    if (warp == 0) {
      const int n = COLS * a.k;
      const int e = lane < n ? sm.idx[lane / a.k][lane % a.k] : 0x400 + lane;
      const uint32_t same = __match_any_sync(0xffffffffu, e);
      const int leader = __ffs(same) - 1;
      const bool first = lane < n && leader == lane;
      const uint32_t firsts = __ballot_sync(0xffffffffu, first);
      if (first) {
        uint32_t w = static_cast<uint32_t>(e);
        for (uint32_t m2 = same; m2; m2 &= m2 - 1) {
          const int b = __ffs(m2) - 1;
          const int c = b / a.k, j = b % a.k;
          w |= (1u << (10 + c)) | (static_cast<uint32_t>(j) << (16 + 4 * c));
        }
        sm.uw[__popc(firsts & ((1u << lane) - 1u))] = w;
      }
      if (lane == 0) sm.nu = __popc(firsts);
    }
  }
  named_bar(bar, kGroupThreads);
  if (t < kRouteCopies) {
    constexpr int RL = route_lines(COLS);
    uint32_t* rec = a.ctr + a.route_base + kCtrLine * RL * t;
    if constexpr (COLS == 1) {
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        w[i] = i < a.k ? static_cast<uint32_t>(sm.idx[0][i]) : 0u;
        w[8 + i] = i < a.k ? __float_as_uint(sm.p[0][i]) : 0u;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
        reinterpret_cast<uint4*>(rec)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
      st_release(rec + kRouteFlag, 1u);
    } else {
      const int nu = sm.nu;
      for (int i = 0; i < 32; i += 4) {
        uint32_t wi[4], wp[4], wu[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int c = (i + q) / kMaxK, j = (i + q) % kMaxK;
          const bool ok = c < COLS && j < a.k;
          wi[q] = ok ? static_cast<uint32_t>(sm.idx[c][j]) : 0u;
          wp[q] = ok ? __float_as_uint(sm.p[c][j]) : 0u;
          wu[q] = i + q < nu ? sm.uw[i + q] : 0u;
        }
        *reinterpret_cast<uint4*>(rec + i) = make_uint4(wi[0], wi[1], wi[2], wi[3]);
        *reinterpret_cast<uint4*>(rec + kCtrLine + i) = make_uint4(wp[0], wp[1], wp[2], wp[3]);
        *reinterpret_cast<uint4*>(rec + 2 * kCtrLine + i) = make_uint4(wu[0], wu[1], wu[2], wu[3]);
      }
      rec[3 * kCtrLine] = static_cast<uint32_t>(nu);
      st_release(rec + 3 * kCtrLine + kRouteFlag, 1u);
    }
  }
}

// ------------------------------------------------------------------ producer side
// Source ranges of the down rows of (unit, chunk).
template <int COLS>
__device__ __forceinline__ void down_src(const DecodeArgs& a, const DecodeSmem<COLS>& sm, int unit,
                                         int chunk, const uint8_t*& c, uint32_t& cbytes,
                                         const uint8_t*& s, uint32_t& sbytes) {
  const bool shared = unit == a.su;
  const DMat& D = shared ? a.sdown : a.down;
  const int e = shared ? 0 : uw_expert(sm.uw[unit]);
  const size_t pc = code_pitch(D.fmt, a.I), ps = scale_pitch(D.fmt, a.I);
  const size_t r0 = static_cast<size_t>(chunk) * kDownRows;
  c = D.codes + e * D.stride_codes + r0 * pc;
  s = D.scales + e * D.stride_scales + r0 * ps;
  cbytes = static_cast<uint32_t>(kDownRows * pc);
  sbytes = static_cast<uint32_t>(kDownRows * ps);
}

// L2 prefetch of this CTA's share of the shared expert's down rows.
template <int COLS>
__device__ void prefetch_shared_down(const DecodeArgs& a, const DecodeSmem<COLS>& sm) {
  const int per = a.H / kDownRows;
  for (int j = blockIdx.x; j < per; j += gridDim.x) {
    const uint8_t *c, *s;
    uint32_t cb, sb;
    down_src<COLS>(a, sm, a.su, j, c, cb, s, sb);
    bulk_prefetch_l2(c, cb);
    bulk_prefetch_l2(s, sb);
  }
}

// Issues the copies of fill un into stage s (lane 0 of the producer warp).
template <int COLS>
__device__ void issue_unit(const DecodeArgs& a, DecodeSmem<COLS>& sm, int s, const Unit& un) {
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
    const int e = shared ? 0 : uw_expert(sm.uw[un.slot]);
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
  if (un.kind == U_DENSE) {
    const DMat& D = a.dense;
    const StageMap mp = dense_map(D.fmt, a.H);
    const size_t pc = code_pitch(D.fmt, a.H), ps = scale_pitch(D.fmt, a.H);
    const size_t r0 = static_cast<size_t>(un.chunk) * kDownRows;
    const uint32_t cbytes = static_cast<uint32_t>(kDownRows * pc);
    const uint32_t sbytes = static_cast<uint32_t>(kDownRows * ps);
    mbar_arrive_expect_tx(bar, cbytes + sbytes + 16);
    bulk_g2s(st + mp.ca, D.codes + r0 * pc, cbytes, bar);
    bulk_g2s(st + mp.sa, D.scales + r0 * ps, sbytes, bar);
    bulk_g2s(sm.stage_cb[s], D.cb, 16, bar);
    return;
  }
  // down fill: weights now, the unit's quantized h (all columns) once it is complete
  const DMat& D = un.kind == U_SDOWN ? a.sdown : a.down;
  const StageMap mp = down_map(D.fmt, a.I, COLS);
  const uint8_t *c, *sc;
  uint32_t cbytes, sbytes;
  down_src<COLS>(a, sm, un.slot, un.chunk, c, cbytes, sc, sbytes);
  const uint32_t hqb = static_cast<uint32_t>(COLS * a.I);
  const uint32_t hdb = static_cast<uint32_t>(COLS * a.hd_stride);
  mbar_arrive_expect_tx(bar, cbytes + sbytes + hqb + hdb + 16);
  bulk_g2s(st + mp.ca, c, cbytes, bar);
  bulk_g2s(st + mp.sa, sc, sbytes, bar);
  const uint32_t w = sm.uw[un.slot];
  const int e = un.kind == U_SDOWN ? 0 : uw_expert(w);
  bulk_g2s(sm.stage_cb[s], D.cb + static_cast<size_t>(e) * D.cb_stride, 16, bar);
  const uint32_t need = static_cast<uint32_t>(a.I / 32) * static_cast<uint32_t>(__popc(uw_mask(w)));
  if (!spin_until_geq(&a.ctr[kCtrHqDone + kCtrLine * un.slot], need, a.spin))
    set_status(a.status, MOEQ_ERR_DEVICE_TIMEOUT);
  asm volatile("fence.proxy.async.global;" ::: "memory");
  bulk_g2s(st + mp.cb, a.hq + static_cast<size_t>(un.slot) * COLS * a.I, hqb, bar);
  bulk_g2s(st + mp.sb, a.hd + static_cast<size_t>(un.slot) * COLS * a.hd_stride, hdb, bar);
}

// ------------------------------------------------------------------ compute side
__device__ __forceinline__ void load_q(const int8_t* p, int* q) {
  const int4 q0 = *reinterpret_cast<const int4*>(p);
  const int4 q1 = *reinterpret_cast<const int4*>(p + 16);
  q[0] = q0.x; q[1] = q0.y; q[2] = q0.z; q[3] = q0.w;
  q[4] = q1.x; q[5] = q1.y; q[6] = q1.z; q[7] = q1.w;
}

// Rows r0 and r1 of the gate and up tiles in the stage against the quantized x
// of column c0 in shared memory: g[0], u[0] for r0 and g[1], u[1] for r1.
// vec: debug vector of (c0, slot).
template <int FMT, bool DBG, int COLS>
__device__ void gu_rows(const DecodeArgs& a, const DecodeSmem<COLS>& sm, const uint8_t* st,
                        const uint32_t* cbg, const uint32_t* cbu, int r0, int r1, int row_base,
                        int c0, int vec, int lane, float* g, float* u) {
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
  const int8_t* xq = sm.xq[c0];
  const float* xdv = sm.xd[c0];
  float ag0 = 0.0f, au0 = 0.0f, ag1 = 0.0f, au1 = 0.0f;
#pragma unroll 1
  for (int b = lane; b < nb; b += 32) {
    int q[8];
    load_q(xq + 32 * b, q);
    const float xd = xdv[b];
    const int sg0 = block_dot<FMT>(gc0 + b * BC, cbg, q);
    const int su0 = block_dot<FMT>(uc0 + b * BC, cbu, q);
    const int sg1 = block_dot<FMT>(gc1 + b * BC, cbg, q);
    const int su1 = block_dot<FMT>(uc1 + b * BC, cbu, q);
    ag0 = fmaf(block_scale<FMT>(gs0, b) * xd, static_cast<float>(sg0), ag0);
    au0 = fmaf(block_scale<FMT>(us0, b) * xd, static_cast<float>(su0), au0);
    ag1 = fmaf(block_scale<FMT>(gs1, b) * xd, static_cast<float>(sg1), ag1);
    au1 = fmaf(block_scale<FMT>(us1, b) * xd, static_cast<float>(su1), au1);
    if (DBG && a.dbg.S_gate) {
      a.dbg.S_gate[(static_cast<size_t>(vec) * a.I + row_base + r0) * nb + b] = sg0;
      a.dbg.S_gate[(static_cast<size_t>(vec) * a.I + row_base + r1) * nb + b] = sg1;
    }
    if (DBG && a.dbg.S_up) {
      a.dbg.S_up[(static_cast<size_t>(vec) * a.I + row_base + r0) * nb + b] = su0;
      a.dbg.S_up[(static_cast<size_t>(vec) * a.I + row_base + r1) * nb + b] = su1;
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

// As gu_rows, for every column: each block is expanded once and dotted with
// the COLS quantized columns. g[j * COLS + c], u[j * COLS + c] for row j.
// vec[c]: debug vector of column c (< 0: the column is not written).
template <int FMT, bool DBG, int COLS>
__device__ void gu_rows_cols(const DecodeArgs& a, const DecodeSmem<COLS>& sm, const uint8_t* st,
                             const uint32_t* cbg, const uint32_t* cbu, int r0, int r1,
                             int row_base, const int* vec, int lane, float* g, float* u) {
  constexpr int BC = block_bytes<FMT>();
  constexpr int SB = FMT == 4 ? 1 : 2;
  const StageMap mp = gu_map(FMT, a.H);
  const int nb = a.H / 32;
  const int rr[2] = {r0, r1};
  float ag[2][COLS], au[2][COLS];
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int c = 0; c < COLS; ++c) ag[j][c] = au[j][c] = 0.0f;
#pragma unroll 1
  for (int b = lane; b < nb; b += 32) {
    int q[COLS][8];
    float xd[COLS];
#pragma unroll
    for (int c = 0; c < COLS; ++c) {
      load_q(sm.xq[c] + 32 * b, q[c]);
      xd[c] = sm.xd[c][b];
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int m = 0; m < 2; ++m) {  // m = 0 gate, 1 up
        const uint8_t* cp = st + (m ? mp.cb : mp.ca) + rr[j] * nb * BC + b * BC;
        const float ws = block_scale<FMT>(st + (m ? mp.sb : mp.sa) + rr[j] * nb * SB, b);
        uint32_t v[8];
        block_expand<FMT>(cp, m ? cbu : cbg, v);
#pragma unroll
        for (int c = 0; c < COLS; ++c) {
          const int S = dot8(v, q[c]);
          float& acc = m ? au[j][c] : ag[j][c];
          acc = fmaf(ws * xd[c], static_cast<float>(S), acc);
          if (DBG && vec[c] >= 0) {
            int32_t* dst = m ? a.dbg.S_up : a.dbg.S_gate;
            if (dst) dst[(static_cast<size_t>(vec[c]) * a.I + row_base + rr[j]) * nb + b] = S;
          }
        }
      }
    }
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) {
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int c = 0; c < COLS; ++c) {
        ag[j][c] += __shfl_xor_sync(0xffffffffu, ag[j][c], d);
        au[j][c] += __shfl_xor_sync(0xffffffffu, au[j][c], d);
      }
  }
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int c = 0; c < COLS; ++c) {
      g[j * COLS + c] = ag[j][c];
      u[j * COLS + c] = au[j][c];
    }
}

// Rows wg, wg + 8, wg + 16, wg + 24 of the down tile in the stage against the
// quantized h of column c0 of the unit, which the producer placed in the same
// stage. vec: debug vector of (c0, slot).
template <int FMT, bool DBG>
__device__ void down_rows(const DecodeArgs& a, const uint8_t* st, const StageMap& mp,
                          const uint32_t* cb, int wg, int lane, int chunk, int c0, int vec,
                          float* o) {
  constexpr int BC = block_bytes<FMT>();
  constexpr int SB = FMT == 4 ? 1 : 2;
  constexpr int R = kDownRows / kGroupWarps;
  const int nb = a.I / 32;
  const int8_t* hq = reinterpret_cast<const int8_t*>(st + mp.cb) + static_cast<size_t>(c0) * a.I;
  const uint16_t* hd = reinterpret_cast<const uint16_t*>(st + mp.sb + c0 * a.hd_stride);
  float acc[R];
#pragma unroll
  for (int j = 0; j < R; ++j) acc[j] = 0.0f;
#pragma unroll 1
  for (int b = lane; b < nb; b += 32) {
    int q[8];
    load_q(hq + 32 * b, q);
    const float hdf = f16_bits_to_f32(hd[b]);
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const int r = wg + kGroupWarps * j;
      const int d = block_dot<FMT>(st + mp.ca + r * nb * BC + b * BC, cb, q);
      acc[j] = fmaf(block_scale<FMT>(st + mp.sa + r * nb * SB, b) * hdf, static_cast<float>(d), acc[j]);
      if (DBG && a.dbg.S_down)
        a.dbg.S_down[(static_cast<size_t>(vec) * a.H + chunk * kDownRows + r) * nb + b] = d;
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

// Rows wg + 8 j of a 32-row tile (codes at ca, scales at sa, K = 32 nb) against
// COLS activation vectors: int8 act + c * act_stride with fp16 scales
// (dh + c * dh_stride, in the stage) or fp32 scales (df[c], shared memory).
// Each block is expanded once. o[j * COLS + c]. vec as in gu_rows_cols.
template <int FMT, bool DBG, int COLS, bool F16SCALES>
__device__ void rows_cols(const DecodeArgs& a, const uint8_t* st, uint32_t ca, uint32_t sa, int nb,
                          const int8_t* act, int act_stride, const uint8_t* dh, int dh_stride,
                          const float (*df)[kMaxH / 32], const uint32_t* cb, int wg, int lane,
                          int row0, const int* vec, float* o) {
  constexpr int BC = block_bytes<FMT>();
  constexpr int SB = FMT == 4 ? 1 : 2;
  constexpr int R = kDownRows / kGroupWarps;
  float acc[R][COLS];
#pragma unroll
  for (int j = 0; j < R; ++j)
#pragma unroll
    for (int c = 0; c < COLS; ++c) acc[j][c] = 0.0f;
#pragma unroll 1
  for (int b = lane; b < nb; b += 32) {
    int q[COLS][8];
    float d[COLS];
#pragma unroll
    for (int c = 0; c < COLS; ++c) {
      load_q(act + static_cast<size_t>(c) * act_stride + 32 * b, q[c]);
      if constexpr (F16SCALES)
        d[c] = f16_bits_to_f32(reinterpret_cast<const uint16_t*>(dh + c * dh_stride)[b]);
      else
        d[c] = df[c][b];
    }
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const int r = wg + kGroupWarps * j;
      uint32_t v[8];
      block_expand<FMT>(st + ca + r * nb * BC + b * BC, cb, v);
      const float ws = block_scale<FMT>(st + sa + r * nb * SB, b);
#pragma unroll
      for (int c = 0; c < COLS; ++c) {
        const int S = dot8(v, q[c]);
        acc[j][c] = fmaf(ws * d[c], static_cast<float>(S), acc[j][c]);
        if (DBG && vec && vec[c] >= 0 && a.dbg.S_down)
          a.dbg.S_down[(static_cast<size_t>(vec[c]) * a.H + row0 + r) * nb + b] = S;
      }
    }
  }
#pragma unroll
  for (int dd = 16; dd >= 1; dd >>= 1) {
#pragma unroll
    for (int j = 0; j < R; ++j)
#pragma unroll
      for (int c = 0; c < COLS; ++c) acc[j][c] += __shfl_xor_sync(0xffffffffu, acc[j][c], dd);
  }
#pragma unroll
  for (int j = 0; j < R; ++j)
#pragma unroll
    for (int c = 0; c < COLS; ++c) o[j * COLS + c] = acc[j][c];
}

// Router row r of the stage against every column: l[c].
template <int COLS>
__device__ void router_row(const DecodeArgs& a, const DecodeSmem<COLS>& sm, const uint8_t* st,
                           int r, int lane, float* l) {
  const uint8_t* wrow = st + static_cast<size_t>(r) * a.H * 2;
  float acc[COLS];
#pragma unroll
  for (int c = 0; c < COLS; ++c) acc[c] = 0.0f;
  for (int i = 0; i < a.H / 256; ++i) {
    const int k0 = 256 * i + 8 * lane;
    const uint4 w = *reinterpret_cast<const uint4*>(wrow + 2 * k0);
#pragma unroll
    for (int c = 0; c < COLS; ++c) {
      const uint4 x = COLS == 1 ? *reinterpret_cast<const uint4*>(sm.xb + k0)
                                : __ldg(reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(c) * a.H + k0));
      float s = acc[c];
      s = fmaf(bf16_lo(x.x), bf16_lo(w.x), s);
      s = fmaf(bf16_hi(x.x), bf16_hi(w.x), s);
      s = fmaf(bf16_lo(x.y), bf16_lo(w.y), s);
      s = fmaf(bf16_hi(x.y), bf16_hi(w.y), s);
      s = fmaf(bf16_lo(x.z), bf16_lo(w.z), s);
      s = fmaf(bf16_hi(x.z), bf16_hi(w.z), s);
      s = fmaf(bf16_lo(x.w), bf16_lo(w.w), s);
      s = fmaf(bf16_hi(x.w), bf16_hi(w.w), s);
      acc[c] = s;
    }
  }
#pragma unroll
  for (int c = 0; c < COLS; ++c) l[c] = warp_sum_canonical(acc[c]);
}

// Rotates (H32) and quantizes (Q8) one 32-block of h of (unit, column c) by
// one warp; lane i holds element i. Publishes the block.
template <int COLS>
__device__ void quantize_h_block(const DecodeArgs& a, float v, int unit, int c, int vec, int blk,
                                 int lane) {
  if (a.signs_h) v = h32_warp(v, __ldg(&a.signs_h[blk]), lane);
  uint16_t db;
  const int8_t q = q8_warp(v, db);
  const size_t hv = static_cast<size_t>(unit) * COLS + c;
  a.hq[hv * a.I + 32 * blk + lane] = q;
  if (lane == 0) reinterpret_cast<uint16_t*>(a.hd + hv * a.hd_stride)[blk] = db;
  if (a.dbg.hq) a.dbg.hq[static_cast<size_t>(vec) * a.I + 32 * blk + lane] = q;
  if (a.dbg.hd && lane == 0) a.dbg.hd[static_cast<size_t>(vec) * (a.I / 32) + blk] = db;
  __syncwarp();
  if (lane == 0) red_add_release(&a.ctr[kCtrHqDone + kCtrLine * unit], 1u);
}

// Computes fill n (unit un) from stage s with the 8 warps of compute group grp
// (wg = warp in group), releasing the stage as soon as it is read, then does
// the fill's share of publishing. first_prev: this group's previous first-half
// gate/up fill (-1 if none).
template <int COLS, bool DBG>
__device__ void compute_unit(const DecodeArgs& a, DecodeSmem<COLS>& sm, int s, int n, const Unit& un,
                             int grp, int wg, int lane, int& first_prev) {
  const uint8_t* st = sm.stage[s];
  const int bar = kBarGroup + grp;
  const int t = wg * 32 + lane;
  constexpr int R = kDownRows / kGroupWarps;
  if (un.kind == U_ROUTE) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[s]);
    route_item<COLS>(a, sm, bar, t);
    return;
  }
  if (un.kind == U_ROUTER) {
    float l[COLS];
    if (wg < kRouterRows) router_row<COLS>(a, sm, st, wg, lane, l);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[s]);
    if (wg < kRouterRows && lane == 0) {
      const int ex = un.chunk * kRouterRows + wg;
#pragma unroll
      for (int c = 0; c < COLS; ++c) {
        a.logits[c * a.E + ex] = l[c];
        if (DBG && a.dbg.logits) a.dbg.logits[c * a.E + ex] = l[c];
      }
    }
    named_bar(bar, kGroupThreads);
    if (t == 0) red_add_release(&a.ctr[kCtrRouter], 1u);
    return;
  }
  if (un.kind == U_DENSE) {
    const DMat& D = a.dense;
    uint32_t cb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) cb[i] = sm.stage_cb[s][i];
    const StageMap mp = dense_map(D.fmt, a.H);
    const int nb = a.H / 32;
    float o[R * COLS];
    const int8_t* act = &sm.xq[0][0];
    if (D.fmt == 2)
      rows_cols<2, false, COLS, false>(a, st, mp.ca, mp.sa, nb, act, kMaxH, nullptr, 0, sm.xd, cb, wg, lane, 0, nullptr, o);
    else if (D.fmt == 3)
      rows_cols<3, false, COLS, false>(a, st, mp.ca, mp.sa, nb, act, kMaxH, nullptr, 0, sm.xd, cb, wg, lane, 0, nullptr, o);
    else
      rows_cols<4, false, COLS, false>(a, st, mp.ca, mp.sa, nb, act, kMaxH, nullptr, 0, sm.xd, cb, wg, lane, 0, nullptr, o);
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&sm.empty[s]);
#pragma unroll
      for (int j = 0; j < R; ++j)
#pragma unroll
        for (int c = 0; c < COLS; ++c)
          a.y_dense[static_cast<size_t>(c) * D.rows + un.chunk * kDownRows + wg + kGroupWarps * j] =
              o[j * COLS + c];
    }
    return;
  }
  const uint32_t uwd = sm.uw[un.slot];
  const uint32_t mask = uw_mask(uwd);
  // a unit used by one column only takes the one-column path
  const bool single = COLS == 1 || __popc(mask) == 1;
  const int c0 = __ffs(mask) - 1;
  if (un.kind == U_SGU || un.kind == U_GU) {
    const int fmt = un.kind == U_SGU ? a.sgate.fmt : a.gate.fmt;
    uint32_t cbg[4], cbu[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      cbg[i] = sm.stage_cb[s][i];
      cbu[i] = sm.stage_cb[s][4 + i];
    }
    const int base = un.chunk * kGuRows;
    float g[2 * COLS], u[2 * COLS];
    if (single) {
      const int vec = dbg_vec(a, c0, uw_slot(uwd, c0));
      float g1[2], u1[2];
      if (fmt == 2) gu_rows<2, DBG, COLS>(a, sm, st, cbg, cbu, wg, wg + kGroupWarps, base, c0, vec, lane, g1, u1);
      else if (fmt == 3) gu_rows<3, DBG, COLS>(a, sm, st, cbg, cbu, wg, wg + kGroupWarps, base, c0, vec, lane, g1, u1);
      else gu_rows<4, DBG, COLS>(a, sm, st, cbg, cbu, wg, wg + kGroupWarps, base, c0, vec, lane, g1, u1);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        g[j * COLS] = g1[j];
        u[j * COLS] = u1[j];
      }
    } else if constexpr (COLS > 1) {
      int vec[COLS];
#pragma unroll
      for (int c = 0; c < COLS; ++c) vec[c] = ((mask >> c) & 1u) ? dbg_vec(a, c, uw_slot(uwd, c)) : -1;
      if (fmt == 2) gu_rows_cols<2, DBG, COLS>(a, sm, st, cbg, cbu, wg, wg + kGroupWarps, base, vec, lane, g, u);
      else if (fmt == 3) gu_rows_cols<3, DBG, COLS>(a, sm, st, cbg, cbu, wg, wg + kGroupWarps, base, vec, lane, g, u);
      else gu_rows_cols<4, DBG, COLS>(a, sm, st, cbg, cbu, wg, wg + kGroupWarps, base, vec, lane, g, u);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[s]);
    const bool first_half = (un.chunk & 1) == 0;
    if (first_half && first_prev >= 0) {
      // the other group must have consumed this group's previous first half
      if (t == 0 && !smem_wait_eq(&sm.hs_ack[grp], first_prev)) set_status(a.status, MOEQ_ERR_DEVICE_TIMEOUT);
      named_bar(bar, kGroupThreads);
    }
    float (*hs)[kGuRows] = first_half ? sm.hs_first[grp] : sm.hs_second[grp];
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r = wg + kGroupWarps * j;
#pragma unroll
        for (int c = 0; c < COLS; ++c) {
          const bool mine = single ? c == c0 : ((mask >> c) & 1u) != 0;
          if (!mine) continue;
          const float gv = single ? g[j * COLS] : g[j * COLS + c];
          const float uv = single ? u[j * COLS] : u[j * COLS + c];
          const float h = gv * uv / (1.0f + expf(-gv));
          hs[c][r] = h;
          if (DBG && a.dbg.h)
            a.dbg.h[static_cast<size_t>(dbg_vec(a, c, uw_slot(uwd, c))) * a.I + base + r] = h;
        }
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
    // second half: the first half was fill n - 1, computed by the other group;
    // warp c quantizes the block of column c
    const int other = grp ^ 1;
    if constexpr (COLS == 1) {
      if (wg == 0) {
        if (lane == 0 && !smem_wait_eq(&sm.hs_seq[other], n - 1)) set_status(a.status, MOEQ_ERR_DEVICE_TIMEOUT);
        __syncwarp();
        __threadfence_block();
        const float v = lane < kGuRows ? sm.hs_first[other][0][lane] : sm.hs_second[grp][0][lane - kGuRows];
        __syncwarp();
        if (lane == 0) {
          __threadfence_block();
          sm.hs_ack[other] = n - 1;
        }
        quantize_h_block<COLS>(a, v, un.slot, 0, dbg_vec(a, 0, uw_slot(uwd, 0)), un.chunk / 2, lane);
      }
    } else {
      const bool qwarp = wg < COLS && ((mask >> wg) & 1u);
      if (t == 0 && !smem_wait_eq(&sm.hs_seq[other], n - 1)) set_status(a.status, MOEQ_ERR_DEVICE_TIMEOUT);
      named_bar(bar, kGroupThreads);
      __threadfence_block();
      float v = 0.0f;
      if (qwarp) v = lane < kGuRows ? sm.hs_first[other][wg][lane] : sm.hs_second[grp][wg][lane - kGuRows];
      named_bar(bar, kGroupThreads);
      if (t == 0) {
        __threadfence_block();
        sm.hs_ack[other] = n - 1;
      }
      if (qwarp) quantize_h_block<COLS>(a, v, un.slot, wg, dbg_vec(a, wg, uw_slot(uwd, wg)), un.chunk / 2, lane);
    }
    return;
  }
  // down rows of the unit, for each column that uses it
  const int fmt = un.kind == U_SDOWN ? a.sdown.fmt : a.down.fmt;
  uint32_t cb[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) cb[i] = sm.stage_cb[s][i];
  const StageMap mp = down_map(fmt, a.I, COLS);
  float o[R * COLS];
  if (single) {
    const int vec = dbg_vec(a, c0, uw_slot(uwd, c0));
    float o1[R];
    if (fmt == 2) down_rows<2, DBG>(a, st, mp, cb, wg, lane, un.chunk, c0, vec, o1);
    else if (fmt == 3) down_rows<3, DBG>(a, st, mp, cb, wg, lane, un.chunk, c0, vec, o1);
    else if (fmt == MOEQ_FP3_PACKED24) down_rows<MOEQ_FP3_PACKED24, DBG>(a, st, mp, cb, wg, lane, un.chunk, c0, vec, o1);
    else down_rows<4, DBG>(a, st, mp, cb, wg, lane, un.chunk, c0, vec, o1);
#pragma unroll
    for (int j = 0; j < R; ++j) o[j * COLS] = o1[j];
  } else if constexpr (COLS > 1) {
    int vec[COLS];
#pragma unroll
    for (int c = 0; c < COLS; ++c) vec[c] = ((mask >> c) & 1u) ? dbg_vec(a, c, uw_slot(uwd, c)) : -1;
    const int8_t* act = reinterpret_cast<const int8_t*>(st + mp.cb);
    const int row0 = un.chunk * kDownRows;
    const int nb = a.I / 32;
    if (fmt == 2)
      rows_cols<2, DBG, COLS, true>(a, st, mp.ca, mp.sa, nb, act, a.I, st + mp.sb, a.hd_stride, nullptr, cb, wg, lane, row0, vec, o);
    else if (fmt == 3)
      rows_cols<3, DBG, COLS, true>(a, st, mp.ca, mp.sa, nb, act, a.I, st + mp.sb, a.hd_stride, nullptr, cb, wg, lane, row0, vec, o);
    else if (fmt == MOEQ_FP3_PACKED24)
      rows_cols<MOEQ_FP3_PACKED24, DBG, COLS, true>(a, st, mp.ca, mp.sa, nb, act, a.I, st + mp.sb, a.hd_stride, nullptr, cb, wg, lane, row0, vec, o);
    else
      rows_cols<4, DBG, COLS, true>(a, st, mp.ca, mp.sa, nb, act, a.I, st + mp.sb, a.hd_stride, nullptr, cb, wg, lane, row0, vec, o);
  }
  __syncwarp();
  if (lane == 0) {
    mbar_arrive(&sm.empty[s]);
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const int row = un.chunk * kDownRows + wg + kGroupWarps * j;
#pragma unroll
      for (int c = 0; c < COLS; ++c) {
        const bool mine = single ? c == c0 : ((mask >> c) & 1u) != 0;
        if (!mine) continue;
        const float v = single ? o[j * COLS] : o[j * COLS + c];
        a.obuf[(static_cast<size_t>(un.slot) * COLS + c) * a.H + row] = v;
        if (DBG && a.dbg.o) a.dbg.o[static_cast<size_t>(dbg_vec(a, c, uw_slot(uwd, c))) * a.H + row] = v;
      }
    }
  }
  named_bar(bar, kGroupThreads);
  if (t == 0) red_add_release(&a.ctr[kCtrDownDone], 1u);
}

template <int COLS, bool DBG>
__global__ void __launch_bounds__(kThreads, 1) ffn_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  DecodeSmem<COLS>& sm = *reinterpret_cast<DecodeSmem<COLS>*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kGroupWarps);
    }
    sm.issued = 0;
    sm.have_route = 0;
    sm.nu = 0;
    for (int g = 0; g < kGroups; ++g) {
      sm.consumed[g] = g - kGroups;
      sm.hs_seq[g] = -1;
      sm.hs_ack[g] = -1;
    }
    // the shared unit: expert 0 of its role, every column, slot k
    uint32_t w = ((1u << COLS) - 1u) << 10;
    for (int c = 0; c < COLS; ++c) w |= static_cast<uint32_t>(a.k) << (16 + 4 * c);
    sm.uw[a.su] = w;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- producer warp
    if (lane == 0 && a.has_shared) prefetch_shared_down<COLS>(a, sm);
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
      if (item > a.route_idx && !sm.have_route) {
        fetch_route<COLS>(a, sm, lane);
        if (lane == 0) {
          sm.have_route = 1;
          trace_ev(a, 1, ntr, MOEQ_TRACE_TOPK, item);
        }
        __syncwarp();
      }
      Unit first{U_END, 0, 0};
      const int nf = item_fills(a, sm.nu, item, first);
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
            issue_unit<COLS>(a, sm, s, un);
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
    if constexpr (COLS == 1) {
      for (int i = tid; i < a.H / 8; i += kComputeThreads)
        reinterpret_cast<uint4*>(sm.xb)[i] = __ldg(reinterpret_cast<const uint4*>(a.x) + i);
      named_bar(kBarCompute, kComputeThreads);
    }
    // Q8 (after H32) of every 32-block of every column, one block per thread
    for (int i = tid; i < COLS * nbH; i += kComputeThreads) {
      const int c = i / nbH, b = i % nbH;
      float v[32];
      if constexpr (COLS == 1) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(static_cast<uint32_t>(sm.xb[32 * b + j]) << 16);
      } else {
        const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(c) * a.H + 32 * b);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 w = __ldg(src + j);
          v[8 * j + 0] = bf16_lo(w.x); v[8 * j + 1] = bf16_hi(w.x);
          v[8 * j + 2] = bf16_lo(w.y); v[8 * j + 3] = bf16_hi(w.y);
          v[8 * j + 4] = bf16_lo(w.z); v[8 * j + 5] = bf16_hi(w.z);
          v[8 * j + 6] = bf16_lo(w.w); v[8 * j + 7] = bf16_hi(w.w);
        }
      }
      if (a.signs_x) h32_thread(v, __ldg(&a.signs_x[b]));
      int qw[8];
      const uint16_t db = q8_thread(v, qw);
      reinterpret_cast<int4*>(sm.xq[c] + 32 * b)[0] = make_int4(qw[0], qw[1], qw[2], qw[3]);
      reinterpret_cast<int4*>(sm.xq[c] + 32 * b)[1] = make_int4(qw[4], qw[5], qw[6], qw[7]);
      sm.xd[c][b] = f16_bits_to_f32(db);
      if (blockIdx.x == 0) {
        if (a.dbg.xq) {
          int8_t* dst = a.dbg.xq + static_cast<size_t>(c) * a.H + 32 * b;
          reinterpret_cast<int4*>(dst)[0] = make_int4(qw[0], qw[1], qw[2], qw[3]);
          reinterpret_cast<int4*>(dst)[1] = make_int4(qw[4], qw[5], qw[6], qw[7]);
        }
        if (a.dbg.xd) a.dbg.xd[c * nbH + b] = db;
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
      compute_unit<COLS, DBG>(a, sm, s, it, un, grp, wg, lane, first_prev);
      if (wg == 0 && lane == 0) trace_ev(a, role, ntr, MOEQ_TRACE_DONE, u);
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  int ntd = 0;  // teardown trace events (role 2, thread 0)
  if (tid == 0) trace_ev(a, 2, ntd, MOEQ_TRACE_START, 0);
  if (warp == kProducerWarp && lane == 0) {
    // fills issued but never waited for (only after a timeout): let them land
    for (int g = 0; g < kGroups; ++g)
      for (int j = sm.consumed[g] + kGroups; j < sm.issued; j += kGroups)
        if (!mbar_wait(&sm.full[j % kStages], (j / kStages) & 1)) break;
  }
  // combine y in slot order once every down item is done; 32 rows per warp
  const int per = a.H / kDownRows;
  const int nchunks = COLS * per;
  constexpr int kWarps = kThreads / 32;
  if (static_cast<int>(blockIdx.x) * kWarps < nchunks) {
    if (warp == 0) {
      if (!sm.have_route) fetch_route<COLS>(a, sm, lane);
      const uint32_t target = static_cast<uint32_t>(a.nSD + sm.nu * per);
      if (lane == 0 && !spin_until_geq(&a.ctr[kCtrDownDone], target, a.spin))
        set_status(a.status, MOEQ_ERR_DEVICE_TIMEOUT);
      if (lane == 0) trace_ev(a, 2, ntd, MOEQ_TRACE_READY, 0);
      __syncwarp();
    }
    __syncthreads();
    const int cc = static_cast<int>(blockIdx.x) * kWarps + warp;
    if (cc < nchunks) {
      const int c = cc / per;
      const int row = (cc % per) * kDownRows + lane;
      // every slot's output in flight at once, then summed in slot order
      float v[kMaxK];
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        v[j] = j < a.k ? __ldcg(&a.obuf[(static_cast<size_t>(sm.uof[c][j]) * COLS + c) * a.H + row]) : 0.0f;
      const float vs = a.has_shared ? __ldcg(&a.obuf[(static_cast<size_t>(a.su) * COLS + c) * a.H + row]) : 0.0f;
      float acc = 0.0f;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        if (j < a.k) acc = fmaf(sm.p[c][j], v[j], acc);
      if (a.has_shared) acc += vs;
      a.y[static_cast<size_t>(c) * a.H + row] = acc;
    }
    __syncthreads();
    if (tid == 0) trace_ev(a, 2, ntd, MOEQ_TRACE_DONE, 0);
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const uint32_t old = atomicAdd(&a.ctr[kCtrDone], 1u);
    trace_ev(a, 2, ntd, MOEQ_TRACE_EPI_END, static_cast<int>(old));
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

// Shapes the kernel handles (beyond the layer validation): every fill fits a stage.
bool shapes_fit(const moeq_layer* L, int cols) {
  if (L->H > kMaxH || L->I > kMaxH || L->E > kMaxE || L->E % kRouterRows || L->k > kMaxK)
    return false;
  if (static_cast<long>(kRouterRows) * L->H * 2 > kStageBytes) return false;
  if (gu_map(L->gate.fmt, L->H).total > static_cast<uint32_t>(kStageBytes)) return false;
  if (down_map(L->down.fmt, L->I, cols).total > static_cast<uint32_t>(kStageBytes)) return false;
  if (L->has_shared) {
    if (gu_map(L->sgate.fmt, L->H).total > static_cast<uint32_t>(kStageBytes)) return false;
    if (down_map(L->sdown.fmt, L->I, cols).total > static_cast<uint32_t>(kStageBytes)) return false;
  }
  return true;
}

// Fills the arguments shared by both entry points from a validated layer.
void fill_args(DecodeArgs& a, const moeq_layer* L, int cols, const uint16_t* x, float* y, void* ws,
               const DecodeWs& wl, int32_t* dev_status, const moeq_debug* dbg) {
  a.H = L->H; a.I = L->I; a.E = L->E; a.k = L->k;
  a.has_shared = L->has_shared ? 1 : 0;
  a.su = cols * L->k;
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
  // a caller's limit for the cross-CTA waits, one column only: with four
  // columns a routing record read before it is complete could name units
  // without columns, so the q=4 kernel keeps the default
  a.spin = kSpinLimit;
  if (cols == 1 && dbg && dbg->spin_limit != 0)
    a.spin = dbg->spin_limit < 0 ? 0u : static_cast<uint32_t>(dbg->spin_limit);
  a.nR = L->E / kRouterRows;
  a.nSG = a.has_shared ? L->I / (2 * kGuRows) : 0;
  a.nSD = a.has_shared ? L->H / kDownRows : 0;
  a.nDN = 0;
  a.route_base = route_base(wl.nunits);
  a.n_ctr = static_cast<int>(wl.n_ctr);
}

template <int COLS>
int launch(DecodeArgs& a, bool want_dbg, moeq_stream stream) {
  a.route_idx = a.nR + a.nSG + a.nDN;
  const DeviceInfo& di = device_info();
  const size_t smem = sizeof(DecodeSmem<COLS>);
  if (smem > di.max_smem_optin) return MOEQ_ERR_CUDA;
  // the debug instantiation carries the stores of intermediates and the timeline
  void (*kern)(const DecodeArgs) = want_dbg ? ffn_kernel<COLS, true> : ffn_kernel<COLS, false>;
  static thread_local int configured_dev = -1;
  if (configured_dev != di.device) {
    if (cudaFuncSetAttribute(ffn_kernel<COLS, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess ||
        cudaFuncSetAttribute(ffn_kernel<COLS, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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

}  // namespace

bool decode_supported(const moeq_layer* L) { return shapes_fit(L, 1); }

}  // namespace moeq

using namespace moeq;

extern "C" int moe_ffn_decode(const moeq_layer* L, const uint16_t* x, float* y, void* ws,
                              size_t ws_bytes, int32_t* dev_status, const moeq_debug* dbg,
                              moeq_stream stream) {
  int rc = validate_layer(L);
  if (rc) return rc;
  if (!x || !y) return MOEQ_ERR_ARG;
  if (!aligned16(x) || !aligned16(y)) return MOEQ_ERR_ALIGN;
  if (!shapes_fit(L, 1)) return MOEQ_ERR_SHAPE;
  const DecodeWs wl = decode_ws_layout(L->H, L->I, L->E, L->k, L->has_shared, 1);
  if (!ws || ws_bytes < wl.total || !aligned16(ws)) return MOEQ_ERR_WORKSPACE;
  DecodeArgs a{};
  fill_args(a, L, 1, x, y, ws, wl, dev_status, dbg);
  return launch<1>(a, dbg != nullptr, stream);
}

extern "C" int moe_ffn_verify_q4(const moeq_layer* L, const moeq_matrix* dense, const uint16_t* x,
                                 float* y, float* y_dense, void* ws, size_t ws_bytes,
                                 int32_t* dev_status, const moeq_debug* dbg, moeq_stream stream) {
  int rc = validate_layer(L);
  if (rc) return rc;
  if (!x || !y) return MOEQ_ERR_ARG;
  if (!aligned16(x) || !aligned16(y)) return MOEQ_ERR_ALIGN;
  if (!shapes_fit(L, 4)) return MOEQ_ERR_SHAPE;
  if (dense) {
    rc = validate_matrix(*dense, dense->rows, L->H, 1);
    if (rc) return rc;
    if (dense->fmt == MOEQ_FP3_PACKED24) return MOEQ_ERR_FORMAT;
    if (dense->rows % kDownRows) return MOEQ_ERR_SHAPE;
    if (dense_map(dense->fmt, L->H).total > static_cast<uint32_t>(kStageBytes)) return MOEQ_ERR_SHAPE;
    if (!y_dense) return MOEQ_ERR_ARG;
    if (!aligned16(y_dense)) return MOEQ_ERR_ALIGN;
  }
  const DecodeWs wl = verify_ws_layout(L->H, L->I, L->E, L->k, L->has_shared);
  if (!ws || ws_bytes < wl.total || !aligned16(ws)) return MOEQ_ERR_WORKSPACE;
  DecodeArgs a{};
  fill_args(a, L, 4, x, y, ws, wl, dev_status, dbg);
  if (dense) {
    a.dense = to_dmat(*dense);
    a.y_dense = y_dense;
    a.nDN = dense->rows / kDownRows;
  }
  return launch<4>(a, dbg != nullptr, stream);
}

// ---------------------------------------------------------------- decode with library-owned scratch
// The decode's scratch (counters, routing record, logits, quantized h,
// per-expert outputs) lives here instead of in a caller workspace, for
// callers that cannot allocate device memory. One array per device (the
// module's copy on each device); its address is looked up per device and
// per CUDA context.
namespace moeq {
namespace {

constexpr size_t kStaticScratchBytes = 160 * 1024;  // decode shapes up to this workspace size
static __device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices];
unsigned long long g_scratch_ctx[kMaxDevices];

// Unique id of the current CUDA context (driver entry points looked up through
// the runtime; 0 when unavailable).
unsigned long long current_context_id() {
  using GetCurrent = int (*)(void**);
  using GetId = int (*)(void*, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
  });
  if (!get_current || !get_id) return 0;
  void* ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != 0 || !ctx || get_id(ctx, &id) != 0) return 0;
  return id;
}

// Address of the current device's scratch, or nullptr. Looked up again when
// the current context differs from the one of the cached address (a device
// reset reloads the module in a new primary context).
void* static_scratch(int device) {
  if (device < 0 || device >= kMaxDevices) return nullptr;
  cudaFree(nullptr);  // make sure the device's primary context is current
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[device] || g_scratch_ctx[device] != ctx || ctx == 0) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[device] = p;
    g_scratch_ctx[device] = ctx;
  }
  return g_scratch_ptr[device];
}

}  // namespace
}  // namespace moeq

extern "C" int moe_ffn_decode_static(const moeq_layer* L, const uint16_t* x, float* y, int32_t* dev_status,
                                     moeq_stream stream) {
  int rc = validate_layer(L);
  if (rc) return rc;
  if (!x || !y) return MOEQ_ERR_ARG;
  if (!aligned16(x) || !aligned16(y)) return MOEQ_ERR_ALIGN;
  if (!shapes_fit(L, 1)) return MOEQ_ERR_SHAPE;
  const DecodeWs wl = decode_ws_layout(L->H, L->I, L->E, L->k, L->has_shared, 1);
  if (wl.total > kStaticScratchBytes) return MOEQ_ERR_WORKSPACE;
  void* ws = static_scratch(device_info().device);
  if (!ws) return MOEQ_ERR_CUDA;
  // the counters must start at zero: clear them on every call, so that a call
  // that ended in a device error does not leave stale counts for the next one
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  rc = cuda_status(cudaMemsetAsync(static_cast<uint8_t*>(ws) + wl.ctr, 0, 4 * wl.n_ctr, s));
  if (rc) return rc;
  DecodeArgs a{};
  fill_args(a, L, 1, x, y, ws, wl, dev_status, nullptr);
  return launch<1>(a, false, stream);
}

extern "C" int moe_ffn_stack_decode(const moeq_layer* layers, int nlayers, const uint16_t* x, float* r,
                                    void* ws, size_t ws_bytes, int32_t* dev_status, moeq_stream stream) {
  if (!layers || nlayers < 1) return MOEQ_ERR_ARG;
  const int H = layers[0].H;
  size_t need = 0;
  for (int l = 0; l < nlayers; ++l) {
    const int rc = validate_layer(&layers[l]);
    if (rc) return rc;
    if (layers[l].H != H) return MOEQ_ERR_SHAPE;
    if (!shapes_fit(&layers[l], 1)) return MOEQ_ERR_SHAPE;
    const DecodeWs wl = decode_ws_layout(layers[l].H, layers[l].I, layers[l].E, layers[l].k,
                                         layers[l].has_shared, 1);
    need = wl.total > need ? wl.total : need;
  }
  if (!x || !r) return MOEQ_ERR_ARG;
  if (!aligned16(x) || !aligned16(r)) return MOEQ_ERR_ALIGN;
  const size_t abytes = align256(2 * static_cast<size_t>(H)), ybytes = align256(4 * static_cast<size_t>(H));
  if (!ws || !aligned16(ws) || ws_bytes < need + abytes + ybytes) return MOEQ_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint16_t* a = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + need);
  float* y = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + need + abytes);
  // r_0 = float(x), a_0 = RMSNorm(r_0); per layer y = FFN_l(a_l), then
  // r_{l+1} = r_l + y and a_{l+1} = RMSNorm(r_{l+1}) (no norm after the last)
  int rc = stack_step_launch(x, nullptr, r, a, H, 1, s);
  for (int l = 0; l < nlayers && !rc; ++l) {
    rc = moe_ffn_decode(&layers[l], a, y, ws, need, dev_status, nullptr, stream);
    if (!rc) rc = stack_step_launch(nullptr, y, r, l + 1 < nlayers ? a : nullptr, H, 1, s);
  }
  return rc;
}

extern "C" int moe_ffn_stack_verify_q4(const moeq_layer* layers, int nlayers, const uint16_t* x, float* r,
                                       void* ws, size_t ws_bytes, int32_t* dev_status, moeq_stream stream) {
  if (!layers || nlayers < 1) return MOEQ_ERR_ARG;
  const int H = layers[0].H;
  size_t need = 0;
  for (int l = 0; l < nlayers; ++l) {
    const int rc = validate_layer(&layers[l]);
    if (rc) return rc;
    if (layers[l].H != H) return MOEQ_ERR_SHAPE;
    if (!shapes_fit(&layers[l], 4)) return MOEQ_ERR_SHAPE;
    const DecodeWs wl =
        verify_ws_layout(layers[l].H, layers[l].I, layers[l].E, layers[l].k, layers[l].has_shared);
    need = wl.total > need ? wl.total : need;
  }
  if (!x || !r) return MOEQ_ERR_ARG;
  if (!aligned16(x) || !aligned16(r)) return MOEQ_ERR_ALIGN;
  const size_t abytes = align256(8 * static_cast<size_t>(H)), ybytes = align256(16 * static_cast<size_t>(H));
  if (!ws || !aligned16(ws) || ws_bytes < need + abytes + ybytes) return MOEQ_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint16_t* a = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + need);
  float* y = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + need + abytes);
  // the decode stack's recurrence on each of the 4 columns; each layer's
  // weights are streamed once for all of them
  int rc = stack_step_launch(x, nullptr, r, a, H, 4, s);
  for (int l = 0; l < nlayers && !rc; ++l) {
    rc = moe_ffn_verify_q4(&layers[l], nullptr, a, y, nullptr, ws, need, dev_status, nullptr, stream);
    if (!rc) rc = stack_step_launch(nullptr, y, r, l + 1 < nlayers ? a : nullptr, H, 4, s);
  }
  return rc;
}
