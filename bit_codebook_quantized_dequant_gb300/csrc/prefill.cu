// Expert-grouped prefill of T tokens: every token gets the decode's result
// up to the rounding of the tensor-core contraction (bf16 operand parts, fp32
// sums; gemm_tc.cu), computed as
//   router + top-k of every token              (route.cu)
//   Q8 of every 32-block of x (after H32)       prep_x_kernel
//   stable counting sort of the (token, slot) pairs by expert
//                                               count_kernel, place_kernel
//   x's code x scale as bf16 parts, grouped     gather_kernel
//   grouped gate GEMM, then up GEMM with the SwiGLU, H32 and Q8 of h in its
//   epilogue, then down GEMM, per expert kind, on the tensor cores
//                                               gemm_tc.cu
//   gather-combine in slot order (+ residual)   combine_kernel
// all enqueued on the caller's stream with no host synchronization; the tile
// lists of the grouped GEMMs are built on the device from the expert counts.
//
// Sources: "deepseek-v4-flash-0731-evox3-rocm", section "The optimization
// ladder" (fused multi-token prefill, H32 on the activations); "Lucebox x
// Geometric ...", section "How the model fits" (layer-major batching of the
// prefill).
#include <cuda_runtime.h>

#include "moeq.h"
#include "moeq_device.cuh"
#include "moeq_host.h"
#include "moeq_layout.h"

namespace moeq {
namespace {

constexpr int kNT = 128;  // grouped rows per GEMM tile (gemm_tc.cu)
constexpr int kMT = 128;  // weight rows per GEMM tile (gemm_tc.cu)

struct PrefillArgs {
  int T, H, I, E, k, has_shared, ns;
  DMat gate, up, down, sgate, sup, sdown;
  const uint16_t* x;
  const uint32_t* signs_x;
  const uint32_t* signs_h;
  int8_t* xq;
  uint16_t* xd;
  int32_t* idx;
  float* p;
  int* counts;
  int* offsets;
  int* tiles_gu;
  int* tiles_dn;
  int* pid;
  int* pos;
  uint16_t* xhi;
  uint16_t* xlo;
  float* g;
  uint16_t* hhi;
  uint16_t* hlo;
  float* o;
  const float* residual;
  float* y;
  int32_t* status;
  moeq_debug dbg;
};

// Q8 (after H32) of every 32-block of x, one block per thread.
__global__ void prep_x_kernel(const PrefillArgs a) {
  const int nbH = a.H / 32;
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<size_t>(a.T) * nbH) return;
  const int b = static_cast<int>(i % nbH);
  const uint4* src = reinterpret_cast<const uint4*>(a.x + 32 * i);
  float v[32];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 w = __ldg(src + j);
    v[8 * j + 0] = bf16_lo(w.x); v[8 * j + 1] = bf16_hi(w.x);
    v[8 * j + 2] = bf16_lo(w.y); v[8 * j + 3] = bf16_hi(w.y);
    v[8 * j + 4] = bf16_lo(w.z); v[8 * j + 5] = bf16_hi(w.z);
    v[8 * j + 6] = bf16_lo(w.w); v[8 * j + 7] = bf16_hi(w.w);
  }
  if (a.signs_x) h32_thread(v, __ldg(&a.signs_x[b]));
  int qw[8];
  const uint16_t db = q8_thread(v, qw);
  int4* dq = reinterpret_cast<int4*>(a.xq + 32 * i);
  dq[0] = make_int4(qw[0], qw[1], qw[2], qw[3]);
  dq[1] = make_int4(qw[4], qw[5], qw[6], qw[7]);
  a.xd[i] = db;
  if (a.dbg.xq) {
    int4* d = reinterpret_cast<int4*>(a.dbg.xq + 32 * i);
    d[0] = dq[0];
    d[1] = dq[1];
  }
  if (a.dbg.xd) a.dbg.xd[i] = db;
}

// Expert histogram of the (token, slot) pairs.
__global__ void count_kernel(const PrefillArgs a) {
  const size_t n = static_cast<size_t>(a.T) * a.k;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int e = a.idx[i];
    if (e < 0 || e >= a.E) {
      set_status(a.status, MOEQ_ERR_DEVICE_INDEX);
      continue;
    }
    atomicAdd(&a.counts[e], 1);
  }
}

__device__ __forceinline__ int group_count(const PrefillArgs& a, int g) {
  return g < a.E ? a.counts[g] : a.T;
}

// Block-wide exclusive prefix of v over blockDim.x threads (multiple of 32);
// returns the prefix and writes the block total to *total.
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += o;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (threadIdx.x == 0) {
    int s = 0;
    for (int w = 0; w < nw; ++w) {
      const int t = warp_sums[w];
      warp_sums[w] = s;
      s += t;
    }
    warp_sums[nw] = s;
  }
  __syncthreads();
  const int r = warp_sums[warp] + incl - v;
  *total = warp_sums[nw];
  __syncthreads();
  return r;
}

// One CTA per group: its row offset and tile offsets (sums over the groups
// before it), then the stable placement of its pairs (ascending pair index =
// ascending token, then slot).
__global__ void place_kernel(const PrefillArgs a) {
  __shared__ int warp_sums[33];
  const int g = blockIdx.x;
  const int groups = a.E + (a.has_shared ? 1 : 0);
  int off = 0, tg = 0, td = 0;
  for (int j = threadIdx.x; j < g; j += blockDim.x) {
    const int n = group_count(a, j);
    off += n;
    const int nt = (n + kNT - 1) / kNT;
    tg += nt * (a.I / kMT);
    td += nt * (a.H / kMT);
  }
  int s_off, s_tg, s_td;
  block_exclusive_scan(off, warp_sums, &s_off);
  block_exclusive_scan(tg, warp_sums, &s_tg);
  block_exclusive_scan(td, warp_sums, &s_td);
  const int n = group_count(a, g);
  if (threadIdx.x == 0) {
    a.offsets[g] = s_off;
    a.tiles_gu[g] = s_tg;
    a.tiles_dn[g] = s_td;
    if (g == groups - 1) {
      const int nt = (n + kNT - 1) / kNT;
      a.offsets[groups] = s_off + n;
      a.tiles_gu[groups] = s_tg + nt * (a.I / kMT);
      a.tiles_dn[groups] = s_td + nt * (a.H / kMT);
    }
  }
  const int Tk = a.T * a.k;
  if (g == a.E) {  // shared expert: every token, in order
    for (int t = threadIdx.x; t < a.T; t += blockDim.x) a.pid[s_off + t] = Tk + t;
    return;
  }
  int run = 0;
  for (int base = 0; base < Tk; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const int f = (i < Tk && a.idx[i] == g) ? 1 : 0;
    int tot;
    const int pre = block_exclusive_scan(f, warp_sums, &tot);
    if (f) {
      const int r = s_off + run + pre;
      a.pid[r] = i;
      a.pos[i] = r;
    }
    run += tot;
  }
}

// Grouped activation parts for the tensor-core GEMM: row r of group order is
// token t = the token of pid[r]; v = q * d (x's int8 code times its block
// scale, exact in fp32) as xhi = bf16(v), xlo = bf16(v - xhi). One warp per
// grouped row.
__global__ void gather_kernel(const PrefillArgs a, int rows) {
  const int r = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const int pid = a.pid[r];
  const int Tk = a.T * a.k;
  const int t = pid >= Tk ? pid - Tk : pid / a.k;
  const int nbH = a.H / 32;
  const int8_t* src = a.xq + static_cast<size_t>(t) * a.H;
  const uint16_t* dsc = a.xd + static_cast<size_t>(t) * nbH;
  uint16_t* dhi = a.xhi + static_cast<size_t>(r) * a.H;
  uint16_t* dlo = a.xlo + static_cast<size_t>(r) * a.H;
  for (int c = lane; c < a.H / 8; c += 32) {  // 8 elements per step
    const uint2 q = *reinterpret_cast<const uint2*>(src + 8 * c);
    const float d = f16_bits_to_f32(dsc[(8 * c) / 32]);
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t w = i < 2 ? q.x : q.y;
      const int sh = 16 * (i & 1);
      const float v0 = __fmul_rn(static_cast<float>(static_cast<int8_t>(w >> sh)), d);
      const float v1 = __fmul_rn(static_cast<float>(static_cast<int8_t>(w >> (sh + 8))), d);
      uint32_t h;
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(v1), "f"(v0));
      const float r0 = __fsub_rn(v0, __uint_as_float(h << 16));
      const float r1 = __fsub_rn(v1, __uint_as_float(h & 0xffff0000u));
      uint32_t l;
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(l) : "f"(r1), "f"(r0));
      hi[i] = h;
      lo[i] = l;
    }
    *reinterpret_cast<uint4*>(dhi + 8 * c) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(dlo + 8 * c) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}

// y[t, :] = sum_s p[t, s] o[pos[t, s], :] (+ o_shared[t, :]) (+ residual[t, :]),
// four columns per thread.
__global__ void combine_kernel(const PrefillArgs a) {
  const int per_row = a.H / 4;
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<size_t>(a.T) * per_row) return;
  const int t = static_cast<int>(i / per_row), c = static_cast<int>(i % per_row);
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (int s = 0; s < a.k; ++s) {
    const float ps = a.p[static_cast<size_t>(t) * a.k + s];
    const int row = a.pos[static_cast<size_t>(t) * a.k + s];
    const float4 v = __ldcg(reinterpret_cast<const float4*>(a.o + static_cast<size_t>(row) * a.H) + c);
    acc.x = fmaf(ps, v.x, acc.x);
    acc.y = fmaf(ps, v.y, acc.y);
    acc.z = fmaf(ps, v.z, acc.z);
    acc.w = fmaf(ps, v.w, acc.w);
  }
  if (a.has_shared) {
    const size_t row = static_cast<size_t>(a.T) * a.k + t;
    const float4 v = __ldcg(reinterpret_cast<const float4*>(a.o + row * a.H) + c);
    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
  }
  if (a.residual) {
    const float4 r = __ldg(reinterpret_cast<const float4*>(a.residual + static_cast<size_t>(t) * a.H) + c);
    acc.x = r.x + acc.x; acc.y = r.y + acc.y; acc.z = r.z + acc.z; acc.w = r.w + acc.w;
  }
  reinterpret_cast<float4*>(a.y + static_cast<size_t>(t) * a.H)[c] = acc;
}

// r = float(x) for a bf16 [n] input.
__global__ void bf16_to_f32_kernel(const uint16_t* __restrict__ x, float* __restrict__ r, size_t n) {
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) r[i] = __uint_as_float(static_cast<uint32_t>(x[i]) << 16);
}

}  // namespace
}  // namespace moeq

using namespace moeq;

extern "C" int moe_ffn_prefill(const moeq_layer* L, const uint16_t* x, int T, const float* residual,
                               float* y, void* ws, size_t ws_bytes, int32_t* dev_status,
                               const moeq_debug* dbg, moeq_stream stream) {
  int rc = validate_layer(L);
  if (rc) return rc;
  if (L->down.fmt == MOEQ_FP3_PACKED24) return MOEQ_ERR_FORMAT;  // decode-only layout
  if (T < 0) return MOEQ_ERR_SHAPE;
  if (T == 0) return MOEQ_OK;
  if (!x || !y) return MOEQ_ERR_ARG;
  if (!aligned16(x) || !aligned16(y) || (residual && !aligned16(residual))) return MOEQ_ERR_ALIGN;
  if (L->E > 1024 || static_cast<long long>(T) * L->k >= (1ll << 31) - L->k) return MOEQ_ERR_SHAPE;
  const PrefillWs wl = prefill_ws_layout(L->H, L->I, L->E, L->k, L->has_shared, T);
  if (!ws || ws_bytes < wl.total || !aligned16(ws)) return MOEQ_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);

  PrefillArgs a{};
  a.T = T; a.H = L->H; a.I = L->I; a.E = L->E; a.k = L->k;
  a.has_shared = L->has_shared ? 1 : 0;
  a.ns = L->k + a.has_shared;
  a.gate = to_dmat(L->gate); a.up = to_dmat(L->up); a.down = to_dmat(L->down);
  if (a.has_shared) {
    a.sgate = to_dmat(L->sgate); a.sup = to_dmat(L->sup); a.sdown = to_dmat(L->sdown);
  }
  a.x = x;
  a.signs_x = L->h32_signs_x;
  a.signs_h = L->h32_signs_h;
  a.xq = reinterpret_cast<int8_t*>(w + wl.xq);
  a.xd = reinterpret_cast<uint16_t*>(w + wl.xd);
  a.idx = reinterpret_cast<int32_t*>(w + wl.idx);
  a.p = reinterpret_cast<float*>(w + wl.p);
  a.counts = reinterpret_cast<int*>(w + wl.counts);
  a.offsets = reinterpret_cast<int*>(w + wl.offsets);
  a.tiles_gu = reinterpret_cast<int*>(w + wl.tiles_gu);
  a.tiles_dn = reinterpret_cast<int*>(w + wl.tiles_dn);
  a.pid = reinterpret_cast<int*>(w + wl.pid);
  a.pos = reinterpret_cast<int*>(w + wl.pos);
  a.xhi = reinterpret_cast<uint16_t*>(w + wl.xhi);
  a.xlo = reinterpret_cast<uint16_t*>(w + wl.xlo);
  a.g = reinterpret_cast<float*>(w + wl.g);
  a.hhi = reinterpret_cast<uint16_t*>(w + wl.hhi);
  a.hlo = reinterpret_cast<uint16_t*>(w + wl.hlo);
  a.o = reinterpret_cast<float*>(w + wl.o);
  a.residual = residual;
  a.y = y;
  a.status = dev_status;
  if (dbg) a.dbg = *dbg;

  const int groups = L->E + a.has_shared;
  if ((rc = cuda_status(cudaMemsetAsync(a.counts, 0, sizeof(int) * (groups + 1), s)))) return rc;
  if ((rc = route_topk_launch(x, T, L->router, L->E, L->H, L->k, a.idx, a.p,
                              dbg ? dbg->logits : nullptr, s)))
    return rc;
  const size_t nblk = static_cast<size_t>(T) * (L->H / 32);
  prep_x_kernel<<<static_cast<unsigned>((nblk + 255) / 256), 256, 0, s>>>(a);
  count_kernel<<<256, 256, 0, s>>>(a);
  place_kernel<<<groups, 256, 0, s>>>(a);
  if ((rc = cuda_status(cudaGetLastError()))) return rc;
  if (dbg && (dbg->idx || dbg->p)) {
    const size_t tk = static_cast<size_t>(T) * L->k;
    if (dbg->idx && (rc = cuda_status(cudaMemcpyAsync(dbg->idx, a.idx, 4 * tk, cudaMemcpyDeviceToDevice, s))))
      return rc;
    if (dbg->p && (rc = cuda_status(cudaMemcpyAsync(dbg->p, a.p, 4 * tk, cudaMemcpyDeviceToDevice, s))))
      return rc;
  }
  const int rows = T * L->k + (a.has_shared ? T : 0);
  gather_kernel<<<(rows + 7) / 8, 256, 0, s>>>(a, rows);
  if ((rc = cuda_status(cudaGetLastError()))) return rc;
  TcGemm g{};
  g.offsets = a.offsets;
  g.rows = rows;
  g.g = a.g;
  g.hhi = a.hhi;
  g.hlo = a.hlo;
  g.signs_h = a.signs_h;
  g.o = a.o;
  g.pid = a.pid;
  g.T = T;
  g.k = L->k;
  g.ns = a.ns;
  g.status = dev_status;
  // gate, then up (+SwiGLU, H32, Q8 of h), then down; routed and shared experts
  for (int pass = 0; pass < 6; ++pass) {
    const int stage = pass / 2;  // 0 gate, 1 up, 2 down
    const bool shared = pass & 1;
    if (shared && !a.has_shared) continue;
    g.epi = stage;
    g.shared = shared ? 1 : 0;
    g.g0 = shared ? L->E : 0;
    g.g1 = shared ? L->E + 1 : L->E;
    g.dbg = a.dbg;
    g.dbg.trace = nullptr;
    if (stage < 2) {
      g.w = stage == 0 ? (shared ? a.sgate : a.gate) : (shared ? a.sup : a.up);
      g.toff = a.tiles_gu;
      g.K = L->H;
      g.R = L->I;
      g.act_hi = a.xhi;
      g.act_lo = a.xlo;
    } else {
      g.w = shared ? a.sdown : a.down;
      g.toff = a.tiles_dn;
      g.K = L->I;
      g.R = L->H;
      g.act_hi = a.hhi;
      g.act_lo = a.hlo;
    }
    if ((rc = tc_grouped_gemm(g, s))) return rc;
  }
  const size_t nout = static_cast<size_t>(T) * (L->H / 4);
  combine_kernel<<<static_cast<unsigned>((nout + 255) / 256), 256, 0, s>>>(a);
  return cuda_status(cudaGetLastError());
}

extern "C" int moe_ffn_stack_prefill(const moeq_layer* layers, int nlayers, const uint16_t* x, int T,
                                     float* r, void* ws, size_t ws_bytes, int32_t* dev_status,
                                     moeq_stream stream) {
  if (!layers || nlayers < 1) return MOEQ_ERR_ARG;
  if (T < 0) return MOEQ_ERR_SHAPE;
  const int H = layers[0].H;
  size_t need = 0;
  for (int l = 0; l < nlayers; ++l) {
    const int rc = validate_layer(&layers[l]);
    if (rc) return rc;
    if (layers[l].down.fmt == MOEQ_FP3_PACKED24) return MOEQ_ERR_FORMAT;
    if (layers[l].H != H) return MOEQ_ERR_SHAPE;
    const PrefillWs wl = prefill_ws_layout(layers[l].H, layers[l].I, layers[l].E, layers[l].k,
                                           layers[l].has_shared, T);
    need = wl.total > need ? wl.total : need;
  }
  if (T == 0) return MOEQ_OK;
  if (!x || !r) return MOEQ_ERR_ARG;
  if (!aligned16(x) || !aligned16(r)) return MOEQ_ERR_ALIGN;
  const size_t abytes = align256(2 * static_cast<size_t>(T) * H);
  if (!ws || !aligned16(ws) || ws_bytes < need + abytes) return MOEQ_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint16_t* a = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + need);
  const size_t n = static_cast<size_t>(T) * H;
  bf16_to_f32_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(x, r, n);
  int rc = cuda_status(cudaGetLastError());
  for (int l = 0; l < nlayers && !rc; ++l) {
    rc = moe_rmsnorm_bf16(r, T, H, a, stream);
    if (!rc) rc = moe_ffn_prefill(&layers[l], a, T, r, r, ws, need, dev_status, nullptr, stream);
  }
  return rc;
}
