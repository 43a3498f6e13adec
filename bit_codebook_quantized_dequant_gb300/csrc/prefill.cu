// Expert-grouped prefill of T tokens: every token gets the decode's result
// (up to fp32 rounding), computed as
//   router + top-k of every token              (route.cu)
//   Q8 of every 32-block of x (after H32)       prep_x_kernel
//   stable counting sort of the (token, slot) pairs by expert
//                                               count_kernel, place_kernel
//   grouped gate/up GEMM per expert, epilogue SwiGLU, H32 and Q8 of h
//                                               gu_kernel
//   grouped down GEMM per expert                down_kernel
//   gather-combine in slot order (+ residual)   combine_kernel
// all enqueued on the caller's stream with no host synchronization; the tile
// lists of the grouped GEMMs are built on the device from the expert counts.
//
// The grouped GEMMs here run on the CUDA cores: a weight block is expanded
// once per thread (byte permutes) and dotted (dp4a) with the int8 blocks of 8
// tokens, with the per-block scales applied in fp32 as in the decode.
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

constexpr int kNT = 64;   // tokens (grouped rows) per GEMM tile
constexpr int kMT = 32;   // weight rows per GEMM tile (one lane each)
constexpr int kKB = 16;   // 32-blocks per K chunk staged in shared memory
constexpr int kGemmThreads = 256;
constexpr int kTokPerWarp = kNT / (kGemmThreads / 32);  // 8

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
  int8_t* hq;
  uint16_t* hd;
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

// Group of a tile from the tile offsets (binary search over groups [g0, g1)).
__device__ __forceinline__ int tile_group(const int* toff, int g0, int g1, int tile) {
  int lo = g0, hi = g1 - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(&toff[mid]) <= tile) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void pid_split(const PrefillArgs& a, int pid, int& t, int& s) {
  const int Tk = a.T * a.k;
  if (pid >= Tk) {
    t = pid - Tk;
    s = a.k;
  } else {
    t = pid / a.k;
    s = pid - t * a.k;
  }
}

template <int FMT>
struct GemmSmem {
  static constexpr int BC = block_bytes<FMT>();
  static constexpr int WP = kKB * BC + 16;  // padded row pitch of a code tile
  uint8_t w[2][kMT][WP];                    // codes of one or two matrices
  uint16_t ws[2][kMT][kKB];                 // raw scales (fp16 bits or E8M0)
  int8_t act[kNT][kKB * 32 + 16];           // int8 activations, one row per grouped row
  float ad[kNT][kKB];                       // activation block scales
  int tok[kNT];                             // activation row (token or grouped row), -1 = none
  uint32_t cb[2][4];                        // codebook records
};

template <int FMT>
__device__ __forceinline__ float raw_scale(uint16_t r) {
  if constexpr (FMT == 4) return e8m0_to_f32(static_cast<uint8_t>(r));
  else return f16_bits_to_f32(r);
}

// Stages K chunk [kc, kc + kb) of rows r0.. of NM matrices and of the tile's
// activation rows into shared memory.
template <int FMT, int NM>
__device__ void stage_chunk(GemmSmem<FMT>& sm, const DMat* const* mats, int e, int r0, int K,
                            int kc, int kb, const int8_t* act, int act_pitch, const uint16_t* adsc,
                            int ad_pitch) {
  constexpr int BC = block_bytes<FMT>();
  const int nb = K / 32;
  const int tid = threadIdx.x;
  // codes: per row kb*BC bytes (a multiple of 8), in 8-byte pieces
  const int pieces = kb * BC / 8;
  for (int m = 0; m < NM; ++m) {
    const DMat& M = *mats[m];
    const uint8_t* base = M.codes + static_cast<size_t>(e) * M.stride_codes;
    for (int i = tid; i < kMT * pieces; i += blockDim.x) {
      const int r = i / pieces, c = i % pieces;
      const uint2 v = *reinterpret_cast<const uint2*>(base + (static_cast<size_t>(r0 + r) * nb + kc) * BC + 8 * c);
      *reinterpret_cast<uint2*>(&sm.w[m][r][8 * c]) = v;
    }
    const uint8_t* sb = M.scales + static_cast<size_t>(e) * M.stride_scales;
    for (int i = tid; i < kMT * kb; i += blockDim.x) {
      const int r = i / kb, c = i % kb;
      const size_t at = static_cast<size_t>(r0 + r) * nb + kc + c;
      sm.ws[m][r][c] = FMT == 4 ? static_cast<uint16_t>(sb[at]) : reinterpret_cast<const uint16_t*>(sb)[at];
    }
  }
  // activations: kb*32 bytes per row in 16-byte pieces
  const int ap = kb * 2;
  for (int i = tid; i < kNT * ap; i += blockDim.x) {
    const int j = i / ap, c = i % ap;
    const int row = sm.tok[j];
    int4 v = make_int4(0, 0, 0, 0);
    if (row >= 0) v = *reinterpret_cast<const int4*>(act + static_cast<size_t>(row) * act_pitch + kc * 32 + 16 * c);
    *reinterpret_cast<int4*>(&sm.act[j][16 * c]) = v;
  }
  for (int i = tid; i < kNT * kb; i += blockDim.x) {
    const int j = i / kb, c = i % kb;
    const int row = sm.tok[j];
    sm.ad[j][c] = row >= 0 ? f16_bits_to_f32(adsc[static_cast<size_t>(row) * ad_pitch + kc + c]) : 0.0f;
  }
}

__device__ __forceinline__ void load_q8(const int8_t* p, int* q) {
  const int4 q0 = *reinterpret_cast<const int4*>(p);
  const int4 q1 = *reinterpret_cast<const int4*>(p + 16);
  q[0] = q0.x; q[1] = q0.y; q[2] = q0.z; q[3] = q0.w;
  q[4] = q1.x; q[5] = q1.y; q[6] = q1.z; q[7] = q1.w;
}

// Grouped gate/up GEMM over the tiles of groups [g0, g1) with matrices G, U
// (routed: expert = group; shared: expert 0). Tile = 32 rows of I x 64
// grouped rows; epilogue: h = silu(g) u, then H32 + Q8 of the 32-block.
template <int FMT>
__global__ void __launch_bounds__(kGemmThreads) gu_kernel(const PrefillArgs a, int g0, int g1, int shared) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  GemmSmem<FMT>& sm = *reinterpret_cast<GemmSmem<FMT>*>(smem_raw);
  constexpr int BC = block_bytes<FMT>();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const DMat& G = shared ? a.sgate : a.gate;
  const DMat& U = shared ? a.sup : a.up;
  const DMat* mats[2] = {&G, &U};
  const int t_begin = a.tiles_gu[g0], t_end = a.tiles_gu[g1];
  const int rtiles = a.I / kMT;
  const int nb = a.H / 32;
  for (int tile = t_begin + blockIdx.x; tile < t_end; tile += gridDim.x) {
    const int g = tile_group(a.tiles_gu, g0, g1, tile);
    const int local = tile - a.tiles_gu[g];
    const int tt = local / rtiles, rt = local % rtiles;
    const int off = a.offsets[g], n = a.offsets[g + 1] - off;
    const int e = shared ? 0 : g;
    const int i0 = rt * kMT;
    __syncthreads();  // the previous tile's shared memory is free
    if (threadIdx.x < kNT) {
      const int j = tt * kNT + threadIdx.x;
      int row = -1;
      if (j < n) {
        int t, s;
        pid_split(a, a.pid[off + j], t, s);
        row = t;
      }
      sm.tok[threadIdx.x] = row;
    }
    if (threadIdx.x < 8) {
      const DMat& M = threadIdx.x < 4 ? G : U;
      sm.cb[threadIdx.x / 4][threadIdx.x % 4] =
          reinterpret_cast<const uint32_t*>(M.cb + static_cast<size_t>(e) * M.cb_stride)[threadIdx.x % 4];
    }
    __syncthreads();
    float ag[kTokPerWarp], au[kTokPerWarp];
#pragma unroll
    for (int t = 0; t < kTokPerWarp; ++t) ag[t] = au[t] = 0.0f;
    for (int kc = 0; kc < nb; kc += kKB) {
      const int kb = min(kKB, nb - kc);
      stage_chunk<FMT, 2>(sm, mats, e, i0, a.H, kc, kb, a.xq, a.H, a.xd, nb);
      __syncthreads();
      const uint32_t* cbg = sm.cb[0];
      const uint32_t* cbu = sm.cb[1];
#pragma unroll 1
      for (int b = 0; b < kb; ++b) {
        uint32_t vg[8], vu[8];
        block_expand<FMT>(&sm.w[0][lane][b * BC], cbg, vg);
        block_expand<FMT>(&sm.w[1][lane][b * BC], cbu, vu);
        const float wsg = raw_scale<FMT>(sm.ws[0][lane][b]);
        const float wsu = raw_scale<FMT>(sm.ws[1][lane][b]);
#pragma unroll
        for (int t = 0; t < kTokPerWarp; ++t) {
          const int j = warp * kTokPerWarp + t;
          int q[8];
          load_q8(&sm.act[j][32 * b], q);
          const float d = sm.ad[j][b];
          ag[t] = fmaf(wsg * d, static_cast<float>(dot8(vg, q)), ag[t]);
          au[t] = fmaf(wsu * d, static_cast<float>(dot8(vu, q)), au[t]);
        }
      }
      __syncthreads();
    }
    // epilogue: lane = row i0 + lane of I, one 32-block of h per token
#pragma unroll 1
    for (int t = 0; t < kTokPerWarp; ++t) {
      const int j = tt * kNT + warp * kTokPerWarp + t;
      if (j >= n) break;  // warp-uniform
      const float h = ag[t] * au[t] / (1.0f + expf(-ag[t]));
      float v = h;
      if (a.signs_h) v = h32_warp(v, __ldg(&a.signs_h[i0 / 32]), lane);
      uint16_t db;
      const int8_t q = q8_warp(v, db);
      const size_t row = static_cast<size_t>(off + j);
      a.hq[row * a.I + i0 + lane] = q;
      if (lane == 0) a.hd[row * (a.I / 32) + i0 / 32] = db;
      if (a.dbg.h || a.dbg.hq || a.dbg.hd) {
        int tk, s;
        pid_split(a, a.pid[off + j], tk, s);
        const size_t vec = static_cast<size_t>(tk) * a.ns + s;
        if (a.dbg.h) a.dbg.h[vec * a.I + i0 + lane] = h;
        if (a.dbg.hq) a.dbg.hq[vec * a.I + i0 + lane] = q;
        if (a.dbg.hd && lane == 0) a.dbg.hd[vec * (a.I / 32) + i0 / 32] = db;
      }
    }
  }
}

// Grouped down GEMM: o[row, :] = W_down[e] hq[row] over the tiles of groups
// [g0, g1). Tile = 32 rows of H x 64 grouped rows.
template <int FMT>
__global__ void __launch_bounds__(kGemmThreads) down_kernel(const PrefillArgs a, int g0, int g1, int shared) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  GemmSmem<FMT>& sm = *reinterpret_cast<GemmSmem<FMT>*>(smem_raw);
  constexpr int BC = block_bytes<FMT>();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const DMat& D = shared ? a.sdown : a.down;
  const DMat* mats[1] = {&D};
  const int t_begin = a.tiles_dn[g0], t_end = a.tiles_dn[g1];
  const int rtiles = a.H / kMT;
  const int nb = a.I / 32;
  for (int tile = t_begin + blockIdx.x; tile < t_end; tile += gridDim.x) {
    const int g = tile_group(a.tiles_dn, g0, g1, tile);
    const int local = tile - a.tiles_dn[g];
    const int tt = local / rtiles, rt = local % rtiles;
    const int off = a.offsets[g], n = a.offsets[g + 1] - off;
    const int e = shared ? 0 : g;
    const int r0 = rt * kMT;
    __syncthreads();
    if (threadIdx.x < kNT) {
      const int j = tt * kNT + threadIdx.x;
      sm.tok[threadIdx.x] = j < n ? off + j : -1;  // activation rows are grouped rows
    }
    if (threadIdx.x < 4)
      sm.cb[0][threadIdx.x] = reinterpret_cast<const uint32_t*>(D.cb + static_cast<size_t>(e) * D.cb_stride)[threadIdx.x];
    __syncthreads();
    float acc[kTokPerWarp];
#pragma unroll
    for (int t = 0; t < kTokPerWarp; ++t) acc[t] = 0.0f;
    for (int kc = 0; kc < nb; kc += kKB) {
      const int kb = min(kKB, nb - kc);
      stage_chunk<FMT, 1>(sm, mats, e, r0, a.I, kc, kb, a.hq, a.I, a.hd, nb);
      __syncthreads();
#pragma unroll 1
      for (int b = 0; b < kb; ++b) {
        uint32_t v[8];
        block_expand<FMT>(&sm.w[0][lane][b * BC], sm.cb[0], v);
        const float ws = raw_scale<FMT>(sm.ws[0][lane][b]);
#pragma unroll
        for (int t = 0; t < kTokPerWarp; ++t) {
          const int j = warp * kTokPerWarp + t;
          int q[8];
          load_q8(&sm.act[j][32 * b], q);
          acc[t] = fmaf(ws * sm.ad[j][b], static_cast<float>(dot8(v, q)), acc[t]);
        }
      }
      __syncthreads();
    }
#pragma unroll 1
    for (int t = 0; t < kTokPerWarp; ++t) {
      const int j = tt * kNT + warp * kTokPerWarp + t;
      if (j >= n) break;
      const size_t row = static_cast<size_t>(off + j);
      a.o[row * a.H + r0 + lane] = acc[t];
      if (a.dbg.o) {
        int tk, s;
        pid_split(a, a.pid[off + j], tk, s);
        a.dbg.o[(static_cast<size_t>(tk) * a.ns + s) * a.H + r0 + lane] = acc[t];
      }
    }
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

template <int FMT>
int launch_gu(const PrefillArgs& a, int g0, int g1, int shared, int grid, cudaStream_t s) {
  const int smem = static_cast<int>(sizeof(GemmSmem<FMT>));
  if (cudaFuncSetAttribute(gu_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return MOEQ_ERR_CUDA;
  gu_kernel<FMT><<<grid, kGemmThreads, smem, s>>>(a, g0, g1, shared);
  return cuda_status(cudaGetLastError());
}

template <int FMT>
int launch_down(const PrefillArgs& a, int g0, int g1, int shared, int grid, cudaStream_t s) {
  const int smem = static_cast<int>(sizeof(GemmSmem<FMT>));
  if (cudaFuncSetAttribute(down_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return MOEQ_ERR_CUDA;
  down_kernel<FMT><<<grid, kGemmThreads, smem, s>>>(a, g0, g1, shared);
  return cuda_status(cudaGetLastError());
}

int gu_any(int fmt, const PrefillArgs& a, int g0, int g1, int shared, int grid, cudaStream_t s) {
  if (fmt == 2) return launch_gu<2>(a, g0, g1, shared, grid, s);
  if (fmt == 3) return launch_gu<3>(a, g0, g1, shared, grid, s);
  return launch_gu<4>(a, g0, g1, shared, grid, s);
}

int down_any(int fmt, const PrefillArgs& a, int g0, int g1, int shared, int grid, cudaStream_t s) {
  if (fmt == 2) return launch_down<2>(a, g0, g1, shared, grid, s);
  if (fmt == 3) return launch_down<3>(a, g0, g1, shared, grid, s);
  return launch_down<4>(a, g0, g1, shared, grid, s);
}

}  // namespace
}  // namespace moeq

using namespace moeq;

extern "C" int moe_ffn_prefill(const moeq_layer* L, const uint16_t* x, int T, const float* residual,
                               float* y, void* ws, size_t ws_bytes, int32_t* dev_status,
                               const moeq_debug* dbg, moeq_stream stream) {
  int rc = validate_layer(L);
  if (rc) return rc;
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
  a.hq = reinterpret_cast<int8_t*>(w + wl.hq);
  a.hd = reinterpret_cast<uint16_t*>(w + wl.hd);
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
  const int grid = device_info().sm_count * 3;
  if ((rc = gu_any(L->gate.fmt, a, 0, L->E, 0, grid, s))) return rc;
  if (a.has_shared && (rc = gu_any(L->sgate.fmt, a, L->E, L->E + 1, 1, grid, s))) return rc;
  if ((rc = down_any(L->down.fmt, a, 0, L->E, 0, grid, s))) return rc;
  if (a.has_shared && (rc = down_any(L->sdown.fmt, a, L->E, L->E + 1, 1, grid, s))) return rc;
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
