// The "generic expand-then-multiply fallback" of "Lucebox x Geometric ...",
// section "Lucebox Engine integration with Geometric" (the fused 3.5-bit
// matvec is reported 2.2x faster than it), rebuilt on GB300 as an ablation of
// the fused decode:
//   moe_expand_bf16          packed experts -> bf16 weights in HBM,
//                            w = bf16_rne(codebook[code] * block scale)
//   moe_ffn_decode_expanded  batch-1 decode over those bf16 weights: the same
//                            router and top-k, then bf16 x fp32 GEMVs with
//                            unquantized activations (x as given, h in fp32)
// Neither is on the fused path; they exist to measure it against the plain
// alternative on the same GPU.
#include <cuda_runtime.h>

#include "moeq.h"
#include "moeq_device.cuh"
#include "moeq_host.h"
#include "moeq_layout.h"

namespace moeq {
namespace {

constexpr int kGemvWarps = 16;
constexpr int kGemvThreads = kGemvWarps * 32;

// One thread per 32-block: 32 codes -> 32 bf16 weights (64 bytes, row-major).
template <int FMT>
__global__ void expand_kernel(DMat m, int e0, int ne, uint16_t* __restrict__ out) {
  constexpr int BC = block_bytes<FMT>();
  const int nb = m.cols / 32;
  const size_t per_e = static_cast<size_t>(m.rows) * nb;
  const size_t n = per_e * ne;
  for (size_t b = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; b < n;
       b += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int e = e0 + static_cast<int>(b / per_e);
    const size_t i = b % per_e;  // block index within the expert (row-major)
    const uint4 rec = __ldg(reinterpret_cast<const uint4*>(m.cb + static_cast<size_t>(e) * m.cb_stride));
    const uint32_t cb[4] = {rec.x, rec.y, rec.z, rec.w};
    uint32_t v[8];
    block_expand<FMT>(m.codes + e * m.stride_codes + i * BC, cb, v);
    const float s = block_scale<FMT>(m.scales + e * m.stride_scales, static_cast<int>(i));
    uint32_t o[16];
#pragma unroll
    for (int w = 0; w < 8; ++w)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float a = __fmul_rn(static_cast<float>(static_cast<int8_t>(v[w] >> (16 * h))), s);
        const float c = __fmul_rn(static_cast<float>(static_cast<int8_t>(v[w] >> (16 * h + 8))), s);
        o[2 * w + h] = f32_to_bf16_rne(a) | (static_cast<uint32_t>(f32_to_bf16_rne(c)) << 16);
      }
    uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<size_t>(e - e0) * per_e + i) * 32);
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
  }
}

struct XArgs {
  int H, I, k, has_shared;
  const uint16_t* x;
  const uint16_t *gate, *up, *down, *sgate, *sup, *sdown;  // bf16 rows
  size_t sg, su, sd;                                      // elements between experts
  const int32_t* idx;
  const float* p;
  float* h;  // [(k + shared) x I]
  float* y;
};

// Router logits of one token, one warp per expert row in the canonical order
// (lane j sums k = 256 i + 8 j + t over i, t with exact bf16 products, then
// the combining rounds 16 .. 1), spread over the grid; the last CTA to arrive
// takes the top-k and the softmax weights with one warp and returns the
// arrival counter to zero for the next call.
constexpr int kRouteWarps = 8;

template <int NPL>
__device__ __forceinline__ void last_cta_topk(const float* logits, int E, int k, int lane, int32_t* idx, float* p) {
  float v[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? __ldcg(logits + e) : 0.0f;
  }
  int id;
  float w;
  warp_topk<NPL>(v, E, k, lane, id, w);
  if (lane < k) {
    idx[lane] = id;
    p[lane] = w;
  }
}

__global__ void __launch_bounds__(kRouteWarps * 32) xroute_kernel(const uint16_t* __restrict__ x,
                                                                   const uint16_t* __restrict__ router, int E, int H,
                                                                   int k, float* logits, uint32_t* arrive,
                                                                   int32_t* idx, float* p) {
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
  if (e < E) {
    const uint16_t* wrow = router + static_cast<size_t>(e) * H;
    float acc = 0.0f;
    for (int i = 0; i < H / 256; ++i) {
      const int k0 = 256 * i + 8 * lane;
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(wrow + k0));
      const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + k0));
      acc = fmaf(bf16_lo(xv.x), bf16_lo(w.x), acc);
      acc = fmaf(bf16_hi(xv.x), bf16_hi(w.x), acc);
      acc = fmaf(bf16_lo(xv.y), bf16_lo(w.y), acc);
      acc = fmaf(bf16_hi(xv.y), bf16_hi(w.y), acc);
      acc = fmaf(bf16_lo(xv.z), bf16_lo(w.z), acc);
      acc = fmaf(bf16_hi(xv.z), bf16_hi(w.z), acc);
      acc = fmaf(bf16_lo(xv.w), bf16_lo(w.w), acc);
      acc = fmaf(bf16_hi(xv.w), bf16_hi(w.w), acc);
    }
    acc = warp_sum_canonical(acc);
    if (lane == 0) {
      logits[e] = acc;
      __threadfence();  // the logit is visible device-wide before this CTA arrives
    }
  }
  __shared__ uint32_t last;
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(arrive, 1u) == gridDim.x - 1 ? 1u : 0u;
  __syncthreads();
  if (!last) return;
  __threadfence();  // every CTA's logits after seeing the last arrival
  if (threadIdx.x < 32) {
    if (E <= 256) last_cta_topk<8>(logits, E, k, lane, idx, p);
    else if (E <= 512) last_cta_topk<16>(logits, E, k, lane, idx, p);
    else last_cta_topk<32>(logits, E, k, lane, idx, p);
    if (lane == 0) *arrive = 0u;
  }
}

__device__ __forceinline__ float bf16x8_dot(const uint4 w, const float* v, float acc) {
  const float4 a = *reinterpret_cast<const float4*>(v);
  const float4 b = *reinterpret_cast<const float4*>(v + 4);
  acc = fmaf(bf16_lo(w.x), a.x, acc);
  acc = fmaf(bf16_hi(w.x), a.y, acc);
  acc = fmaf(bf16_lo(w.y), a.z, acc);
  acc = fmaf(bf16_hi(w.y), a.w, acc);
  acc = fmaf(bf16_lo(w.z), b.x, acc);
  acc = fmaf(bf16_hi(w.z), b.y, acc);
  acc = fmaf(bf16_lo(w.w), b.z, acc);
  acc = fmaf(bf16_hi(w.w), b.w, acc);
  return acc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

// Gate/up rows of every slot: one warp per (slot, row), the gate and up rows
// streamed together; h = silu(g) * u.
__global__ void __launch_bounds__(kGemvThreads) xgu_kernel(const XArgs a) {
  extern __shared__ __align__(16) float xs[];  // x as fp32 [H]
  for (int i = threadIdx.x; i < a.H; i += blockDim.x) xs[i] = __uint_as_float(static_cast<uint32_t>(a.x[i]) << 16);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int ns = a.k + a.has_shared;
  const int nrows = ns * a.I;
  for (int w = blockIdx.x * kGemvWarps + (threadIdx.x >> 5); w < nrows; w += gridDim.x * kGemvWarps) {
    const int s = w / a.I, r = w % a.I;
    const bool shared = s == a.k;
    const size_t e = shared ? 0 : static_cast<size_t>(a.idx[s]);
    const uint16_t* gr = (shared ? a.sgate : a.gate) + e * a.sg + static_cast<size_t>(r) * a.H;
    const uint16_t* ur = (shared ? a.sup : a.up) + e * a.su + static_cast<size_t>(r) * a.H;
    float g = 0.0f, u = 0.0f;
#pragma unroll 4
    for (int k0 = 8 * lane; k0 < a.H; k0 += 256) {
      const uint4 wg = __ldg(reinterpret_cast<const uint4*>(gr + k0));
      const uint4 wu = __ldg(reinterpret_cast<const uint4*>(ur + k0));
      g = bf16x8_dot(wg, xs + k0, g);
      u = bf16x8_dot(wu, xs + k0, u);
    }
    g = warp_sum(g);
    u = warp_sum(u);
    if (lane == 0) a.h[static_cast<size_t>(s) * a.I + r] = g * u / (1.0f + expf(-g));
  }
}

// Down rows and the combine: one warp per output row, every slot's row
// streamed together; lane partials p_s * (w_s . h_s) summed per lane in slot
// order, then across the lanes: y = sum_s p_s o_s + o_shared.
__global__ void __launch_bounds__(kGemvThreads) xdown_kernel(const XArgs a) {
  extern __shared__ __align__(16) float hs[];  // h of every slot [(k + shared) x I]
  const int ns = a.k + a.has_shared;
  for (int i = threadIdx.x; i < ns * a.I; i += blockDim.x) hs[i] = __ldcg(a.h + i);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  for (int r = blockIdx.x * kGemvWarps + (threadIdx.x >> 5); r < a.H; r += gridDim.x * kGemvWarps) {
    float part[kMaxTopK + 1];
#pragma unroll
    for (int s = 0; s <= kMaxTopK; ++s) part[s] = 0.0f;
    for (int k0 = 8 * lane; k0 < a.I; k0 += 256) {
#pragma unroll
      for (int s = 0; s <= kMaxTopK; ++s) {
        if (s < ns) {
          const bool shared = s == a.k;
          const uint16_t* row = shared ? a.sdown + static_cast<size_t>(r) * a.I
                                       : a.down + static_cast<size_t>(a.idx[s]) * a.sd + static_cast<size_t>(r) * a.I;
          part[s] = bf16x8_dot(__ldg(reinterpret_cast<const uint4*>(row + k0)), hs + static_cast<size_t>(s) * a.I + k0,
                               part[s]);
        }
      }
    }
    float acc = 0.0f;
#pragma unroll
    for (int s = 0; s <= kMaxTopK; ++s)
      if (s < ns) acc = s == a.k ? acc + part[s] : fmaf(a.p[s], part[s], acc);
    acc = warp_sum(acc);
    if (lane == 0) a.y[r] = acc;
  }
}

int check_bf16_matrix(const moeq_matrix& m, int rows, int cols, int experts) {
  if (m.fmt != MOEQ_BF16) return MOEQ_ERR_FORMAT;
  if (m.rows != rows || m.cols != cols || m.num_experts != experts) return MOEQ_ERR_SHAPE;
  if (!m.codes) return MOEQ_ERR_ARG;
  if (!aligned16(m.codes)) return MOEQ_ERR_ALIGN;
  const unsigned long long need = 2ull * rows * cols;
  if (experts > 1 && (m.expert_stride_codes < need || m.expert_stride_codes % 16)) return MOEQ_ERR_SHAPE;
  return MOEQ_OK;
}

}  // namespace
}  // namespace moeq

using namespace moeq;

extern "C" int moe_expand_bf16(const moeq_matrix* m, int e0, int ne, uint16_t* out_bf16, moeq_stream stream) {
  if (!m || !out_bf16) return MOEQ_ERR_ARG;
  int rc = validate_matrix(*m, m->rows, m->cols, m->num_experts);
  if (rc) return rc;
  if (e0 < 0 || ne < 0 || e0 + ne > m->num_experts) return MOEQ_ERR_ARG;
  if (!aligned16(out_bf16)) return MOEQ_ERR_ALIGN;
  if (ne == 0) return MOEQ_OK;
  const DMat d = to_dmat(*m);
  const DeviceInfo& di = device_info();
  const int grid = 8 * (di.sm_count > 0 ? di.sm_count : 1);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (d.fmt == 2)
    expand_kernel<2><<<grid, 256, 0, s>>>(d, e0, ne, out_bf16);
  else if (d.fmt == 3)
    expand_kernel<3><<<grid, 256, 0, s>>>(d, e0, ne, out_bf16);
  else if (d.fmt == MOEQ_FP3_PACKED24)
    expand_kernel<MOEQ_FP3_PACKED24><<<grid, 256, 0, s>>>(d, e0, ne, out_bf16);
  else
    expand_kernel<4><<<grid, 256, 0, s>>>(d, e0, ne, out_bf16);
  return cuda_status(cudaGetLastError());
}

// Workspace: idx [k], p [k], the arrival counter, logits [E], h [(k + shared) x I].
extern "C" size_t moe_ffn_expanded_workspace(int H, int I, int E, int k, int has_shared) {
  if (H <= 0 || I <= 0 || E < 1 || E > 1024 || k < 1 || k > kMaxTopK || k > E) return 0;
  (void)H;
  return align256(4 * static_cast<size_t>(kMaxTopK)) * 3 + align256(4 * static_cast<size_t>(E)) +
         align256(4 * static_cast<size_t>(k + (has_shared ? 1 : 0)) * I);
}

extern "C" int moe_ffn_decode_expanded(const moeq_layer* L, const uint16_t* x, float* y, void* ws,
                                       size_t ws_bytes, int32_t* dev_status, moeq_stream stream) {
  (void)dev_status;
  if (!L || !x || !y) return MOEQ_ERR_ARG;
  const int H = L->H, I = L->I, E = L->E, k = L->k;
  if (H <= 0 || I <= 0 || E <= 0 || H % 256 || I % 128 || E > 1024) return MOEQ_ERR_SHAPE;
  if (k < 1 || k > kMaxTopK || k > E) return MOEQ_ERR_ARG;
  if (L->h32_signs_x || L->h32_signs_h) return MOEQ_ERR_FORMAT;  // no rotation on this path
  if (!L->router) return MOEQ_ERR_ARG;
  if (!aligned16(L->router) || !aligned16(x) || !aligned16(y)) return MOEQ_ERR_ALIGN;
  int rc;
  if ((rc = check_bf16_matrix(L->gate, I, H, E)) || (rc = check_bf16_matrix(L->up, I, H, E)) ||
      (rc = check_bf16_matrix(L->down, H, I, E)))
    return rc;
  if (L->has_shared && ((rc = check_bf16_matrix(L->sgate, I, H, 1)) || (rc = check_bf16_matrix(L->sup, I, H, 1)) ||
                        (rc = check_bf16_matrix(L->sdown, H, I, 1))))
    return rc;
  const size_t need = moe_ffn_expanded_workspace(H, I, E, k, L->has_shared);
  if (!ws || !aligned16(ws) || ws_bytes < need) return MOEQ_ERR_WORKSPACE;
  const int ns = k + (L->has_shared ? 1 : 0);
  const size_t hsmem = 4 * static_cast<size_t>(ns) * I;
  const DeviceInfo& di = device_info();
  if (hsmem > di.max_smem_optin || 4 * static_cast<size_t>(H) > di.max_smem_optin) return MOEQ_ERR_SHAPE;
  uint8_t* w = static_cast<uint8_t*>(ws);
  XArgs a{};
  a.H = H; a.I = I; a.k = k; a.has_shared = L->has_shared ? 1 : 0;
  a.x = x;
  a.gate = static_cast<const uint16_t*>(L->gate.codes);
  a.up = static_cast<const uint16_t*>(L->up.codes);
  a.down = static_cast<const uint16_t*>(L->down.codes);
  a.sg = L->gate.expert_stride_codes / 2;
  a.su = L->up.expert_stride_codes / 2;
  a.sd = L->down.expert_stride_codes / 2;
  if (a.has_shared) {
    a.sgate = static_cast<const uint16_t*>(L->sgate.codes);
    a.sup = static_cast<const uint16_t*>(L->sup.codes);
    a.sdown = static_cast<const uint16_t*>(L->sdown.codes);
  }
  const size_t rec = align256(4 * static_cast<size_t>(kMaxTopK));
  int32_t* idx = reinterpret_cast<int32_t*>(w);
  float* p = reinterpret_cast<float*>(w + rec);
  uint32_t* arrive = reinterpret_cast<uint32_t*>(w + 2 * rec);
  float* logits = reinterpret_cast<float*>(w + 3 * rec);
  a.idx = idx;
  a.p = p;
  a.h = reinterpret_cast<float*>(w + 3 * rec + align256(4 * static_cast<size_t>(E)));
  a.y = y;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  xroute_kernel<<<(E + kRouteWarps - 1) / kRouteWarps, kRouteWarps * 32, 0, s>>>(x, L->router, E, H, k, logits,
                                                                                 arrive, idx, p);
  if ((rc = cuda_status(cudaGetLastError()))) return rc;
  static thread_local int configured_dev = -1;
  if (configured_dev != di.device) {
    const int lim = static_cast<int>(di.max_smem_optin);
    if (cudaFuncSetAttribute(xdown_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, lim) != cudaSuccess ||
        cudaFuncSetAttribute(xgu_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, lim) != cudaSuccess)
      return MOEQ_ERR_CUDA;
    configured_dev = di.device;
  }
  const int sms = di.sm_count > 0 ? di.sm_count : 1;
  xgu_kernel<<<4 * sms, kGemvThreads, 4 * static_cast<size_t>(H), s>>>(a);
  if ((rc = cuda_status(cudaGetLastError()))) return rc;
  xdown_kernel<<<2 * sms, kGemvThreads, hsmem, s>>>(a);
  return cuda_status(cudaGetLastError());
}
