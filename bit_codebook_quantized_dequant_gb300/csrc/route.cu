// Router + top-k for T tokens, the H32 rotation and the RMSNorm of the layer
// stack.
//
// Router ("DeepSeek V4 Flash: 284B model, up to 32 tok/s on AMD Ryzen AI MAX+
// 395", section "Decode: up to 32 tok/s": routing with dedicated TOP_K
// kernels): a CTA takes 8 tokens; their bf16 rows sit in shared memory and each
// warp streams 4 router rows at a time from global memory (16-byte loads, lane j
// reading elements 256 i + 8 j .. +7), accumulating each of the 8 tokens' dot
// products in fp32 in that order, then the combining rounds 16, 8, 4, 2, 1. The logits stay in
// shared memory and one warp per token selects the top k.
#include <cuda_runtime.h>

#include "moeq.h"
#include "moeq_device.cuh"
#include "moeq_host.h"
#include "moeq_layout.h"

namespace moeq {
namespace {

constexpr int kRtTokens = 8;
constexpr int kRtWarps = 16;
constexpr int kRtExp = 4;  // router rows per warp pass

// Top-k + softmax weights of one token by one warp from E logits in memory `l`.
template <int NPL>
__device__ void token_topk(const float* l, int E, int k, int lane, int32_t* idx_out, float* w_out) {
  float v[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? l[e] : 0.0f;
  }
  int idx;
  float p;
  warp_topk<NPL>(v, E, k, lane, idx, p);
  if (lane < k) {
    idx_out[lane] = idx;
    w_out[lane] = p;
  }
}

__device__ void warp_topk_any(const float* l, int E, int k, int lane, int32_t* idx_out, float* w_out) {
  if (E <= 256) token_topk<8>(l, E, k, lane, idx_out, w_out);
  else if (E <= 512) token_topk<16>(l, E, k, lane, idx_out, w_out);
  else token_topk<32>(l, E, k, lane, idx_out, w_out);
}

__global__ void __launch_bounds__(kRtWarps * 32) route_kernel(
    const uint16_t* __restrict__ x, int T, const uint16_t* __restrict__ router, int E, int H,
    int k, int32_t* __restrict__ idx, float* __restrict__ w, float* __restrict__ logits_out) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem_raw);                           // [8][H]
  float* ls = reinterpret_cast<float*>(smem_raw + static_cast<size_t>(kRtTokens) * H * 2);  // [8][E]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * kRtTokens;
  const int nt = min(kRtTokens, T - t0);
  const int vec_per_row = H / 8;
  for (int i = tid; i < kRtTokens * vec_per_row; i += blockDim.x) {
    const int tt = i / vec_per_row, c = i % vec_per_row;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (tt < nt) v = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(t0 + tt) * H) + c);
    reinterpret_cast<uint4*>(xs + static_cast<size_t>(tt) * H)[c] = v;
  }
  __syncthreads();
  // a warp takes kRtExp router rows at a time, so that each activation read
  // from shared memory feeds kRtExp dot products (rows past E read as zero and
  // are not stored)
  for (int e0 = warp * kRtExp; e0 < E; e0 += kRtWarps * kRtExp) {
    float acc[kRtExp][kRtTokens];
#pragma unroll
    for (int j = 0; j < kRtExp; ++j)
#pragma unroll
      for (int tt = 0; tt < kRtTokens; ++tt) acc[j][tt] = 0.0f;
    for (int i = 0; i < H / 256; ++i) {
      const int k0 = 256 * i + 8 * lane;
      uint4 wv[kRtExp];
#pragma unroll
      for (int j = 0; j < kRtExp; ++j)
        wv[j] = e0 + j < E ? __ldg(reinterpret_cast<const uint4*>(router + static_cast<size_t>(e0 + j) * H + k0))
                           : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int tt = 0; tt < kRtTokens; ++tt) {
        const uint4 xv = *reinterpret_cast<const uint4*>(xs + static_cast<size_t>(tt) * H + k0);
#pragma unroll
        for (int j = 0; j < kRtExp; ++j) {
          float a = acc[j][tt];
          a = fmaf(bf16_lo(xv.x), bf16_lo(wv[j].x), a);
          a = fmaf(bf16_hi(xv.x), bf16_hi(wv[j].x), a);
          a = fmaf(bf16_lo(xv.y), bf16_lo(wv[j].y), a);
          a = fmaf(bf16_hi(xv.y), bf16_hi(wv[j].y), a);
          a = fmaf(bf16_lo(xv.z), bf16_lo(wv[j].z), a);
          a = fmaf(bf16_hi(xv.z), bf16_hi(wv[j].z), a);
          a = fmaf(bf16_lo(xv.w), bf16_lo(wv[j].w), a);
          a = fmaf(bf16_hi(xv.w), bf16_hi(wv[j].w), a);
          acc[j][tt] = a;
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kRtExp; ++j)
#pragma unroll
      for (int tt = 0; tt < kRtTokens; ++tt) {
        const float l = warp_sum_canonical(acc[j][tt]);
        if (lane == 0 && e0 + j < E) {
          ls[tt * E + e0 + j] = l;
          if (logits_out && tt < nt) logits_out[static_cast<size_t>(t0 + tt) * E + e0 + j] = l;
        }
      }
  }
  __syncthreads();
  if (warp < nt)
    warp_topk_any(ls + warp * E, E, k, lane, idx + static_cast<size_t>(t0 + warp) * k,
                  w + static_cast<size_t>(t0 + warp) * k);
}

__global__ void h32_kernel(const float* __restrict__ in, float* out, int nblk,
                           const uint32_t* __restrict__ signs) {
  const int b = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= nblk) return;
  const float v = in[static_cast<size_t>(b) * 32 + lane];
  out[static_cast<size_t>(b) * 32 + lane] = h32_warp(v, signs ? signs[b] : 0u, lane);
}

// RMSNorm of one row by one warp: sum of squares in the canonical order,
// correctly rounded fp32 steps, then a = bf16_rne(r * inv).
// 1 / sqrt(mean(row^2) + 1e-6) of one row by one warp: the sum of squares in
// the router's canonical order (lane j over h = 256 i + 8 j + t, each square
// rounded, then the combining rounds), each step correctly rounded.
__device__ __forceinline__ float rms_inv(const float* row, int H, int lane) {
  float s = 0.0f;
  for (int i = 0; i < H / 256; ++i) {
    const float4 v0 = *reinterpret_cast<const float4*>(row + 256 * i + 8 * lane);
    const float4 v1 = *reinterpret_cast<const float4*>(row + 256 * i + 8 * lane + 4);
    s = __fadd_rn(s, __fmul_rn(v0.x, v0.x));
    s = __fadd_rn(s, __fmul_rn(v0.y, v0.y));
    s = __fadd_rn(s, __fmul_rn(v0.z, v0.z));
    s = __fadd_rn(s, __fmul_rn(v0.w, v0.w));
    s = __fadd_rn(s, __fmul_rn(v1.x, v1.x));
    s = __fadd_rn(s, __fmul_rn(v1.y, v1.y));
    s = __fadd_rn(s, __fmul_rn(v1.z, v1.z));
    s = __fadd_rn(s, __fmul_rn(v1.w, v1.w));
  }
  s = warp_sum_canonical(s);
  const float ms = __fdiv_rn(s, static_cast<float>(H));
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, 1e-6f)));
}

__device__ __forceinline__ void rmsnorm_row(const float* row, int H, uint16_t* out, int lane) {
  const float inv = rms_inv(row, H, lane);
  for (int k0 = 8 * lane; k0 < H; k0 += 256) {
    const float4 v0 = *reinterpret_cast<const float4*>(row + k0);
    const float4 v1 = *reinterpret_cast<const float4*>(row + k0 + 4);
    uint4 o;
    o.x = f32_to_bf16_rne(__fmul_rn(v0.x, inv)) | (static_cast<uint32_t>(f32_to_bf16_rne(__fmul_rn(v0.y, inv))) << 16);
    o.y = f32_to_bf16_rne(__fmul_rn(v0.z, inv)) | (static_cast<uint32_t>(f32_to_bf16_rne(__fmul_rn(v0.w, inv))) << 16);
    o.z = f32_to_bf16_rne(__fmul_rn(v1.x, inv)) | (static_cast<uint32_t>(f32_to_bf16_rne(__fmul_rn(v1.y, inv))) << 16);
    o.w = f32_to_bf16_rne(__fmul_rn(v1.z, inv)) | (static_cast<uint32_t>(f32_to_bf16_rne(__fmul_rn(v1.w, inv))) << 16);
    *reinterpret_cast<uint4*>(out + k0) = o;
  }
}

__global__ void rmsnorm_kernel(const float* __restrict__ r, int T, int H, uint16_t* __restrict__ a) {
  const int t = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  rmsnorm_row(r + static_cast<size_t>(t) * H, H, a + static_cast<size_t>(t) * H, lane);
}

// One step of a decode stack, one CTA per row of the residual stream: r =
// float(x) when x is given, else r = r + y when y is given (correctly rounded
// fp32 adds), by every thread with all loads in flight; then, when a is given,
// a = RMSNorm(r) with rmsnorm_row's arithmetic (its sum of squares by warp 0 in
// the canonical order, from a shared-memory copy of the row), so a equals
// moe_rmsnorm_bf16 of r bit for bit.
constexpr int kStepThreads = 512;

__global__ void __launch_bounds__(kStepThreads) stack_step_kernel(const uint16_t* __restrict__ x,
                                                                   const float* __restrict__ y,
                                                                   float* __restrict__ r, uint16_t* __restrict__ a,
                                                                   int H) {
  extern __shared__ __align__(16) float rs[];  // the row after the step [H]
  __shared__ float inv_s;
  const size_t off = static_cast<size_t>(blockIdx.x) * H;
  r += off;
  if (x) x += off;
  if (y) y += off;
  for (int k = threadIdx.x; k < H; k += blockDim.x) {
    float v;
    if (x) v = __uint_as_float(static_cast<uint32_t>(x[k]) << 16);
    else if (y) v = __fadd_rn(r[k], y[k]);
    else v = r[k];
    if (x || y) r[k] = v;
    rs[k] = v;
  }
  __syncthreads();
  if (!a) return;
  if (threadIdx.x < 32) {
    const float inv = rms_inv(rs, H, threadIdx.x);
    if (threadIdx.x == 0) inv_s = inv;
  }
  __syncthreads();
  const float inv = inv_s;
  a += off;
  for (int k = threadIdx.x; k < H; k += blockDim.x) a[k] = f32_to_bf16_rne(__fmul_rn(rs[k], inv));
}

}  // namespace

// Enqueues router + top-k (used by moe_route_topk and by the prefill).
int route_topk_launch(const uint16_t* x, int T, const uint16_t* router, int E, int H, int k,
                      int32_t* idx, float* w, float* logits, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(kRtTokens) * H * 2 + static_cast<size_t>(kRtTokens) * E * 4;
  const DeviceInfo& di = device_info();
  if (smem > di.max_smem_optin) return MOEQ_ERR_SHAPE;
  if (cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MOEQ_ERR_CUDA;
  const int grid = (T + kRtTokens - 1) / kRtTokens;
  route_kernel<<<grid, kRtWarps * 32, smem, s>>>(x, T, router, E, H, k, idx, w, logits);
  return cuda_status(cudaGetLastError());
}

}  // namespace moeq

using namespace moeq;

extern "C" int moe_route_topk(const uint16_t* x, int T, const uint16_t* router, int E, int H, int k,
                              int32_t* idx, float* w, float* logits_opt, int32_t* dev_status,
                              moeq_stream stream) {
  (void)dev_status;
  if (T < 0 || E < 1 || E > 1024 || H < 256 || H % 256) return MOEQ_ERR_SHAPE;
  if (k < 1 || k > kMaxTopK || k > E) return MOEQ_ERR_ARG;
  if (T == 0) return MOEQ_OK;
  if (!x || !router || !idx || !w) return MOEQ_ERR_ARG;
  if (!aligned16(x) || !aligned16(router)) return MOEQ_ERR_ALIGN;
  return route_topk_launch(x, T, router, E, H, k, idx, w, logits_opt,
                           reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int h32_rotate(const float* in, float* out, int nblk, const uint32_t* signs,
                          moeq_stream stream) {
  if (nblk < 0) return MOEQ_ERR_SHAPE;
  if (nblk == 0) return MOEQ_OK;
  if (!in || !out) return MOEQ_ERR_ARG;
  const int per = 8;  // blocks per CTA
  h32_kernel<<<(nblk + per - 1) / per, per * 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      in, out, nblk, signs);
  return cuda_status(cudaGetLastError());
}

// Enqueues one stack step over `rows` rows (see stack_step_kernel).
int moeq::stack_step_launch(const uint16_t* x, const float* y, float* r, uint16_t* a, int H, int rows,
                            cudaStream_t s) {
  stack_step_kernel<<<rows, kStepThreads, static_cast<size_t>(H) * 4, s>>>(x, y, r, a, H);
  return cuda_status(cudaGetLastError());
}

extern "C" int moe_rmsnorm_bf16(const float* r, int T, int H, uint16_t* a, moeq_stream stream) {
  if (T < 0 || H < 256 || H % 256) return MOEQ_ERR_SHAPE;
  if (T == 0) return MOEQ_OK;
  if (!r || !a) return MOEQ_ERR_ARG;
  if (!aligned16(r) || !aligned16(a)) return MOEQ_ERR_ALIGN;
  const int per = 8;
  rmsnorm_kernel<<<(T + per - 1) / per, per * 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(r, T, H, a);
  return cuda_status(cudaGetLastError());
}
