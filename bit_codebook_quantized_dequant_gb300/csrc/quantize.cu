// moe_quantize_expert: codebook quantization of one expert matrix (fp32
// weights -> per-32-block scales, a per-expert int8 codebook of 2^fmt sorted
// entries, and one code per weight), the mechanics behind the "learned
// per-expert codebooks" of "Lucebox x Geometric ...", section "How the model
// fits on AMD Strix Halo". How the pages learn their codebooks is not printed;
// the procedure here is the library's reading, deterministic and exact in its
// integer steps (see include/moeq.h):
//   scales   FP2/FP3 d = fp16(max|w| / 127); FP4 d = 2^e, the smallest e with
//            127 * 2^e >= max|w| (E8M0, e in [-127, 127])
//   grid     v = w / d (fp32), g = clamp(rint(v), -127, 127), histogram of g
//   codebook mid-quantile start, 8 Lloyd steps on the histogram in integers
//   codes    the entry nearest to v in fp32, ties to the lower index
// Three kernels: scales + histogram (one warp per 32-block), the codebook
// (one CTA over the 255 histogram bins), codes (one thread per weight).
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "moeq.h"
#include "moeq_device.cuh"
#include "moeq_host.h"

namespace moeq {
namespace {

constexpr int kBins = 255;  // g = -127 .. 127
constexpr int kLloydSteps = 8;

// Block scale of one 32-block held by a warp (lane j: weight j); returns the
// fp32 value of d and, on lane 0, stores its encoding.
__device__ __forceinline__ float warp_block_scale(int fmt, float x, void* scales, size_t i, int lane) {
  float m = fabsf(x);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (fmt == 4) {
    int e = -127;
    if (m > 0.0f) {
      int ex;
      frexpf(m, &ex);                       // m in [2^(ex-1), 2^ex)
      e = max(-127, ex - 8);                // 127 * 2^(ex-8) < 2^(ex-1) <= m
      while (e < 127 && ldexpf(127.0f, e) < m) ++e;
    }
    if (lane == 0) static_cast<uint8_t*>(scales)[i] = static_cast<uint8_t>(e + 127);
    return ldexpf(1.0f, e);
  }
  __half dh = __float2half_rn(__fdiv_rn(m, 127.0f));
  uint16_t bits = __half_as_ushort(dh);
  if ((bits & 0x7C00u) == 0x7C00u) bits = 0x7BFFu;  // overflow: the largest finite fp16
  if (lane == 0) static_cast<uint16_t*>(scales)[i] = bits;
  return __half2float(__ushort_as_half(bits));
}

__global__ void scale_hist_kernel(int fmt, int rows, int cols, const float* __restrict__ w, void* scales,
                                  uint32_t* __restrict__ hist) {
  __shared__ uint32_t h[kBins];
  for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const size_t nblk = static_cast<size_t>(rows) * (cols / 32);
  const size_t warps = static_cast<size_t>(gridDim.x) * (blockDim.x / 32);
  for (size_t b = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); b < nblk; b += warps) {
    const float x = w[32 * b + lane];
    const float d = warp_block_scale(fmt, x, scales, b, lane);
    const float v = d == 0.0f ? 0.0f : __fdiv_rn(x, d);
    const float g = fminf(fmaxf(rintf(v), -127.0f), 127.0f);
    atomicAdd(&h[static_cast<int>(g) + 127], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kBins; i += blockDim.x)
    if (h[i]) atomicAdd(&hist[i], h[i]);
}

__device__ __forceinline__ long long floor_div64(long long a, long long b) {  // b > 0
  long long q = a / b;
  if ((a % b) != 0 && a < 0) q -= 1;
  return q;
}

// The codebook from the histogram, one CTA of 256 threads (thread t: bin t).
__global__ void codebook_kernel(int K, long long N, const uint32_t* __restrict__ hist, int8_t* __restrict__ cb) {
  __shared__ long long c[16], S[16], n[16];
  const int t = threadIdx.x;
  const long long cnt = t < kBins ? static_cast<long long>(hist[t]) : 0;
  if (t == 0) {
    // entry i: the smallest g whose cumulative count exceeds floor((2i+1) N / 2K)
    for (int i = 0; i < K; ++i) {
      const long long target = ((2LL * i + 1) * N) / (2LL * K);
      long long cum = 0;
      int g = 0;
      for (; g < kBins; ++g) {
        cum += hist[g];
        if (cum > target) break;
      }
      c[i] = g - 127;
    }
  }
  __syncthreads();
  for (int it = 0; it < kLloydSteps; ++it) {
    if (t < K) S[t] = n[t] = 0;
    __syncthreads();
    if (cnt) {
      const long long x = t - 127;
      int best = 0;
      long long bd = llabs(x - c[0]);
      for (int i = 1; i < K; ++i) {
        const long long dd = llabs(x - c[i]);
        if (dd < bd) {
          bd = dd;
          best = i;
        }
      }
      atomicAdd(reinterpret_cast<unsigned long long*>(&S[best]), static_cast<unsigned long long>(cnt * x));
      atomicAdd(reinterpret_cast<unsigned long long*>(&n[best]), static_cast<unsigned long long>(cnt));
    }
    __syncthreads();
    if (t < K && n[t]) c[t] = floor_div64(2 * S[t] + n[t], 2 * n[t]);
    __syncthreads();
    if (t == 0)
      for (int i = 1; i < K; ++i)  // ascending (a stable insertion sort)
        for (int j = i; j > 0 && c[j - 1] > c[j]; --j) {
          const long long tmp = c[j];
          c[j] = c[j - 1];
          c[j - 1] = tmp;
        }
    __syncthreads();
  }
  if (t < K) cb[t] = static_cast<int8_t>(c[t]);
}

__global__ void codes_kernel(int fmt, int rows, int cols, const float* __restrict__ w, const void* scales,
                             const int8_t* __restrict__ cb, uint8_t* __restrict__ codes) {
  __shared__ float c[16];
  const int K = 1 << fmt;
  if (threadIdx.x < K) c[threadIdx.x] = static_cast<float>(cb[threadIdx.x]);
  __syncthreads();
  const size_t n = static_cast<size_t>(rows) * cols;
  for (size_t o = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; o < n;
       o += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t b = o / 32;
    const float d = fmt == 4 ? e8m0_to_f32(static_cast<const uint8_t*>(scales)[b])
                             : __half2float(__ushort_as_half(static_cast<const uint16_t*>(scales)[b]));
    const float v = d == 0.0f ? 0.0f : __fdiv_rn(w[o], d);
    int best = 0;
    float bd = fabsf(__fsub_rn(v, c[0]));
    for (int i = 1; i < K; ++i) {
      const float dd = fabsf(__fsub_rn(v, c[i]));
      if (dd < bd) {
        bd = dd;
        best = i;
      }
    }
    codes[o] = static_cast<uint8_t>(best);
  }
}

}  // namespace
}  // namespace moeq

using namespace moeq;

extern "C" int moe_quantize_expert(int fmt, int rows, int cols, const float* w, uint8_t* codes_u8, void* scales,
                                   int8_t* codebook, void* ws, size_t ws_bytes, int32_t* dev_status,
                                   moeq_stream stream) {
  (void)dev_status;
  if (fmt != 2 && fmt != 3 && fmt != 4) return MOEQ_ERR_FORMAT;
  if (rows <= 0 || cols <= 0 || cols % 32) return MOEQ_ERR_SHAPE;
  if (static_cast<long long>(rows) * cols >= (1LL << 31)) return MOEQ_ERR_SHAPE;
  if (!w || !codes_u8 || !scales || !codebook) return MOEQ_ERR_ARG;
  if (!aligned16(w)) return MOEQ_ERR_ALIGN;
  if (!ws || ws_bytes < kBins * sizeof(uint32_t) || !aligned16(ws)) return MOEQ_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t* hist = static_cast<uint32_t*>(ws);
  int rc = cuda_status(cudaMemsetAsync(hist, 0, kBins * sizeof(uint32_t), s));
  if (rc) return rc;
  const DeviceInfo& di = device_info();
  const int grid = 4 * (di.sm_count > 0 ? di.sm_count : 1);
  scale_hist_kernel<<<grid, 256, 0, s>>>(fmt, rows, cols, w, scales, hist);
  if ((rc = cuda_status(cudaGetLastError()))) return rc;
  codebook_kernel<<<1, 256, 0, s>>>(1 << fmt, static_cast<long long>(rows) * cols, hist, codebook);
  if ((rc = cuda_status(cudaGetLastError()))) return rc;
  codes_kernel<<<grid, 256, 0, s>>>(fmt, rows, cols, w, scales, codebook, codes_u8);
  return cuda_status(cudaGetLastError());
}
