// Device twin of the seeded input generator (see include/moeq_synth.h).
#include <cuda_runtime.h>

#include "moeq_host.h"
#include "moeq_synth.h"

namespace moeq {
namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void synth_codes_kernel(uint64_t key, int bits, size_t nwords, uint8_t* out) {
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= nwords) return;
  const uint64_t u = mix64(key + (i + 1) * kGamma);
  const uint32_t mask = (1u << bits) - 1u;
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t v = 0;
#pragma unroll
    for (int t = 0; t < 4; ++t) v |= ((static_cast<uint32_t>(u >> (4 * (4 * q + t)))) & mask) << (8 * t);
    w[q] = v;
  }
  reinterpret_cast<uint4*>(out)[i] = make_uint4(w[0], w[1], w[2], w[3]);
}

__global__ void synth_scales_kernel(uint64_t key, int bits, size_t n, void* out) {
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint64_t hi = mix64(key + (i + 1) * kGamma) >> 32;
  if (bits == 4) {
    static_cast<uint8_t*>(out)[i] = static_cast<uint8_t>(114u + hi % 7u);
  } else {
    static_cast<uint16_t*>(out)[i] = static_cast<uint16_t>(0x068Eu + hi % (0x211Fu - 0x068Eu + 1u));
  }
}

}  // namespace
}  // namespace moeq

using namespace moeq;

extern "C" int moeq_synth_codes(uint64_t seed, uint64_t stream, int bits, size_t n, uint8_t* out,
                                moeq_stream s) {
  if (bits < 1 || bits > 4 || n % 16) return MOEQ_ERR_ARG;
  if (n == 0) return MOEQ_OK;
  if (!out || !aligned16(out)) return MOEQ_ERR_ALIGN;
  const uint64_t key = mix64(seed * kGamma + stream);
  const size_t nwords = n / 16;
  const int threads = 256;
  synth_codes_kernel<<<static_cast<unsigned>((nwords + threads - 1) / threads), threads, 0,
                       reinterpret_cast<cudaStream_t>(s)>>>(key, bits, nwords, out);
  return cuda_status(cudaGetLastError());
}

extern "C" int moeq_synth_scales(uint64_t seed, uint64_t stream, int bits, size_t n, void* out,
                                 moeq_stream s) {
  if (bits < 2 || bits > 4) return MOEQ_ERR_ARG;
  if (n == 0) return MOEQ_OK;
  if (!out) return MOEQ_ERR_ARG;
  const uint64_t key = mix64(seed * kGamma + stream);
  const int threads = 256;
  synth_scales_kernel<<<static_cast<unsigned>((n + threads - 1) / threads), threads, 0,
                        reinterpret_cast<cudaStream_t>(s)>>>(key, bits, n, out);
  return cuda_status(cudaGetLastError());
}
