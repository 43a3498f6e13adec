// moe_pack_expert: one code per byte -> the FP2 / FP3 / FP4 code plane of
// include/moeq.h (block sizes from "DeepSeek V4 Flash: 284B model, up to 32
// tok/s on AMD Ryzen AI MAX+ 395", section "ROCmFPX: fitting 284B weights into
// 128 GB"). One thread packs one 32-weight block from two 16-byte loads.
#include <cuda_runtime.h>

#include "moeq.h"
#include "moeq_device.cuh"
#include "moeq_host.h"

namespace moeq {
namespace {

__device__ __forceinline__ uint32_t byte_of(const uint4& v, int j) {
  const uint32_t w = j < 4 ? v.x : j < 8 ? v.y : j < 12 ? v.z : v.w;
  return (w >> (8 * (j & 3))) & 0xffu;
}

__global__ void pack_kernel(int fmt, size_t nblk, const uint8_t* __restrict__ codes,
                            uint8_t* __restrict__ out, int32_t* status) {
  const size_t blk = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (blk >= nblk) return;
  const uint4 c0 = __ldg(reinterpret_cast<const uint4*>(codes + 32 * blk));
  const uint4 c1 = __ldg(reinterpret_cast<const uint4*>(codes + 32 * blk + 16));
  const uint32_t lim = 1u << (fmt == MOEQ_FP3_PACKED24 ? 3 : fmt);
  uint32_t c[32];
  bool bad = false;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    c[j] = j < 16 ? byte_of(c0, j) : byte_of(c1, j - 16);
    bad |= c[j] >= lim;
    c[j] &= lim - 1;
  }
  if (bad) set_status(status, MOEQ_ERR_DEVICE_INDEX);
  if (fmt == MOEQ_FP3_PACKED24) {  // code j at bits 3j..3j+2 of the 96-bit block
    uint32_t w[3] = {0, 0, 0};
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int bit = 3 * j;
      w[bit >> 5] |= c[j] << (bit & 31);
      if ((bit & 31) > 29) w[(bit >> 5) + 1] |= c[j] >> (32 - (bit & 31));  // the field crosses a word
    }
    uint32_t* o = reinterpret_cast<uint32_t*>(out + 12 * blk);
    o[0] = w[0];
    o[1] = w[1];
    o[2] = w[2];
    return;
  }
  if (fmt == 4) {
    uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
    for (int j = 0; j < 32; ++j) w[j >> 3] |= c[j] << (4 * (j & 7));
    reinterpret_cast<uint4*>(out)[blk] = make_uint4(w[0], w[1], w[2], w[3]);
    return;
  }
  // element j = 16 w + 8 h + n: low bits at 4n + 2h of word w;
  // FP3 bit 2 at 4n + p(w, h) of word 2, p = {{2, 3}, {0, 1}}
  uint32_t w0 = 0, w1 = 0, hi = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int wi = j >> 4, h = (j >> 3) & 1, n = j & 7;
    const uint32_t lo = (c[j] & 3u) << (4 * n + 2 * h);
    if (wi == 0) w0 |= lo; else w1 |= lo;
    const int p = wi == 0 ? (h == 0 ? 2 : 3) : (h == 0 ? 0 : 1);
    hi |= ((c[j] >> 2) & 1u) << (4 * n + p);
  }
  if (fmt == 2) {
    reinterpret_cast<uint2*>(out)[blk] = make_uint2(w0, w1);
  } else {
    uint32_t* o = reinterpret_cast<uint32_t*>(out + 12 * blk);
    o[0] = w0;
    o[1] = w1;
    o[2] = hi;
  }
}

}  // namespace
}  // namespace moeq

using namespace moeq;

extern "C" int moe_pack_expert(int fmt, int rows, int cols, const uint8_t* codes_u8,
                               const void* scales, void* out_codes, void* out_scales,
                               int32_t* dev_status, moeq_stream stream) {
  if (fmt != 2 && fmt != 3 && fmt != 4 && fmt != MOEQ_FP3_PACKED24) return MOEQ_ERR_FORMAT;
  if (rows < 0 || cols < 0 || cols % 32) return MOEQ_ERR_SHAPE;
  if (rows == 0 || cols == 0) return MOEQ_OK;
  if (!codes_u8 || !out_codes) return MOEQ_ERR_ARG;
  if (!aligned16(codes_u8) || !aligned16(out_codes)) return MOEQ_ERR_ALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t nblk = static_cast<size_t>(rows) * (cols / 32);
  const int threads = 256;
  const size_t grid = (nblk + threads - 1) / threads;
  if (grid > 0x7fffffffull) return MOEQ_ERR_SHAPE;
  pack_kernel<<<static_cast<unsigned>(grid), threads, 0, s>>>(
      fmt, nblk, codes_u8, static_cast<uint8_t*>(out_codes), dev_status);
  if (cudaGetLastError() != cudaSuccess) return MOEQ_ERR_CUDA;
  if (scales && out_scales && scales != out_scales) {
    const size_t sbytes = nblk * fmt_scale_bytes(fmt);
    if (cudaMemcpyAsync(out_scales, scales, sbytes, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return MOEQ_ERR_CUDA;
  }
  return MOEQ_OK;
}
