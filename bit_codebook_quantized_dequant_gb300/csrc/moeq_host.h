// Host-side internals of the moeq library: the device view of a packed matrix,
// descriptor validation and cached device attributes.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moeq.h"

namespace moeq {

// Device view of one role's matrices (plain data, passed to kernels by value).
struct DMat {
  const uint8_t* codes;
  const uint8_t* scales;
  const int8_t* cb;
  unsigned long long stride_codes;   // bytes between experts
  unsigned long long stride_scales;  // bytes between experts
  int cb_stride;                     // bytes between codebook records
  int rows, cols, fmt;
};

inline int fmt_block_bytes(int fmt) {
  return fmt == 2 ? 8 : fmt == 3 || fmt == MOEQ_FP3_PACKED24 ? 12 : fmt == 4 ? 16 : 0;
}
inline int fmt_code_bits(int fmt) { return fmt == MOEQ_FP3_PACKED24 ? 3 : fmt; }
inline int fmt_scale_bytes(int fmt) { return fmt == 4 ? 1 : 2; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline DMat to_dmat(const moeq_matrix& m) {
  DMat d;
  d.codes = static_cast<const uint8_t*>(m.codes);
  d.scales = static_cast<const uint8_t*>(m.scales);
  d.cb = m.codebooks;
  d.stride_codes = m.expert_stride_codes;
  d.stride_scales = m.expert_stride_scales;
  d.cb_stride = m.cb_stride;
  d.rows = m.rows;
  d.cols = m.cols;
  d.fmt = m.fmt;
  return d;
}

// Checks one matrix descriptor against an expected shape. Returns MOEQ_OK or
// an error code; codebook checks follow the order missing, truncated,
// mismatched, duplicated.
int validate_matrix(const moeq_matrix& m, int rows, int cols, int experts);

// Checks a layer descriptor (all roles, shapes, router, signs).
int validate_layer(const moeq_layer* L);

// Cached per-device attributes.
struct DeviceInfo {
  int device;
  int sm_count;
  size_t max_smem_optin;
};
const DeviceInfo& device_info();

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOEQ_OK : MOEQ_ERR_CUDA; }

// One grouped GEMM of the prefill on the tensor cores (gemm_tc.cu): tiles of
// 128 weight rows x 128 grouped rows over groups [g0, g1) with matrix w
// (expert = group, or expert 0 for the shared expert). act_hi / act_lo: the
// bf16 parts [rows x K] of the grouped activations (code times block scale).
// epi 0: write g [rows x R] fp32; 1: read g, SwiGLU + H32 + Q8 of h, write
// h's parts hhi / hlo [rows x R]; 2: write o [rows x R] fp32.
struct TcGemm {
  int epi;
  DMat w;
  int shared, g0, g1;
  const int* toff;
  const int* offsets;
  int K, R, rows;
  const uint16_t* act_hi;
  const uint16_t* act_lo;
  float* g;
  uint16_t* hhi;
  uint16_t* hlo;
  const uint32_t* signs_h;
  float* o;
  const int* pid;
  int T, k, ns;
  moeq_debug dbg;
  int32_t* status;
};
int tc_grouped_gemm(const TcGemm& g, cudaStream_t s);

// One step of a decode stack on `rows` tokens (route.cu), row by row: r =
// float(x) if x, else r += y if y; then a = RMSNorm(r) if a. One CTA a row.
int stack_step_launch(const uint16_t* x, const float* y, float* r, uint16_t* a, int H, int rows,
                      cudaStream_t s);

// Router + top-k of T tokens enqueued on s (route.cu).
int route_topk_launch(const uint16_t* x, int T, const uint16_t* router, int E, int H, int k,
                      int32_t* idx, float* w, float* logits, cudaStream_t s);

}  // namespace moeq
