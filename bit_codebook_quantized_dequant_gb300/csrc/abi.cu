// Host-side parts of the C ABI: sizes, descriptor validation, workspace helpers.
#include <cuda_runtime.h>

#include <deque>
#include <mutex>
#include <vector>

#include "moeq.h"
#include "moeq_host.h"
#include "moeq_layout.h"

namespace moeq {

int validate_matrix(const moeq_matrix& m, int rows, int cols, int experts) {
  if (m.fmt != 2 && m.fmt != 3 && m.fmt != 4 && m.fmt != MOEQ_FP3_PACKED24) return MOEQ_ERR_FORMAT;
  if (m.rows != rows || m.cols != cols || m.num_experts != experts) return MOEQ_ERR_SHAPE;
  if (cols <= 0 || rows <= 0 || cols % 128 != 0) return MOEQ_ERR_SHAPE;
  if (!m.codes || !m.scales) return MOEQ_ERR_ARG;
  if (!aligned16(m.codes) || !aligned16(m.scales)) return MOEQ_ERR_ALIGN;
  const size_t nblk = static_cast<size_t>(rows) * (cols / 32);
  const size_t cbytes = nblk * fmt_block_bytes(m.fmt), sbytes = nblk * fmt_scale_bytes(m.fmt);
  if (experts > 1) {
    if (m.expert_stride_codes % 16 || m.expert_stride_scales % 16) return MOEQ_ERR_ALIGN;
    if (m.expert_stride_codes < cbytes || m.expert_stride_scales < sbytes) return MOEQ_ERR_SHAPE;
  }
  if (!m.codebooks) return MOEQ_ERR_CODEBOOK_MISSING;
  const int need = 1 << fmt_code_bits(m.fmt);
  if (m.cb_len < need) return MOEQ_ERR_CODEBOOK_TRUNCATED;
  if (m.cb_len > need) return MOEQ_ERR_CODEBOOK_MISMATCH;
  if (experts > 1 && m.cb_stride < m.cb_len) return MOEQ_ERR_CODEBOOK_DUPLICATE;
  if (!aligned16(m.codebooks) || (experts > 1 && m.cb_stride % 16)) return MOEQ_ERR_ALIGN;
  return MOEQ_OK;
}

int validate_layer(const moeq_layer* L) {
  if (!L) return MOEQ_ERR_ARG;
  const int H = L->H, I = L->I, E = L->E, k = L->k;
  if (H <= 0 || I <= 0 || E <= 0) return MOEQ_ERR_SHAPE;
  if (H % 256 || I % 128) return MOEQ_ERR_SHAPE;
  if (k < 1 || k > kMaxTopK || k > E) return MOEQ_ERR_ARG;
  if (!L->router) return MOEQ_ERR_ARG;
  if (!aligned16(L->router)) return MOEQ_ERR_ALIGN;
  int rc;
  if ((rc = validate_matrix(L->gate, I, H, E))) return rc;
  if ((rc = validate_matrix(L->up, I, H, E))) return rc;
  if ((rc = validate_matrix(L->down, H, I, E))) return rc;
  if (L->gate.fmt != L->up.fmt) return MOEQ_ERR_FORMAT;
  // the Packed24 layout is decoded for the routed down projection only
  if (L->gate.fmt == MOEQ_FP3_PACKED24) return MOEQ_ERR_FORMAT;
  if (L->has_shared) {
    if ((rc = validate_matrix(L->sgate, I, H, 1))) return rc;
    if ((rc = validate_matrix(L->sup, I, H, 1))) return rc;
    if ((rc = validate_matrix(L->sdown, H, I, 1))) return rc;
    if (L->sgate.fmt != L->sup.fmt) return MOEQ_ERR_FORMAT;
    if (L->sgate.fmt == MOEQ_FP3_PACKED24 || L->sdown.fmt == MOEQ_FP3_PACKED24) return MOEQ_ERR_FORMAT;
  }
  return MOEQ_OK;
}

const DeviceInfo& device_info() {
  static std::mutex mu;
  static std::deque<DeviceInfo> cache;  // references stay valid as devices are added
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(mu);
  for (const auto& d : cache)
    if (d.device == dev) return d;
  DeviceInfo d{};
  d.device = dev;
  cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
  int optin = 0;
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  d.max_smem_optin = static_cast<size_t>(optin);
  cache.push_back(d);
  return cache.back();
}

}  // namespace moeq

using namespace moeq;

extern "C" int moeq_packed_bytes(int fmt, int rows, int cols, size_t* code_bytes,
                                 size_t* scale_bytes) {
  if (fmt == MOEQ_BF16) {  // unpacked rows
    if (rows < 0 || cols < 0) return MOEQ_ERR_SHAPE;
    if (code_bytes) *code_bytes = 2 * static_cast<size_t>(rows) * static_cast<size_t>(cols);
    if (scale_bytes) *scale_bytes = 0;
    return MOEQ_OK;
  }
  if (fmt != 2 && fmt != 3 && fmt != 4 && fmt != MOEQ_FP3_PACKED24) return MOEQ_ERR_FORMAT;
  if (rows < 0 || cols < 0 || cols % 32) return MOEQ_ERR_SHAPE;
  const size_t nblk = static_cast<size_t>(rows) * (cols / 32);
  if (code_bytes) *code_bytes = nblk * fmt_block_bytes(fmt);
  if (scale_bytes) *scale_bytes = nblk * fmt_scale_bytes(fmt);
  return MOEQ_OK;
}

extern "C" int moeq_validate_layer(const moeq_layer* L) { return validate_layer(L); }

extern "C" size_t moe_ffn_workspace(const moeq_layer* L, int T_max, int mode) {
  if (validate_layer(L) != MOEQ_OK || T_max < 1) return 0;
  if (mode == 0) return decode_ws_layout(L->H, L->I, L->E, L->k, L->has_shared).total;
  if (mode == 1) return verify_ws_layout(L->H, L->I, L->E, L->k, L->has_shared).total;
  if (mode == 2) return prefill_ws_layout(L->H, L->I, L->E, L->k, L->has_shared, T_max).total;
  if (mode == 4)  // decode stack of layers shaped like L: decode workspace + a [H] bf16 + y [H] fp32
    return decode_ws_layout(L->H, L->I, L->E, L->k, L->has_shared).total + align256(2 * static_cast<size_t>(L->H)) +
           align256(4 * static_cast<size_t>(L->H));
  if (mode == 5)  // q=4 stack: q=4 workspace + a [4 x H] bf16 + y [4 x H] fp32
    return verify_ws_layout(L->H, L->I, L->E, L->k, L->has_shared).total + align256(8 * static_cast<size_t>(L->H)) +
           align256(16 * static_cast<size_t>(L->H));
  if (mode == 3)  // a stack of layers shaped like L: prefill workspace + the bf16 RMSNorm output
    return prefill_ws_layout(L->H, L->I, L->E, L->k, L->has_shared, T_max).total +
           align256(2 * static_cast<size_t>(T_max) * L->H);
  return 0;
}

extern "C" int moe_ffn_workspace_init(void* ws, size_t ws_bytes, moeq_stream stream) {
  if (!ws || !aligned16(ws)) return MOEQ_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" const char* moeq_version(void) { return "moeq 0.1 sm_103a"; }
