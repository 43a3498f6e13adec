// Expert-grouped prefill (see include/moeq.h).
#include <cuda_runtime.h>

#include "moeq.h"
#include "moeq_host.h"

using namespace moeq;

extern "C" int moe_ffn_prefill(const moeq_layer* L, const uint16_t* x, int T, const float* residual,
                               float* y, void* ws, size_t ws_bytes, int32_t* dev_status,
                               const moeq_debug* dbg, moeq_stream stream) {
  (void)L; (void)x; (void)T; (void)residual; (void)y; (void)ws; (void)ws_bytes;
  (void)dev_status; (void)dbg; (void)stream;
  return MOEQ_ERR_SHAPE;
}
