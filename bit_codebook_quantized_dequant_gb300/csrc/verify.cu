// q=4 verification (see include/moeq.h).
#include <cuda_runtime.h>

#include "moeq.h"
#include "moeq_host.h"

using namespace moeq;

extern "C" int moe_ffn_verify_q4(const moeq_layer* L, const moeq_matrix* dense, const uint16_t* x,
                                 float* y, float* y_dense, void* ws, size_t ws_bytes,
                                 int32_t* dev_status, const moeq_debug* dbg, moeq_stream stream) {
  (void)L; (void)dense; (void)x; (void)y; (void)y_dense; (void)ws; (void)ws_bytes;
  (void)dev_status; (void)dbg; (void)stream;
  return MOEQ_ERR_SHAPE;
}
