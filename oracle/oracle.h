/*
 * CPU oracle for the codebook-quantized MoE FFN -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded C restatement of what the hot path computes,
 * used by the tests, by __graft_entry__.smoke() and by the CPU-baseline leg of
 * bench.py to check the CUDA library. Nothing in the library links, includes or
 * calls this code, and this code includes nothing of the library.
 *
 * Sources (page title, section):
 *   - "DeepSeek V4 Flash: 284B model, up to 32 tok/s on AMD Ryzen AI MAX+ 395",
 *     section "ROCmFPX: fitting 284B weights into 128 GB": 32-weight blocks of
 *     packed low-bit codes plus small scales; ROCmFP2 10 B/block (2.50 bpw),
 *     ROCmFP3 3.50 bpw, ROCmFP4 4.25 bpw; kernels expand small codebooks and
 *     feed integer dot products.
 *   - "Lucebox x Geometric: DeepSeek V4 Flash 0731 reaches 32.7 tok/s on AMD
 *     Strix Halo", section "How the model fits on AMD Strix Halo": learned
 *     per-expert codebooks for routed experts; gate/up at 2.5 bpw, down at
 *     3.5 bpw, shared expert at 4.25 bpw.
 *   - soothill.io page "deepseek-v4-flash-0731-evox3-rocm" (no printed title),
 *     section "The optimization ladder": H32 rotations of expert tensors, fused
 *     basis, shared rotated input, multi-token and layer-major prefill.
 *   - same page 2, section "Decode: up to 32 tok/s": q=4 verification decodes
 *     each packed dense weight once and applies it to all four columns.
 * The pages fix bytes per block and the mechanism only; bit layouts, scale
 * encodings, rounding and reduction orders are this library's specification,
 * restated in each function's comment below.
 *
 * Floating-point results the method defines are computed in fp64. Steps whose
 * outcome is an integer decided by fp32 arithmetic (activation quantization,
 * router logits that decide the top-k, the RMSNorm that rounds to bf16) are
 * written in fp32 with the IEEE operations named, so that both sides take the
 * same decision. Build with -O2 -ffp-contract=off and without fast-math.
 */
#ifndef MOEQ_ORACLE_H
#define MOEQ_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* One role of a layer (e.g. all routed gate matrices): per-expert host pointers
 * to packed planes; entries for experts the caller did not materialize may be
 * NULL, and touching one returns ORC_ERR_MISSING. */
typedef struct {
  int fmt;            /* 2, 3 or 4 bits per code, or 24: 3-bit codes in the Packed24 layout */
  int rows, cols;     /* cols % 32 == 0 */
  const uint8_t* const* codes;  /* [E] code planes: rows x (cols/32) blocks */
  const void* const* scales;    /* [E] scale planes: fp16 bits (fmt 2,3) or E8M0 bytes (fmt 4) */
  const int8_t* const* cb;      /* [E] codebooks of 2^bits entries */
} orc_matrix;

typedef struct {
  int H, I, E, k;
  const uint16_t* router;       /* bf16 [E x H], row-major */
  orc_matrix gate, up, down;    /* routed experts */
  int has_shared;
  orc_matrix sgate, sup, sdown; /* shared expert, expert index 0 */
  const uint32_t* signs_x;      /* [H/32] H32 sign masks for x, NULL = no rotation */
  const uint32_t* signs_h;      /* [I/32] H32 sign masks for h, NULL = no rotation */
} orc_layer;

/* Optional intermediates of one decode; every pointer may be NULL. Slot order is
 * the top-k order; index k (the (k+1)-th entry) holds the shared expert. */
typedef struct {
  int8_t* xq; uint16_t* xd;         /* [H], [H/32] */
  float* logits;                    /* [E] */
  int32_t* idx; double* p;          /* [k], [k] */
  int32_t* S_gate; int32_t* S_up;   /* [(k+1) x I x H/32] per-block int32 partials */
  double* g; double* u; double* h;  /* [(k+1) x I] */
  int8_t* hq; uint16_t* hd;         /* [(k+1) x I], [(k+1) x I/32] */
  int32_t* S_down;                  /* [(k+1) x H x I/32] */
  double* o;                        /* [(k+1) x H] */
  /* teacher forcing: when non-NULL, these replace the oracle's own quantized h
   * ([(k+1) x I] and [(k+1) x I/32]) before the down projection */
  const int8_t* force_hq; const uint16_t* force_hd;
  /* when non-NULL, these replace the oracle's own routing ([k] each) */
  const int32_t* force_idx;
} orc_trace;

enum { ORC_OK = 0, ORC_ERR_ARG = -1, ORC_ERR_MISSING = -2 };

/* number conversions (RNE) */
uint16_t orc_f32_to_f16(float f);
double orc_f16_to_f64(uint16_t h);
uint16_t orc_f32_to_bf16(float f);
float orc_bf16_to_f32(uint16_t b);

/* packing */
int orc_packed_bytes(int fmt, int rows, int cols, size_t* code_bytes, size_t* scale_bytes);
int orc_pack(int fmt, int rows, int cols, const uint8_t* codes, uint8_t* out_codes);
int orc_unpack(int fmt, int rows, int cols, const uint8_t* packed, uint8_t* codes_out);
double orc_scale_value(int fmt, const void* scales, size_t i);

/* activation quantization (per 32-block int8 + fp16 scale) */
void orc_q8(const float* v, int n, int8_t* q, uint16_t* d);

/* H32 rotation: fp32 butterfly (the specified arithmetic) and fp64 matrix form */
void orc_h32_f32(const float* in, const uint32_t* signs, int nblk, float* out);
void orc_h32_f64(const double* in, const uint32_t* signs, int nblk, double* out);

/* router */
float orc_router_logit(const uint16_t* x, const uint16_t* w, int H);
void orc_router(const uint16_t* x, int T, const uint16_t* Wr, int E, int H, float* logits);
void orc_topk(const float* logits, int E, int k, int32_t* idx, double* p);

/* block-quantized matrix-vector product */
int orc_block_partials(const orc_matrix* m, int expert, int row, const int8_t* q, int32_t* S);
int orc_matvec(const orc_matrix* m, int expert, const int8_t* q, const uint16_t* d,
               double* out, int32_t* S_out);

/* FFN */
int orc_ffn_decode(const orc_layer* L, const uint16_t* x, double* y, orc_trace* tr);
int orc_ffn_verify_q4(const orc_layer* L, const orc_matrix* dense, const uint16_t* x,
                      double* y, double* y_dense, orc_trace* tr4);
int orc_ffn_prefill(const orc_layer* L, const uint16_t* x, int T, double* y);

/* layer stack helpers */
void orc_rmsnorm_bf16(const float* r, int H, uint16_t* a);
int orc_quantize_expert(int fmt, int rows, int cols, const float* w, uint8_t* codes, void* scales,
                        int8_t* cb);

#ifdef __cplusplus
}
#endif
#endif
