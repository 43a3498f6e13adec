/*
 * moeq -- codebook-quantized mixture-of-experts FFN for GB300 (sm_103a).
 *
 * C ABI. Plain pointers and sizes; no framework types. Unless stated
 * otherwise every pointer argument is a DEVICE pointer owned by the caller,
 * every call only enqueues work on the given CUDA stream (no call
 * synchronizes with the host), and the library allocates no device memory.
 *
 * Errors in arguments, shapes, alignment, formats and codebooks are returned
 * synchronously as a negative moeq_status before anything is enqueued.
 * Errors found on the device (a bounded wait that ran out, an index out of
 * range) are written as a nonzero value into *dev_status, a device int32 the
 * caller zeroes and reads after its own synchronization. No kernel traps.
 *
 * Formats ("DeepSeek V4 Flash: 284B model, up to 32 tok/s on AMD Ryzen AI MAX+
 * 395", section "ROCmFPX: fitting 284B weights into 128 GB"): 32-weight blocks
 * of packed low-bit codes plus a small scale -- FP2 10 B/block (2.50 bpw),
 * FP3 14 B/block (3.50 bpw), FP4 17 B/block (4.25 bpw) -- with a per-expert
 * int8 codebook ("Lucebox x Geometric: DeepSeek V4 Flash 0731 reaches 32.7
 * tok/s on AMD Strix Halo", section "How the model fits on AMD Strix Halo").
 * The pages fix sizes, not bits; the layout below is this library's:
 *
 *   matrix [rows x cols], cols % 128 == 0, nb = cols / 32 blocks per row
 *   code plane : block (r, b) at byte (r*nb + b) * Bc, Bc = 8 / 12 / 16
 *   scale plane: entry r*nb + b, fp16 bits (FP2, FP3) or E8M0 byte (FP4,
 *                value 2^(e-127), e = 255 invalid)
 *   FP2 block  : LE words w0, w1; element j = 16w + 8h + n has its code at
 *                bits 4n+2h .. 4n+2h+1 of word w
 *   FP3 block  : low two bits as FP2 in w0, w1; bit 2 of element (w, h, n) at
 *                bit 4n + p(w,h) of w2, p(0,0)=2, p(0,1)=3, p(1,0)=0, p(1,1)=1
 *   FP4 block  : element j in nibble j%8 of word j/8
 *   FP3 Packed24 block (format code 24): the same 12 bytes and fp16 scale
 *                as FP3, code j at bits 3j .. 3j+2 of the block read as one
 *                96-bit little-endian integer (8 codes per 24 bits)
 *   weight     : scale(r, b) * codebook[code]
 */
#ifndef MOEQ_H
#define MOEQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moeq_stream; /* a cudaStream_t; NULL = legacy default stream */

/* Weight formats. FP2/FP3/FP4: packed 32-weight codebook blocks (the layer
 * roles). MOEQ_FP3_PACKED24: FP3 codes in the Packed24 bit order (the
 * "Packed24 FP3" variant of "deepseek-v4-flash-0731-evox3-rocm", section "The
 * optimization ladder", which names it only; the bit order above is this
 * library's reading), same bytes per block as FP3, accepted for the routed
 * down projection of the decode and q=4 entry points (and by pack, expand)
 * and rejected with MOEQ_ERR_FORMAT elsewhere: a layout to weigh the decode's
 * integer-pipe cost of unpacking 3-bit fields against FP3's planes.
 * MOEQ_BF16: unpacked bf16 rows, no scales or codebooks (the router's format;
 * no packed role takes it, moeq_packed_bytes sizes it as rows x cols x 2
 * bytes of codes and no scale plane). */
typedef enum {
  MOEQ_FP2 = 2,
  MOEQ_FP3 = 3,
  MOEQ_FP4 = 4,
  MOEQ_BF16 = 16,
  MOEQ_FP3_PACKED24 = 24
} moeq_fmt;

typedef enum {
  MOEQ_OK = 0,
  MOEQ_ERR_ARG = -1,                 /* NULL where a pointer is required, bad k, T, ... */
  MOEQ_ERR_SHAPE = -2,               /* unsupported or inconsistent sizes */
  MOEQ_ERR_ALIGN = -3,               /* pointer or stride not 16-byte aligned */
  MOEQ_ERR_FORMAT = -4,              /* fmt not 2, 3 or 4, or not allowed for the role */
  MOEQ_ERR_CODEBOOK_MISSING = -5,    /* codebooks == NULL */
  MOEQ_ERR_CODEBOOK_TRUNCATED = -6,  /* cb_len < 2^fmt */
  MOEQ_ERR_CODEBOOK_MISMATCH = -7,   /* cb_len > 2^fmt */
  MOEQ_ERR_CODEBOOK_DUPLICATE = -8,  /* per-expert codebook records overlap (stride < len) */
  MOEQ_ERR_WORKSPACE = -9,           /* workspace NULL, too small or misaligned */
  MOEQ_ERR_CUDA = -10,               /* a CUDA runtime call failed */
  MOEQ_ERR_DEVICE_TIMEOUT = -11,     /* (device status) a bounded wait ran out */
  MOEQ_ERR_DEVICE_INDEX = -12        /* (device status) an index read on the device was out of range */
} moeq_status;

/* All experts of one role (e.g. the 256 routed gate matrices) share format and
 * shape; expert e's planes start at codes + e*expert_stride_codes and
 * scales + e*expert_stride_scales; its codebook at codebooks + e*cb_stride. */
typedef struct {
  int fmt;                      /* moeq_fmt */
  int rows, cols;               /* cols % 128 == 0 */
  int num_experts;              /* E for routed roles, 1 for shared / dense */
  const void* codes;            /* 16-byte aligned */
  size_t expert_stride_codes;   /* bytes, multiple of 16 */
  const void* scales;           /* 16-byte aligned */
  size_t expert_stride_scales;  /* bytes, multiple of 16 */
  const int8_t* codebooks;      /* [num_experts] records of cb_len int8; 16-byte aligned */
  int cb_len;                   /* must equal 2^fmt */
  int cb_stride;                /* bytes between records: >= cb_len, multiple of 16 */
} moeq_matrix;

typedef struct {
  int H, I, E, k;               /* hidden, expert intermediate, experts, top-k */
  const uint16_t* router;       /* bf16 [E x H] row-major */
  moeq_matrix gate, up;         /* [I x H] per expert */
  moeq_matrix down;             /* [H x I] per expert */
  int has_shared;               /* 1: always-on shared expert with weight 1 */
  moeq_matrix sgate, sup, sdown;
  const uint32_t* h32_signs_x;  /* [H/32] H32 sign masks for x, NULL = no rotation */
  const uint32_t* h32_signs_h;  /* [I/32] H32 sign masks for h, NULL = no rotation */
} moeq_layer;

/* Optional intermediates for parity tests; any pointer may be NULL. For
 * T tokens (T = 1 for a decode, 4 columns for a q=4 verification), "slots" =
 * k routed experts followed by the shared one (if any); vectors are ordered
 * (token, slot). */
typedef struct {
  int8_t* xq; uint16_t* xd;     /* [T x H], [T x H/32] quantized (rotated) input */
  float* logits;                /* [T x E] */
  int32_t* idx; float* p;       /* [T x k] expert indices, combine weights */
  float* h;                     /* [T x slots x I] SwiGLU output before rotation */
  int8_t* hq; uint16_t* hd;     /* [T x slots x I], [T x slots x I/32] */
  float* o;                     /* [T x slots x H] expert outputs before the combine */
  int32_t* S_gate, *S_up;       /* decode / q=4: [T x slots x I x H/32] int32 block partials */
  int32_t* S_down;              /* decode / q=4: [T x slots x H x I/32] */
  uint64_t* trace;              /* decode / q=4: timeline, [grid x 4 roles x trace_cap x 2]
                                   of (globaltimer ns, event << 32 | unit), see MOEQ_TRACE_*;
                                   prefill: CTA 0 of the routed gate/up GEMM, [4 roles x
                                   trace_cap x 2] (roles: expansion, activation producer,
                                   MMA issue, epilogue) */
  int trace_cap;                /* events per (CTA, role) */
  int spin_limit;               /* decode only: polls of each wait on another CTA's progress
                                   before it gives up with MOEQ_ERR_DEVICE_TIMEOUT; 0 = the
                                   default (2^20 polls of up to ~0.2 us), < 0 = give up at
                                   once (tests of the timeout path); the q=4 entry point
                                   always uses the default */
} moeq_debug;

/* Timeline events of moe_ffn_decode and moe_ffn_verify_q4 (role 0 = compute
 * group 0, 1 = producer warp, 3 = compute group 1, 2 = the CTA's teardown:
 * START when its compute ended, READY when the wait for every down item
 * passed, DONE when its combined rows of y are written (CTAs that combine),
 * EPI_END at its arrival on the done counter, unit = arrivals before it).
 * Unused entries stay as the caller left them. */
enum {
  MOEQ_TRACE_START = 1,      /* compute: x quantized; producer: first unit taken */
  MOEQ_TRACE_TAKE = 2,       /* producer: unit taken from the queue */
  MOEQ_TRACE_TOPK = 3,       /* producer: top-k known */
  MOEQ_TRACE_ISSUED = 4,     /* producer: all copies of the unit issued */
  MOEQ_TRACE_READY = 5,      /* compute: the unit's stage is full */
  MOEQ_TRACE_DONE = 6,       /* compute: unit computed */
  MOEQ_TRACE_EPI_BEGIN = 7,  /* epilogue: unit handed over */
  MOEQ_TRACE_EPI_END = 8,    /* epilogue: results published */
  MOEQ_TRACE_SPIN = 9        /* producer: routing wait; first the value seen, then the polls */
};

/* ---------------------------------------------------------------- sizes */

/* Bytes of the two planes of one matrix of format fmt (for MOEQ_BF16 the
 * code plane is the bf16 rows and the scale plane is empty). Returns MOEQ_OK
 * or an error. */
int moeq_packed_bytes(int fmt, int rows, int cols, size_t* code_bytes, size_t* scale_bytes);

/* Host-side checks of a layer descriptor (shapes, formats, alignment,
 * codebook records); enqueues nothing. The codebook checks mirror the loader
 * validation for "missing, duplicated, truncated, or mismatched codebooks" of
 * "Lucebox x Geometric ...", section "Lucebox Engine integration with
 * Geometric". Returns MOEQ_OK or the first error found. */
int moeq_validate_layer(const moeq_layer* L);

/* Workspace bytes for a call: mode 0 = decode, 1 = q=4 verify, 2 = prefill of
 * up to T_max tokens, 3 = moe_ffn_stack_prefill of up to T_max tokens through
 * layers shaped like L, 4 = moe_ffn_stack_decode through layers shaped like L,
 * 5 = moe_ffn_stack_verify_q4 through layers shaped like L (T_max is ignored
 * for modes 0, 1, 4 and 5). 0 on an invalid descriptor. */
size_t moe_ffn_workspace(const moeq_layer* L, int T_max, int mode);

/* Zero a freshly allocated workspace (enqueued memset). Needed once; every
 * FFN call leaves the workspace ready for the next one on the same stream. */
int moe_ffn_workspace_init(void* ws, size_t ws_bytes, moeq_stream stream);

/* ---------------------------------------------------------------- entry points */

/* Pack one matrix into the block formats of "DeepSeek V4 Flash: 284B model,
 * up to 32 tok/s on AMD Ryzen AI MAX+ 395", section "ROCmFPX: fitting 284B
 * weights into 128 GB" (blocks of 32 weights stored as small codebook codes
 * with one small scale each; FP2 2.5, FP3 3.5, FP4 4.25 bits per weight):
 * codes_u8 [rows x cols] (one code per byte, below 2^bits) and scales
 * [rows x cols/32] (fp16 bits for FP2/FP3, E8M0 bytes for FP4, row-major) go
 * to the code plane out_codes (per 32-block: FP2 8 bytes of 2-bit codes, FP3
 * 12 bytes: the low two bits of the codes in two words and their third bits in
 * a third, FP3 Packed24 12 bytes of consecutive 3-bit fields, FP4 16 bytes of
 * nibbles) and the scale plane out_scales (the input's layout; it is copied).
 * fmt is 2, 3, 4 or MOEQ_FP3_PACKED24 (MOEQ_ERR_FORMAT otherwise); cols % 32
 * == 0; all pointers are device pointers owned by the caller, 16-byte aligned.
 * A code out of range sets *dev_status to MOEQ_ERR_DEVICE_INDEX and is packed
 * masked to the format's bits. */
int moe_pack_expert(int fmt, int rows, int cols, const uint8_t* codes_u8, const void* scales,
                    void* out_codes, void* out_scales, int32_t* dev_status, moeq_stream stream);

/* Codebook quantization of one expert matrix: fp32 weights -> the inputs of
 * moe_pack_expert (codes, block scales) and the expert's codebook. The pages
 * name "learned per-expert codebooks" ("Lucebox x Geometric ...", section
 * "How the model fits on AMD Strix Halo") without printing how they are
 * learned; this is the library's reading, deterministic and exact in its
 * integer steps:
 *   1. per 32-block, m = max |w|: FP2/FP3 scale d = fp16_rne(m / 127) (fp32
 *      division; the largest finite fp16 on overflow); FP4 E8M0 byte e + 127
 *      with e the smallest integer >= -127 such that 127 * 2^e >= m (<= 127);
 *   2. v = w / d (fp32; 0 where d == 0), g = clamp(rint(v), -127, 127), and
 *      the histogram of g over the whole matrix;
 *   3. 2^fmt int8 entries start at the histogram's mid-quantiles (entry i =
 *      the smallest g whose cumulative count exceeds floor((2i+1)N / 2^(fmt+1)),
 *      N weights), then 8 Lloyd steps on the histogram in integers (each g to
 *      its nearest entry, ties to the lower index; each entry with a non-empty
 *      cell to the cell's mean rounded half up; entries sorted ascending);
 *   4. each weight's code = the entry nearest to v in fp32, ties to the lower
 *      index.
 * w [rows x cols] fp32 (16-byte aligned), codes_u8 [rows x cols], scales
 * [rows x cols/32] (fp16 bits for FP2/FP3, E8M0 bytes for FP4), codebook
 * [2^fmt] int8; all device memory owned by the caller. ws: >= 1 KiB of device
 * memory (16-byte aligned), cleared by the call. cols % 32 == 0,
 * rows * cols < 2^31. Three kernels enqueued on the stream. */
int moe_quantize_expert(int fmt, int rows, int cols, const float* w, uint8_t* codes_u8, void* scales,
                        int8_t* codebook, void* ws, size_t ws_bytes, int32_t* dev_status,
                        moeq_stream stream);

/* The "generic expand-then-multiply fallback" that "Lucebox x Geometric ...",
 * section "Lucebox Engine integration with Geometric", measures the fused
 * matvec against (2.2x), as an ablation on this GPU; not on the fused path.
 *
 * moe_expand_bf16: experts e0 .. e0+ne-1 of the packed matrix m to bf16
 * weights out_bf16 [ne x rows x cols], w = bf16_rne(codebook[code] * block
 * scale) (the product is exact in fp32). m is validated as a packed role;
 * out_bf16 is device memory of the caller, 16-byte aligned.
 *
 * moe_ffn_decode_expanded: batch-1 decode of a layer whose gate, up, down
 * (and shared) matrices are MOEQ_BF16 rows (codes = bf16 [rows x cols] per
 * expert, expert_stride_codes bytes apart; scales and codebooks unused): the
 * router logits, top-k and weights of moe_route_topk (the same canonical
 * order, one warp per router row over the grid), then per slot g = W_gate x,
 * u = W_up x (bf16 weights, x as given, fp32 sums), h = silu(g) u in fp32 (no
 * quantization), o = W_down h, y = sum_slot p o + o_shared in slot order.
 * H a multiple of 256, I of 128, E <= 1024, no H32 rotation. ws: at least
 * moe_ffn_expanded_workspace(H, I, E, k, has_shared) bytes of device memory,
 * zeroed once (each call leaves its arrival counter at zero); layout idx
 * [k] int32 at byte 0, then p, the counter, logits and h, 256-byte aligned.
 * Three kernels enqueued on the stream. */
int moe_expand_bf16(const moeq_matrix* m, int e0, int ne, uint16_t* out_bf16, moeq_stream stream);
size_t moe_ffn_expanded_workspace(int H, int I, int E, int k, int has_shared);
int moe_ffn_decode_expanded(const moeq_layer* L, const uint16_t* x, float* y, void* ws, size_t ws_bytes,
                            int32_t* dev_status, moeq_stream stream);

/* Router and top-k for T tokens ("DeepSeek V4 Flash: 284B model ...", section
 * "Decode: up to 32 tok/s": routing with dedicated TOP_K kernels):
 * logits[t,e] = sum_h router[e,h] x[t,h] with bf16 operands and an fp32 sum in
 * the canonical order (32 partials j over h = 256 i + 8 j + t', then pairwise
 * rounds 16, 8, 4, 2, 1); idx = the k largest (ties to the lower index);
 * w = softmax over all E logits at those indices (no renormalization).
 * x [T x H] bf16, router [E x H] bf16, idx [T x k], w [T x k], logits_opt
 * [T x E] or NULL. H % 256 == 0, 1 <= k <= min(E, 8), E <= 1024. */
int moe_route_topk(const uint16_t* x, int T, const uint16_t* router, int E, int H, int k,
                   int32_t* idx, float* w, float* logits_opt, int32_t* dev_status,
                   moeq_stream stream);

/* Batch-1 decode of one layer: y [H] fp32 from x [H] bf16 (see the layer
 * comment above for the computation: Q8 of the optionally H32-rotated x,
 * router + top-k, per selected expert fused dequant gate/up GEMV, SwiGLU,
 * optional H32 + Q8 of h, down GEMV, combine sum_slot p*o + shared in slot
 * order). One persistent cooperative kernel; no host synchronization
 * ("Lucebox x Geometric ...", section "Lucebox Engine integration with
 * Geometric": fused matvec and sync-free MoE decode). ws: a workspace of
 * moe_ffn_workspace(L, 1, 0) bytes, zeroed once with moe_ffn_workspace_init;
 * calls that share a workspace must be ordered (same stream). dbg may be NULL.
 * Requires H <= 4096 and a multiple of 256, I <= 4096 and a multiple of 128,
 * E <= 512 and a multiple of 4; k <= 8. */
int moe_ffn_decode(const moeq_layer* L, const uint16_t* x, float* y, void* ws, size_t ws_bytes,
                   int32_t* dev_status, const moeq_debug* dbg, moeq_stream stream);

/* Batch-1 decode like moe_ffn_decode, for callers that cannot allocate device
 * memory (for example a C program or a foreign runtime that holds device
 * pointers to the weights and activations but has no device allocator): the
 * scratch is a static array of the library, 160 KiB per device, instead of a
 * caller workspace. This entry point has no counterpart on the source pages.
 *   - Shapes whose decode workspace (moe_ffn_workspace(L, 1, 0)) exceeds
 *     160 KiB are rejected with MOEQ_ERR_WORKSPACE before anything is
 *     enqueued (the decode layer H=4096, I=2048, E=256, k=6 + shared expert
 *     needs 131.5 KiB).
 *   - The scratch's counters must start at zero: each call clears them with
 *     an enqueued memset before its kernel, so a call that ended in a device
 *     error does not affect the next one.
 *   - Every call on a device uses the same scratch: calls that may overlap in
 *     time (different streams, or different host threads without ordering)
 *     race on it and give wrong results. Order them, e.g. on one stream.
 *   - The first call on a device (and the first after the device's context
 *     was reset) looks up the scratch's address (host side, no allocation);
 *     make that first call before any stream capture.
 * Results are those of moe_ffn_decode; no debug output. */
int moe_ffn_decode_static(const moeq_layer* L, const uint16_t* x, float* y, int32_t* dev_status,
                          moeq_stream stream);

/* q=4 verification ("DeepSeek V4 Flash: 284B model ...", section "Decode: up
 * to 32 tok/s": the verifier decodes each packed weight once and applies it
 * to all four columns): four columns x [4 x H] bf16, each routed
 * independently; y [4 x H] fp32 = the decode of each column, bit for bit
 * what four moe_ffn_decode calls return. Every packed block of every selected
 * expert (read once for all columns that select it), of the shared expert and
 * of the optional dense projection is expanded once per call and applied to
 * every column that uses it. dense: NULL or one matrix [D x H] (any format,
 * D % 32 == 0, one codebook record); y_dense [4 x D] fp32 = dense applied to
 * the column's quantized (and, with h32_signs_x, rotated) input -- the same
 * Q8 operand as the FFN; with dense NULL y_dense is not touched and may be
 * NULL. One persistent cooperative kernel. ws: moe_ffn_workspace(L, 4, 1)
 * bytes, zeroed once; calls that share a workspace must be ordered. Same shape
 * limits as moe_ffn_decode. */
int moe_ffn_verify_q4(const moeq_layer* L, const moeq_matrix* dense, const uint16_t* x, float* y,
                      float* y_dense, void* ws, size_t ws_bytes, int32_t* dev_status,
                      const moeq_debug* dbg, moeq_stream stream);

/* Expert-grouped prefill of T tokens ("deepseek-v4-flash-0731-evox3-rocm",
 * section "The optimization ladder": fused multi-token prefill): per token
 * the result of moe_ffn_decode (bit-identical xq, xd, logits, indices and
 * weights) up to the rounding of the tensor-core contraction: the weights
 * (code x block scale) and activations (code x scale) enter as two bf16
 * parts each, and the products a_hi x_hi + a_hi x_lo + a_lo x_hi are within
 * 3.1e-5 of each a x, summed in fp32. Computed as router + top-k for all
 * tokens, a stable counting sort of the (token, slot) pairs by expert
 * (ascending token, then slot), grouped GEMMs for gate/up (+SwiGLU, H32, Q8
 * of h) and down on the tensor cores, and a gather-combine in slot order.
 * H and I must be multiples of 128 (as every matrix's cols). If
 * residual is not NULL, y = residual + FFN(x) rounded once (the residual add
 * of a stacked layer; y may equal residual). x [T x H] bf16, y [T x H] fp32.
 * ws: at least moe_ffn_workspace(L, T, 2) bytes (contents need no zeroing);
 * too small -> MOEQ_ERR_WORKSPACE. T = 0 enqueues nothing. Several kernels
 * on the stream, no host synchronization; dbg (NULL or [T x slots] vectors)
 * receives xq, xd, logits, idx, p, h, hq, hd and o. */
int moe_ffn_prefill(const moeq_layer* L, const uint16_t* x, int T, const float* residual, float* y,
                    void* ws, size_t ws_bytes, int32_t* dev_status, const moeq_debug* dbg,
                    moeq_stream stream);

/* Prefill of T tokens through a stack of nlayers layers (layers[l], all with
 * the same H) with an fp32 residual stream ("Lucebox x Geometric ...",
 * section "How the model fits": the prompt is pushed layer by layer through
 * the whole stack):
 *   r_0 = float(x);  a_l = moe_rmsnorm_bf16(r_l);  r_{l+1} = r_l + FFN_l(a_l)
 * with FFN_l = moe_ffn_prefill of layer l (residual form, in place). x [T x H]
 * bf16; r [T x H] fp32 receives r_nlayers. ws: at least
 * moe_ffn_workspace(L, T, 3) bytes for the largest layer shape. Enqueued on
 * the stream, no host synchronization. */
int moe_ffn_stack_prefill(const moeq_layer* layers, int nlayers, const uint16_t* x, int T, float* r,
                          void* ws, size_t ws_bytes, int32_t* dev_status, moeq_stream stream);

/* One decode token through a stack of nlayers layers (layers[l], all with the
 * same H) with an fp32 residual stream ("DeepSeek V4 Flash: 284B model ...",
 * section "ROCmFPX: fitting 284B weights into 128 GB": every generated token
 * streams the active weights of every layer):
 *   r_0 = float(x);  a_l = moe_rmsnorm_bf16(r_l);  r_{l+1} = r_l + y_l
 * with y_l = moe_ffn_decode of layer l on a_l and correctly rounded fp32 adds.
 * x [H] bf16; r [H] fp32 receives r_nlayers. ws: at least
 * moe_ffn_workspace(L, 1, 4) bytes for the largest layer shape, zeroed once
 * with moe_ffn_workspace_init (its decode part is reused by every layer in
 * turn). 2 * nlayers + 1 kernels enqueued on the stream, no host
 * synchronization; the shapes each decode takes are those of moe_ffn_decode. */
int moe_ffn_stack_decode(const moeq_layer* layers, int nlayers, const uint16_t* x, float* r,
                         void* ws, size_t ws_bytes, int32_t* dev_status, moeq_stream stream);

/* q=4 verification through a stack of nlayers layers: four independently
 * routed columns ("DeepSeek V4 Flash: 284B model ...", section "Decode: up to
 * 32 tok/s": every packed weight a call touches is decoded once for all the
 * columns that use it), each carried through the layers with the recurrence
 * of moe_ffn_stack_decode:
 *   r_0[c] = float(x[c]);  a_l[c] = RMSNorm(r_l[c]);  r_{l+1}[c] = r_l[c] + y_l[c]
 * with y_l = moe_ffn_verify_q4 of layer l on the four a_l (no dense
 * projection). Column c of r_nlayers equals moe_ffn_stack_decode of x[c] bit
 * for bit. x [4 x H] bf16; r [4 x H] fp32 receives r_nlayers. ws: at least
 * moe_ffn_workspace(L, 1, 5) bytes for the largest layer shape, zeroed once
 * with moe_ffn_workspace_init. 2 * nlayers + 1 kernels enqueued on the
 * stream, no host synchronization; shapes as for moe_ffn_verify_q4. */
int moe_ffn_stack_verify_q4(const moeq_layer* layers, int nlayers, const uint16_t* x, float* r,
                            void* ws, size_t ws_bytes, int32_t* dev_status, moeq_stream stream);

/* H32 rotation ("deepseek-v4-flash-0731-evox3-rocm", section "The optimization
 * ladder"): out = H D in per 32-block, H the 32x32 Sylvester Hadamard matrix
 * (unnormalized), D = diag(-1 where bit i of signs[b] is set); fp32 butterfly
 * stages 0..4, (a, b) -> (a + b, a - b). signs NULL = no sign flips. in and
 * out [nblk x 32] fp32 (may alias). */
int h32_rotate(const float* in, float* out, int nblk, const uint32_t* signs, moeq_stream stream);

/* RMSNorm with unit weight between stacked layers, rounded to bf16:
 * a[t,:] = bf16_rne(r[t,:] / sqrt(sum(r^2)/H + 1e-6)) with the sum of squares
 * in fp32 in the router's canonical order and correctly rounded fp32
 * operations. r [T x H] fp32, a [T x H] bf16, H % 256 == 0. */
int moe_rmsnorm_bf16(const float* r, int T, int H, uint16_t* a, moeq_stream stream);

/* Version string of the library build. */
const char* moeq_version(void);

#ifdef __cplusplus
}
#endif
#endif
