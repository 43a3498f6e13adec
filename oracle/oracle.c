/*
 * CPU oracle for the codebook-quantized MoE FFN -- TEST INFRASTRUCTURE ONLY.
 * See oracle.h for the sources and the precision rules. Single-threaded, no
 * blocking, no fusion: each function does one step of the method, in the order
 * the method states it.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Number conversions                                                        */
/* ------------------------------------------------------------------------ */

/* IEEE binary16 bits -> value (exact in double). */
double orc_f16_to_f64(uint16_t h) {
  int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0) v = ldexp((double)m, -24);
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp((double)(m | 1024), e - 25);
  return s ? -v : v;
}

/* float -> binary16, round to nearest even, overflow to infinity. The value is
 * scaled by a power of two (exact in double) so that the kept significand is an
 * integer, and rint() (ties to even in the default rounding mode) rounds it. */
uint16_t orc_f32_to_f16(float f) {
  uint32_t x;
  memcpy(&x, &f, 4);
  uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
  if ((x & 0x7fffffffu) > 0x7f800000u) return (uint16_t)(sign | 0x7e00u);
  double v = fabs((double)f);
  if (v == 0.0) return sign;
  if (v >= 65520.0) return (uint16_t)(sign | 0x7c00u);
  int E;
  frexp(v, &E);
  E -= 1; /* v = 1.f x 2^E */
  if (E < -14) {
    double m = rint(ldexp(v, 24)); /* subnormal: units of 2^-24; 1024 becomes the smallest normal */
    return (uint16_t)(sign | (uint16_t)m);
  }
  double m = rint(ldexp(v, 10 - E)); /* in [1024, 2048] */
  if (m == 2048.0) { m = 1024.0; E += 1; }
  if (E > 15) return (uint16_t)(sign | 0x7c00u);
  return (uint16_t)(sign | (uint16_t)(((E + 15) << 10) | ((int)m - 1024)));
}

uint16_t orc_f32_to_bf16(float f) {
  uint32_t x;
  memcpy(&x, &f, 4);
  if ((x & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((x >> 16) | 0x40u);
  uint32_t lsb = (x >> 16) & 1u;
  x += 0x7fffu + lsb;
  return (uint16_t)(x >> 16);
}

float orc_bf16_to_f32(uint16_t b) {
  uint32_t x = (uint32_t)b << 16;
  float f;
  memcpy(&f, &x, 4);
  return f;
}

/* ------------------------------------------------------------------------ */
/* Block formats                                                             */
/*                                                                          */
/* A matrix [rows x cols] is cut along each row into nb = cols/32 blocks of   */
/* 32 consecutive weights. Two planes:                                        */
/*   codes : block (r, b) at byte (r*nb + b)*Bc, Bc = 8 (FP2), 12 (FP3),       */
/*           16 (FP4);                                                        */
/*   scales: entry r*nb + b, an fp16 (FP2/FP3) or an E8M0 byte (FP4).          */
/* So a block costs 10, 14 or 17 bytes: 2.50, 3.50 and 4.25 bits per weight,  */
/* the ROCmFP2/3/4 sizes. Inside a block (32-bit little-endian words w0..):    */
/*   FP2: element j = 16w + 8h + n has its code at bits 4n+2h .. 4n+2h+1 of w. */
/*   FP3: the low two bits as FP2 in w0, w1; bit 2 of element (w, h, n) at     */
/*        bit 4n + p(w,h) of w2, with p(0,0)=2, p(0,1)=3, p(1,0)=0, p(1,1)=1.  */
/*   FP4: element j has its 4-bit code in nibble j%8 of word j/8.             */
/*   FP3, Packed24 layout (format code 24; the "Packed24 FP3" variant of      */
/*        "deepseek-v4-flash-0731-evox3-rocm", section "The optimization      */
/*        ladder", which names it only): the same 12 bytes, code j at bits   */
/*        3j .. 3j+2 of the block read as one 96-bit little-endian integer,  */
/*        i.e. 8 codes per 24 bits; its fp16 scale plane is FP3's.           */
/* Weight value: scale(r, b) * codebook[code].                                */
/* ------------------------------------------------------------------------ */

#define ORC_FP3_PACKED24 24

static int block_bytes(int fmt) {
  return fmt == 2 ? 8 : fmt == 3 || fmt == ORC_FP3_PACKED24 ? 12 : fmt == 4 ? 16 : -1;
}

/* bits per code of a format code */
static int code_bits(int fmt) { return fmt == ORC_FP3_PACKED24 ? 3 : fmt; }

int orc_packed_bytes(int fmt, int rows, int cols, size_t* code_bytes, size_t* scale_bytes) {
  int bc = block_bytes(fmt);
  if (bc < 0 || rows < 0 || cols < 0 || cols % 32) return ORC_ERR_ARG;
  size_t nblk = (size_t)rows * (size_t)(cols / 32);
  if (code_bytes) *code_bytes = nblk * (size_t)bc;
  if (scale_bytes) *scale_bytes = nblk * (size_t)(fmt == 4 ? 1 : 2);
  return ORC_OK;
}

static uint32_t rd32(const uint8_t* p) {
  return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

static void wr32(uint8_t* p, uint32_t v) {
  p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); p[2] = (uint8_t)(v >> 16); p[3] = (uint8_t)(v >> 24);
}

static const int fp3_p[2][2] = {{2, 3}, {0, 1}}; /* p(w, h) */

static void pack_block(int fmt, const uint8_t* c, uint8_t* out) {
  if (fmt == ORC_FP3_PACKED24) {
    memset(out, 0, 12);
    for (int j = 0; j < 32; j++)
      for (int t = 0; t < 3; t++) {
        int bit = 3 * j + t;
        out[bit / 8] |= (uint8_t)(((c[j] >> t) & 1) << (bit % 8));
      }
  } else if (fmt == 2 || fmt == 3) {
    uint32_t w[2] = {0, 0}, hi = 0;
    for (int j = 0; j < 32; j++) {
      int wi = j >> 4, h = (j >> 3) & 1, n = j & 7;
      w[wi] |= (uint32_t)(c[j] & 3) << (4 * n + 2 * h);
      if (fmt == 3) hi |= (uint32_t)((c[j] >> 2) & 1) << (4 * n + fp3_p[wi][h]);
    }
    wr32(out, w[0]);
    wr32(out + 4, w[1]);
    if (fmt == 3) wr32(out + 8, hi);
  } else {
    for (int wi = 0; wi < 4; wi++) {
      uint32_t w = 0;
      for (int n = 0; n < 8; n++) w |= (uint32_t)(c[8 * wi + n] & 15) << (4 * n);
      wr32(out + 4 * wi, w);
    }
  }
}

static void unpack_block(int fmt, const uint8_t* in, int* c) {
  if (fmt == ORC_FP3_PACKED24) {
    for (int j = 0; j < 32; j++) {
      int v = 0;
      for (int t = 0; t < 3; t++) {
        int bit = 3 * j + t;
        v |= ((in[bit / 8] >> (bit % 8)) & 1) << t;
      }
      c[j] = v;
    }
  } else if (fmt == 2 || fmt == 3) {
    uint32_t w[2] = {rd32(in), rd32(in + 4)};
    uint32_t hi = fmt == 3 ? rd32(in + 8) : 0;
    for (int j = 0; j < 32; j++) {
      int wi = j >> 4, h = (j >> 3) & 1, n = j & 7;
      int v = (int)((w[wi] >> (4 * n + 2 * h)) & 3);
      if (fmt == 3) v |= (int)((hi >> (4 * n + fp3_p[wi][h])) & 1) << 2;
      c[j] = v;
    }
  } else {
    for (int j = 0; j < 32; j++) c[j] = (int)((rd32(in + 4 * (j >> 3)) >> (4 * (j & 7))) & 15);
  }
}

int orc_pack(int fmt, int rows, int cols, const uint8_t* codes, uint8_t* out_codes) {
  int bc = block_bytes(fmt);
  if (bc < 0 || cols % 32 || rows < 0) return ORC_ERR_ARG;
  int nb = cols / 32;
  for (size_t i = 0; i < (size_t)rows * (size_t)cols; i++)
    if (codes[i] >> code_bits(fmt)) return ORC_ERR_ARG;
  for (int r = 0; r < rows; r++)
    for (int b = 0; b < nb; b++)
      pack_block(fmt, codes + (size_t)r * cols + 32 * b, out_codes + ((size_t)r * nb + b) * bc);
  return ORC_OK;
}

int orc_unpack(int fmt, int rows, int cols, const uint8_t* packed, uint8_t* codes_out) {
  int bc = block_bytes(fmt);
  if (bc < 0 || cols % 32 || rows < 0) return ORC_ERR_ARG;
  int nb = cols / 32, c[32];
  for (int r = 0; r < rows; r++)
    for (int b = 0; b < nb; b++) {
      unpack_block(fmt, packed + ((size_t)r * nb + b) * bc, c);
      for (int j = 0; j < 32; j++) codes_out[(size_t)r * cols + 32 * b + j] = (uint8_t)c[j];
    }
  return ORC_OK;
}

/* FP2/FP3: fp16 scale. FP4: E8M0 exponent byte e, value 2^(e-127), e=255 invalid. */
double orc_scale_value(int fmt, const void* scales, size_t i) {
  if (fmt == 4) {
    uint8_t e = ((const uint8_t*)scales)[i];
    return e == 255 ? NAN : ldexp(1.0, (int)e - 127);
  }
  return orc_f16_to_f64(((const uint16_t*)scales)[i]);
}

/* ------------------------------------------------------------------------ */
/* Activation quantization Q8: per 32-block, fp32 arithmetic                  */
/*   amax = max |v|;  d = fp16_rne(amax / 127)  (fp32 division, RN)           */
/*   d == 0  ->  q = 0                                                       */
/*   else r = 1 / float(d) (fp32, RN); q = clamp(rint(v * r), -127, 127)     */
/*   with the product rounded to fp32 and rint ties to even.                  */
/* ------------------------------------------------------------------------ */
void orc_q8(const float* v, int n, int8_t* q, uint16_t* d) {
  for (int b = 0; b < n / 32; b++) {
    const float* blk = v + 32 * b;
    float amax = 0.0f;
    for (int j = 0; j < 32; j++) {
      float a = fabsf(blk[j]);
      if (a > amax) amax = a;
    }
    volatile float dq = amax / 127.0f;
    uint16_t dh = orc_f32_to_f16(dq);
    d[b] = dh;
    float df = (float)orc_f16_to_f64(dh);
    if (df == 0.0f) {
      for (int j = 0; j < 32; j++) q[32 * b + j] = 0;
      continue;
    }
    volatile float r = 1.0f / df;
    for (int j = 0; j < 32; j++) {
      volatile float t = blk[j] * r;
      float rr = rintf(t);
      if (rr > 127.0f) rr = 127.0f;
      if (rr < -127.0f) rr = -127.0f;
      q[32 * b + j] = (int8_t)rr;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* H32: v' = H D v per 32-block, H[i][j] = (-1)^popcount(i & j) (Sylvester,  */
/* unnormalized), D = diag(s), s_i = -1 where bit i of the block's mask is set.*/
/* fp32 form: signs applied, then stages s = 0..4 pair i with i + 2^s (bit s  */
/* of i clear): (a, b) -> (a + b, a - b), each result rounded to fp32.         */
/* ------------------------------------------------------------------------ */
void orc_h32_f32(const float* in, const uint32_t* signs, int nblk, float* out) {
  for (int b = 0; b < nblk; b++) {
    float t[32];
    uint32_t s = signs ? signs[b] : 0u;
    for (int i = 0; i < 32; i++) t[i] = ((s >> i) & 1u) ? -in[32 * b + i] : in[32 * b + i];
    for (int st = 0; st < 5; st++) {
      int bit = 1 << st;
      for (int i = 0; i < 32; i++) {
        if (i & bit) continue;
        volatile float a = t[i], c = t[i | bit];
        volatile float sum = a + c, dif = a - c;
        t[i] = sum;
        t[i | bit] = dif;
      }
    }
    for (int i = 0; i < 32; i++) out[32 * b + i] = t[i];
  }
}

static int popcount32(uint32_t x) {
  int n = 0;
  while (x) { n += (int)(x & 1u); x >>= 1; }
  return n;
}

/* The definition itself: matrix-vector product with H and D, in fp64. */
void orc_h32_f64(const double* in, const uint32_t* signs, int nblk, double* out) {
  for (int b = 0; b < nblk; b++) {
    uint32_t s = signs ? signs[b] : 0u;
    for (int i = 0; i < 32; i++) {
      double acc = 0.0;
      for (int j = 0; j < 32; j++) {
        double hij = (popcount32((uint32_t)(i & j)) & 1) ? -1.0 : 1.0;
        double dj = ((s >> j) & 1u) ? -1.0 : 1.0;
        acc += hij * dj * in[32 * b + j];
      }
      out[32 * b + i] = acc;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Router logit l = sum_h W[h] x[h], bf16 operands (their product is exact in  */
/* fp32), summed in fp32 in the canonical order: 32 partial sums j = 0..31,    */
/* partial j adds the products of k = 256 i + 8 j + t for i = 0..H/256-1,      */
/* t = 0..7 in that order, starting from +0; then five combining rounds with   */
/* distances 16, 8, 4, 2, 1 replace every partial j by (partial j) +           */
/* (partial j^d); the result is partial 0. Requires H % 256 == 0.              */
/* ------------------------------------------------------------------------ */
float orc_router_logit(const uint16_t* x, const uint16_t* w, int H) {
  float acc[32], nxt[32];
  for (int j = 0; j < 32; j++) {
    volatile float a = 0.0f;
    for (int i = 0; i < H / 256; i++)
      for (int t = 0; t < 8; t++) {
        int k = 256 * i + 8 * j + t;
        volatile float p = orc_bf16_to_f32(x[k]) * orc_bf16_to_f32(w[k]);
        a = a + p;
      }
    acc[j] = a;
  }
  for (int d = 16; d >= 1; d >>= 1) {
    for (int j = 0; j < 32; j++) {
      volatile float s = acc[j] + acc[j ^ d];
      nxt[j] = s;
    }
    memcpy(acc, nxt, sizeof acc);
  }
  return acc[0];
}

void orc_router(const uint16_t* x, int T, const uint16_t* Wr, int E, int H, float* logits) {
  for (int t = 0; t < T; t++)
    for (int e = 0; e < E; e++)
      logits[(size_t)t * E + e] = orc_router_logit(x + (size_t)t * H, Wr + (size_t)e * H, H);
}

/* ------------------------------------------------------------------------ */
/* Top-k: the k largest logits, larger value first, equal values by lower      */
/* index; NaN ranks below every number. Weights: softmax over all E logits     */
/* (fp64), p_e = exp(l_e - max) / sum exp(l - max), taken at the chosen        */
/* indices with no renormalization over the k.                                 */
/* ------------------------------------------------------------------------ */
static int ranks_before(float a, int ia, float b, int ib) {
  int na = isnan(a), nb_ = isnan(b);
  if (na != nb_) return nb_;          /* a number beats NaN */
  if (!na && a != b) return a > b;
  return ia < ib;
}

void orc_topk(const float* l, int E, int k, int32_t* idx, double* p) {
  char* taken = (char*)calloc((size_t)E, 1);
  for (int s = 0; s < k; s++) {
    int best = -1;
    for (int e = 0; e < E; e++) {
      if (taken[e]) continue;
      if (best < 0 || ranks_before(l[e], e, l[best], best)) best = e;
    }
    taken[best] = 1;
    idx[s] = best;
  }
  free(taken);
  double m = -INFINITY;
  for (int e = 0; e < E; e++) if (!isnan(l[e]) && (double)l[e] > m) m = (double)l[e];
  double z = 0.0;
  for (int e = 0; e < E; e++) if (!isnan(l[e])) z += exp((double)l[e] - m);
  if (p)
    for (int s = 0; s < k; s++) p[s] = exp((double)l[idx[s]] - m) / z;
}

/* ------------------------------------------------------------------------ */
/* Block-quantized matrix-vector product                                       */
/*   S[r, b] = sum_{j<32} codebook[code(r, 32b+j)] * q[32b+j]   (exact int32)  */
/*   out[r]  = sum_b scale(r, b) * d[b] * S[r, b]               (fp64)         */
/* ------------------------------------------------------------------------ */
int orc_block_partials(const orc_matrix* m, int e, int row, const int8_t* q, int32_t* S) {
  const uint8_t* codes = m->codes[e];
  const int8_t* cb = m->cb[e];
  if (!codes || !cb) return ORC_ERR_MISSING;
  int nb = m->cols / 32, bc = block_bytes(m->fmt), c[32];
  for (int b = 0; b < nb; b++) {
    unpack_block(m->fmt, codes + ((size_t)row * nb + b) * bc, c);
    int32_t s = 0;
    for (int j = 0; j < 32; j++) s += (int32_t)cb[c[j]] * (int32_t)q[32 * b + j];
    S[b] = s;
  }
  return ORC_OK;
}

int orc_matvec(const orc_matrix* m, int e, const int8_t* q, const uint16_t* d, double* out,
               int32_t* S_out) {
  if (!m->codes[e] || !m->scales[e] || !m->cb[e]) return ORC_ERR_MISSING;
  int nb = m->cols / 32;
  int32_t* S = (int32_t*)malloc(sizeof(int32_t) * (size_t)nb);
  for (int r = 0; r < m->rows; r++) {
    orc_block_partials(m, e, r, q, S);
    double acc = 0.0;
    for (int b = 0; b < nb; b++)
      acc += orc_scale_value(m->fmt, m->scales[e], (size_t)r * nb + b) * orc_f16_to_f64(d[b]) *
             (double)S[b];
    out[r] = acc;
    if (S_out) memcpy(S_out + (size_t)r * nb, S, sizeof(int32_t) * (size_t)nb);
  }
  free(S);
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Activation preparation: bf16 x -> fp32 (exact) -> optional H32 -> Q8.      */
/* ------------------------------------------------------------------------ */
static void prep_x(const orc_layer* L, const uint16_t* x, int8_t* xq, uint16_t* xd) {
  int H = L->H;
  float* xf = (float*)malloc(sizeof(float) * (size_t)H);
  for (int i = 0; i < H; i++) xf[i] = orc_bf16_to_f32(x[i]);
  if (L->signs_x) orc_h32_f32(xf, L->signs_x, H / 32, xf);
  orc_q8(xf, H, xq, xd);
  free(xf);
}

/* One expert: g, u = the gate and up rows against (xq, xd); h = silu(g) u with
 * silu(g) = g / (1 + exp(-g)) (fp64); h rounded to fp32, optional H32, Q8 ->
 * (hq, hd); o = down rows against (hq, hd). */
static int expert_ffn(const orc_layer* L, const orc_matrix* G, const orc_matrix* U,
                      const orc_matrix* D, int e, const int8_t* xq, const uint16_t* xd,
                      int slot, orc_trace* tr, double* o) {
  int H = L->H, I = L->I, nbH = H / 32, nbI = I / 32, rc;
  double* g = (double*)malloc(sizeof(double) * (size_t)I);
  double* u = (double*)malloc(sizeof(double) * (size_t)I);
  float* hf = (float*)malloc(sizeof(float) * (size_t)I);
  int8_t* hq = (int8_t*)malloc((size_t)I);
  uint16_t* hd = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)nbI);
  rc = orc_matvec(G, e, xq, xd, g, tr && tr->S_gate ? tr->S_gate + (size_t)slot * I * nbH : NULL);
  if (!rc) rc = orc_matvec(U, e, xq, xd, u, tr && tr->S_up ? tr->S_up + (size_t)slot * I * nbH : NULL);
  if (!rc) {
    for (int r = 0; r < I; r++) {
      double h = g[r] * u[r] / (1.0 + exp(-g[r]));
      hf[r] = (float)h;
      if (tr && tr->g) tr->g[(size_t)slot * I + r] = g[r];
      if (tr && tr->u) tr->u[(size_t)slot * I + r] = u[r];
      if (tr && tr->h) tr->h[(size_t)slot * I + r] = h;
    }
    if (L->signs_h) orc_h32_f32(hf, L->signs_h, nbI, hf);
    orc_q8(hf, I, hq, hd);
    if (tr && tr->hq) memcpy(tr->hq + (size_t)slot * I, hq, (size_t)I);
    if (tr && tr->hd) memcpy(tr->hd + (size_t)slot * nbI, hd, sizeof(uint16_t) * (size_t)nbI);
    const int8_t* useq = hq;
    const uint16_t* used = hd;
    if (tr && tr->force_hq) useq = tr->force_hq + (size_t)slot * I;
    if (tr && tr->force_hd) used = tr->force_hd + (size_t)slot * nbI;
    rc = orc_matvec(D, e, useq, used, o,
                    tr && tr->S_down ? tr->S_down + (size_t)slot * H * nbI : NULL);
  }
  if (!rc && tr && tr->o) memcpy(tr->o + (size_t)slot * H, o, sizeof(double) * (size_t)H);
  free(g); free(u); free(hf); free(hq); free(hd);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* Decode of one token: y = sum_slot p_slot o_slot + o_shared, the sum taken  */
/* in slot order with the shared expert (weight 1) last. The router reads the */
/* unrotated x.                                                                */
/* ------------------------------------------------------------------------ */
int orc_ffn_decode(const orc_layer* L, const uint16_t* x, double* y, orc_trace* tr) {
  int H = L->H, E = L->E, k = L->k, rc = ORC_OK;
  if (H % 256 || L->I % 32 || k < 1 || k > E) return ORC_ERR_ARG;
  int8_t* xq = (int8_t*)malloc((size_t)H);
  uint16_t* xd = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(H / 32));
  float* lg = (float*)malloc(sizeof(float) * (size_t)E);
  int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
  double* p = (double*)malloc(sizeof(double) * (size_t)k);
  double* o = (double*)malloc(sizeof(double) * (size_t)H);
  prep_x(L, x, xq, xd);
  if (tr && tr->xq) memcpy(tr->xq, xq, (size_t)H);
  if (tr && tr->xd) memcpy(tr->xd, xd, sizeof(uint16_t) * (size_t)(H / 32));
  for (int e = 0; e < E; e++) lg[e] = orc_router_logit(x, L->router + (size_t)e * H, H);
  orc_topk(lg, E, k, idx, p);
  if (tr && tr->force_idx) {
    memcpy(idx, tr->force_idx, sizeof(int32_t) * (size_t)k);
    double m = -INFINITY, z = 0.0;
    for (int e = 0; e < E; e++) if ((double)lg[e] > m) m = (double)lg[e];
    for (int e = 0; e < E; e++) z += exp((double)lg[e] - m);
    for (int s = 0; s < k; s++) p[s] = exp((double)lg[idx[s]] - m) / z;
  }
  if (tr && tr->logits) memcpy(tr->logits, lg, sizeof(float) * (size_t)E);
  if (tr && tr->idx) memcpy(tr->idx, idx, sizeof(int32_t) * (size_t)k);
  if (tr && tr->p) memcpy(tr->p, p, sizeof(double) * (size_t)k);
  for (int r = 0; r < H; r++) y[r] = 0.0;
  for (int s = 0; s < k && !rc; s++) {
    rc = expert_ffn(L, &L->gate, &L->up, &L->down, idx[s], xq, xd, s, tr, o);
    for (int r = 0; r < H && !rc; r++) y[r] += p[s] * o[r];
  }
  if (!rc && L->has_shared) {
    rc = expert_ffn(L, &L->sgate, &L->sup, &L->sdown, 0, xq, xd, k, tr, o);
    for (int r = 0; r < H && !rc; r++) y[r] += o[r];
  }
  free(xq); free(xd); free(lg); free(idx); free(p); free(o);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* q=4 verification: four columns, each routed and computed as one decode;    */
/* the optional dense projection is y_dense[c] = W_dense applied to the same  */
/* quantized (and, if configured, rotated) column as the FFN input.           */
/* ------------------------------------------------------------------------ */
int orc_ffn_verify_q4(const orc_layer* L, const orc_matrix* dense, const uint16_t* x, double* y,
                      double* y_dense, orc_trace* tr4) {
  int H = L->H, rc = ORC_OK;
  for (int c = 0; c < 4 && !rc; c++)
    rc = orc_ffn_decode(L, x + (size_t)c * H, y + (size_t)c * H, tr4 ? &tr4[c] : NULL);
  if (!rc && dense && y_dense) {
    int8_t* xq = (int8_t*)malloc((size_t)H);
    uint16_t* xd = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(H / 32));
    for (int c = 0; c < 4 && !rc; c++) {
      prep_x(L, x + (size_t)c * H, xq, xd);
      rc = orc_matvec(dense, 0, xq, xd, y_dense + (size_t)c * dense->rows, NULL);
    }
    free(xq); free(xd);
  }
  return rc;
}

/* Prefill of T tokens: every token is computed as its own decode. */
int orc_ffn_prefill(const orc_layer* L, const uint16_t* x, int T, double* y) {
  int rc = ORC_OK;
  for (int t = 0; t < T && !rc; t++)
    rc = orc_ffn_decode(L, x + (size_t)t * L->H, y + (size_t)t * L->H, NULL);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* RMSNorm with unit weight between stacked layers, rounded to bf16:          */
/*   ss = sum r_k^2 in fp32, each square rounded, in the router's canonical    */
/*        order (32 partials over k = 256 i + 8 j + t, then combining rounds   */
/*        16, 8, 4, 2, 1);                                                     */
/*   ms = ss / H;  den = sqrt(ms + 1e-6);  inv = 1 / den   (fp32, RN each)     */
/*   a_k = bf16_rne(r_k * inv)                                                 */
/* ------------------------------------------------------------------------ */
void orc_rmsnorm_bf16(const float* r, int H, uint16_t* a) {
  float acc[32], nxt[32];
  for (int j = 0; j < 32; j++) {
    volatile float s = 0.0f;
    for (int i = 0; i < H / 256; i++)
      for (int t = 0; t < 8; t++) {
        int k = 256 * i + 8 * j + t;
        volatile float sq = r[k] * r[k];
        s = s + sq;
      }
    acc[j] = s;
  }
  for (int d = 16; d >= 1; d >>= 1) {
    for (int j = 0; j < 32; j++) {
      volatile float s = acc[j] + acc[j ^ d];
      nxt[j] = s;
    }
    memcpy(acc, nxt, sizeof acc);
  }
  volatile float ms = acc[0] / (float)H;
  volatile float den = sqrtf(ms + 1e-6f);
  volatile float inv = 1.0f / den;
  for (int k = 0; k < H; k++) {
    volatile float v = r[k] * inv;
    a[k] = orc_f32_to_bf16(v);
  }
}

/* ------------------------------------------------------------------------ */
/* Codebook quantization of one expert matrix w [rows x cols] fp32 into the  */
/* block formats ("Lucebox x Geometric ...", section "How the model fits on */
/* AMD Strix Halo": learned per-expert codebooks; how they are learned is    */
/* not printed, so this is the library's reading, plain and deterministic):  */
/*  1. block scale d per 32-block, m = max |w| of the block:                 */
/*     FP2/FP3: d = fp16_rne(m / 127) (fp32 division, RN; the Q8 rule),      */
/*              the largest finite fp16 if that overflows;                   */
/*     FP4: E8M0 byte b = e + 127, e the smallest integer with               */
/*          127 * 2^e >= m, clamped to [-127, 127] (m = 0 gives e = -127).   */
/*  2. v = w / d in fp32 (RN); v = 0 where d == 0.                            */
/*  3. histogram of g = clamp(rint(v), -127, 127) over the whole matrix.      */
/*  4. K = 2^fmt int8 entries: entry i starts at the smallest g whose        */
/*     cumulative count exceeds floor((2i+1) N / (2K)) (N weights); then 8    */
/*     Lloyd steps on the histogram, exact in integers: each grid value goes  */
/*     to its nearest entry (ties to the lower index), each entry with a     */
/*     non-empty cell becomes floor((2 S + n) / (2 n)) (S the cell's sum of  */
/*     g, n its count: the mean rounded half up), then the entries are       */
/*     sorted ascending.                                                     */
/*  5. code of each weight = the entry nearest to v, |v - c| in fp32, ties   */
/*     to the lower index.                                                   */
/* Outputs: codes [rows x cols] one per byte, scales [rows x cols/32] (fp16  */
/* bits or E8M0 bytes), cb [2^fmt].                                          */
/* ------------------------------------------------------------------------ */
static int64_t floor_div64(int64_t a, int64_t b) { /* b > 0 */
  int64_t q = a / b;
  if ((a % b) != 0 && a < 0) q -= 1;
  return q;
}

static float block_scale_q(int fmt, const float* blk, void* scales, size_t i) {
  float m = 0.0f;
  for (int j = 0; j < 32; j++) {
    float a = fabsf(blk[j]);
    if (a > m) m = a;
  }
  if (fmt == 4) {
    int e = -127;
    while (e < 127 && ldexp(127.0, e) < (double)m) e++;
    ((uint8_t*)scales)[i] = (uint8_t)(e + 127);
    return (float)ldexp(1.0, e);
  }
  volatile float dq = m / 127.0f;
  uint16_t dh = orc_f32_to_f16(dq);
  if ((dh & 0x7C00u) == 0x7C00u) dh = 0x7BFFu; /* overflow: the largest finite fp16 */
  ((uint16_t*)scales)[i] = dh;
  return (float)orc_f16_to_f64(dh);
}

int orc_quantize_expert(int fmt, int rows, int cols, const float* w, uint8_t* codes, void* scales,
                        int8_t* cb) {
  if (fmt < 2 || fmt > 4) return ORC_ERR_ARG;
  if (rows <= 0 || cols <= 0 || cols % 32) return ORC_ERR_ARG;
  const int K = 1 << fmt, nb = cols / 32;
  int64_t hist[255] = {0};
  const size_t N = (size_t)rows * cols;
  float* v = (float*)malloc(N * sizeof(float));
  if (!v) return ORC_ERR_ARG;
  for (int r = 0; r < rows; r++)
    for (int b = 0; b < nb; b++) {
      const size_t o = (size_t)r * cols + 32 * b;
      const float d = block_scale_q(fmt, w + o, scales, (size_t)r * nb + b);
      for (int j = 0; j < 32; j++) {
        volatile float t = d == 0.0f ? 0.0f : w[o + j] / d;
        v[o + j] = t;
        float g = rintf(t);
        if (g > 127.0f) g = 127.0f;
        if (g < -127.0f) g = -127.0f;
        hist[(int)g + 127]++;
      }
    }
  int64_t c[16];
  for (int i = 0; i < K; i++) {
    const int64_t t = ((2 * (int64_t)i + 1) * (int64_t)N) / (2 * (int64_t)K);
    int64_t cum = 0;
    int g = 0;
    for (; g < 255; g++) {
      cum += hist[g];
      if (cum > t) break;
    }
    c[i] = g - 127;
  }
  for (int it = 0; it < 8; it++) {
    int64_t S[16] = {0}, n[16] = {0};
    for (int g = 0; g < 255; g++) {
      if (!hist[g]) continue;
      const int64_t x = g - 127;
      int best = 0;
      int64_t bd = llabs(x - c[0]);
      for (int i = 1; i < K; i++) {
        const int64_t dd = llabs(x - c[i]);
        if (dd < bd) { bd = dd; best = i; }
      }
      S[best] += hist[g] * x;
      n[best] += hist[g];
    }
    for (int i = 0; i < K; i++)
      if (n[i]) c[i] = floor_div64(2 * S[i] + n[i], 2 * n[i]);
    for (int i = 1; i < K; i++) /* insertion sort, ascending */
      for (int j = i; j > 0 && c[j - 1] > c[j]; j--) {
        int64_t tmp = c[j]; c[j] = c[j - 1]; c[j - 1] = tmp;
      }
  }
  for (int i = 0; i < K; i++) cb[i] = (int8_t)c[i];
  for (size_t o = 0; o < N; o++) {
    int best = 0;
    float bd = fabsf(v[o] - (float)c[0]);
    for (int i = 1; i < K; i++) {
      const float dd = fabsf(v[o] - (float)c[i]);
      if (dd < bd) { bd = dd; best = i; }
    }
    codes[o] = (uint8_t)best;
  }
  free(v);
  return ORC_OK;
}
