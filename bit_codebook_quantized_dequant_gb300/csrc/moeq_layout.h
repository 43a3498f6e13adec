// Workspace layouts of the FFN entry points (host and device agree on them).
// Every region starts on a 256-byte boundary of the caller's workspace.
#pragma once

#include <stddef.h>

#ifdef __CUDACC__
#define MOEQ_HD __host__ __device__
#else
#define MOEQ_HD
#endif

namespace moeq {

constexpr int kMaxTopK = 8;

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Counter words of the persistent decode / verify kernels. Every counter that
// many CTAs poll or update has its own 128-byte line:
//   kCtrQueue      work queue (items taken)
//   kCtrRouter     router items done
//   kCtrDownDone   down items done
//   kCtrDone       CTAs finished (the last one resets the counters)
//   kCtrHqDone + kCtrLine * u   quantized 32-blocks of h of unit u
// followed by kRouteCopies copies of the routing record, every copy read by a
// few CTAs only. A record is route_lines(cols) lines with a ready flag in the
// last word, stored with release semantics after the rest of the record:
//   1 column:  idx[8], p[8] (fp32 bits) in one line;
//   4 columns: idx[c*8 + j], then p[c*8 + j], then the unit words, then the
//              unit count in word 0 of the last line.
constexpr int kCtrLine = 32;  // words per 128-byte line
constexpr int kCtrQueue = 0;
constexpr int kCtrRouter = 1 * kCtrLine;
constexpr int kCtrDownDone = 2 * kCtrLine;
constexpr int kCtrDone = 3 * kCtrLine;
constexpr int kCtrHqDone = 4 * kCtrLine;
constexpr int kRouteCopies = 16;
constexpr int kRouteFlag = kCtrLine - 1;
MOEQ_HD inline constexpr int route_lines(int cols) { return cols == 1 ? 1 : 4; }
MOEQ_HD inline constexpr int route_base(int max_units) { return kCtrHqDone + kCtrLine * max_units; }
MOEQ_HD inline constexpr int ctr_words(int max_units, int cols) {
  return route_base(max_units) + kCtrLine * kRouteCopies * route_lines(cols);
}

// Bytes between the fp16 scales of consecutive h vectors (16-byte multiple so
// that they can be moved with bulk copies).
inline size_t hd_stride(int I) { return (2 * static_cast<size_t>(I / 32) + 15) & ~static_cast<size_t>(15); }

// Decode (cols = 1) and q=4 verification (cols = 4). A "unit" is one expert
// whose weights are read once: up to cols*k distinct routed experts, then the
// shared expert at index cols*k. h and the expert outputs are kept per (unit,
// column): vector u*cols + c.
struct DecodeWs {
  int nunits, nvec;
  size_t ctr, n_ctr, logits, hq, hd, obuf, total;
};

inline DecodeWs decode_ws_layout(int H, int I, int E, int k, int has_shared, int cols = 1) {
  DecodeWs w;
  w.nunits = cols * k + (has_shared ? 1 : 0);
  w.nvec = w.nunits * cols;
  size_t off = 0;
  w.ctr = off;
  w.n_ctr = static_cast<size_t>(ctr_words(w.nunits, cols));
  off += align256(4 * w.n_ctr);
  w.logits = off;
  off += align256(4 * static_cast<size_t>(cols) * E);
  w.hq = off;
  off += align256(static_cast<size_t>(w.nvec) * I);
  w.hd = off;
  off += align256(hd_stride(I) * static_cast<size_t>(w.nvec));
  w.obuf = off;
  off += align256(4 * static_cast<size_t>(w.nvec) * H);
  w.total = off;
  return w;
}

inline DecodeWs verify_ws_layout(int H, int I, int E, int k, int has_shared) {
  return decode_ws_layout(H, I, E, k, has_shared, 4);
}

// Prefill workspace for up to T tokens. Groups: the E routed experts, then
// the shared expert (if any). Grouped rows: the (token, slot) pairs of every
// routed expert in a stable order (ascending token, then slot), then the T
// rows of the shared expert. pid[row] = token * k + slot for routed rows and
// T * k + token for shared rows; pos[token * k + slot] = its row.
// The tensor-core GEMMs read the activations in grouped order as two bf16
// parts of (code x block scale): xhi / xlo [rows x H] for x, hhi / hlo
// [rows x I] for h; g [rows x I] fp32 holds the gate projection between the
// gate and the up GEMM.
struct PrefillWs {
  size_t xq, xd, idx, p, counts, offsets, tiles_gu, tiles_dn, pid, pos, xhi, xlo, g, hhi, hlo, o, total;
};

inline PrefillWs prefill_ws_layout(int H, int I, int E, int k, int has_shared, int T) {
  PrefillWs w;
  const size_t Tk = static_cast<size_t>(T) * k;
  const size_t rows = Tk + (has_shared ? static_cast<size_t>(T) : 0);
  const size_t groups = static_cast<size_t>(E) + (has_shared ? 1 : 0);
  size_t off = 0;
  w.xq = off;       off += align256(static_cast<size_t>(T) * H);
  w.xd = off;       off += align256(2 * static_cast<size_t>(T) * (H / 32));
  w.idx = off;      off += align256(4 * Tk);
  w.p = off;        off += align256(4 * Tk);
  w.counts = off;   off += align256(4 * (groups + 1));
  w.offsets = off;  off += align256(4 * (groups + 1));
  w.tiles_gu = off; off += align256(4 * (groups + 1));
  w.tiles_dn = off; off += align256(4 * (groups + 1));
  w.pid = off;      off += align256(4 * rows);
  w.pos = off;      off += align256(4 * Tk);
  w.xhi = off;      off += align256(2 * rows * H);
  w.xlo = off;      off += align256(2 * rows * H);
  w.g = off;        off += align256(4 * rows * I);
  w.hhi = off;      off += align256(2 * rows * I);
  w.hlo = off;      off += align256(2 * rows * I);
  w.o = off;        off += align256(4 * rows * H);
  w.total = off;
  return w;
}

}  // namespace moeq
