// Workspace layouts of the FFN entry points (host and device agree on them).
// Every region starts on a 256-byte boundary of the caller's workspace.
#pragma once

#include <stddef.h>

namespace moeq {

constexpr int kMaxTopK = 8;

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Counter words of the persistent decode / verify kernels.
//   [0] unit queue  [1] router units done  [2] CTAs finished
//   [8 + s] quantized 32-blocks of h done for slot s
//   [kPairBase ...]  one word per (slot, 32-block of h): halves written
//   [after pairs ...] one word per 32-row chunk of y: slot outputs written
constexpr int kCtrHqDone = 8;
constexpr int kPairBase = 48;

struct DecodeWs {
  int nslots;
  size_t ctr, n_ctr, logits, hbuf, hq, hd, obuf, total;
};

inline DecodeWs decode_ws_layout(int H, int I, int E, int k, int has_shared, int cols = 1) {
  DecodeWs w;
  // cols > 1 (q=4 verification): one slot per (column, routed choice) plus the shared expert
  // per column; slot bookkeeping is the same.
  w.nslots = cols * (k + (has_shared ? 1 : 0));
  size_t off = 0;
  w.ctr = off;
  w.n_ctr = kPairBase + static_cast<size_t>(w.nslots) * (I / 32) + static_cast<size_t>(cols) * (H / 32);
  off += align256(4 * w.n_ctr);
  w.logits = off;
  off += align256(4 * static_cast<size_t>(cols) * E);
  w.hbuf = off;
  off += align256(4 * static_cast<size_t>(w.nslots) * I);
  w.hq = off;
  off += align256(static_cast<size_t>(w.nslots) * I);
  w.hd = off;
  off += align256(2 * static_cast<size_t>(w.nslots) * (I / 32));
  w.obuf = off;
  off += align256(4 * static_cast<size_t>(w.nslots) * H);
  w.total = off;
  return w;
}

inline DecodeWs verify_ws_layout(int H, int I, int E, int k, int has_shared) {
  return decode_ws_layout(H, I, E, k, has_shared, 4);
}

// Prefill workspace for up to T tokens.
struct PrefillWs {
  size_t xq, xd, idx, p, counts, offsets, perm, pos, hq, hd, o, total;
};

inline PrefillWs prefill_ws_layout(int H, int I, int E, int k, int has_shared, int T) {
  PrefillWs w;
  const size_t Tk = static_cast<size_t>(T) * k;
  const size_t rows = Tk + (has_shared ? static_cast<size_t>(T) : 0);  // grouped rows incl. shared
  const int groups = E + (has_shared ? 1 : 0);
  size_t off = 0;
  w.xq = off;      off += align256(static_cast<size_t>(T) * H);
  w.xd = off;      off += align256(2 * static_cast<size_t>(T) * (H / 32));
  w.idx = off;     off += align256(4 * Tk);
  w.p = off;       off += align256(4 * Tk);
  w.counts = off;  off += align256(4 * static_cast<size_t>(groups + 1) * 2);
  w.offsets = off; off += align256(4 * static_cast<size_t>(groups + 1));
  w.perm = off;    off += align256(4 * rows);
  w.pos = off;     off += align256(4 * Tk);
  w.hq = off;      off += align256(rows * I);
  w.hd = off;      off += align256(2 * rows * (I / 32));
  w.o = off;       off += align256(4 * rows * H);
  w.total = off;
  return w;
}

}  // namespace moeq
