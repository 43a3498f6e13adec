"""Helpers shared by the GPU parity tests: oracle-side layers for the tokens a
test uses, and the FFN output tolerance

    |y - y*| <= 2e-3 * B_r,   B_r = sum_slot p_slot * sum_k |w_down[r,k]| |h~_k|
                                   + sum_k |w_sdown[r,k]| |h~s_k|

with h~ the dequantized quantized h, plus relative L2 <= 1e-4 per token."""
from __future__ import annotations

import numpy as np

import oracle as O
from oracle import workload as W
from bit_codebook_quantized_dequant_gb300 import synth as S

REL_L2 = 1e-4
ELEM = 2e-3


def host_layer_for(seed, layer_idx, cfg, x_tokens):
    """Oracle layer with the experts any of the tokens routes to."""
    experts = set()
    for t in range(x_tokens.shape[0]):
        idx, _ = O.topk(O.router_logits(x_tokens[t], S.router_weights(seed, layer_idx, cfg))[0],
                        cfg["k"])
        experts.update(int(e) for e in idx)
    return W.layer(seed, layer_idx, cfg, experts)


def _abs_dense(m: O.Matrix, e: int) -> np.ndarray:
    codes = O.unpack(m.fmt, m.rows, m.cols, m.codes[e])
    sv = O.scale_values(m.fmt, m.scales[e]).reshape(m.rows, m.cols // 32)
    return np.abs(np.repeat(sv, 32, axis=1) * m.cb[e].astype(np.float64)[codes])


def slot_bounds(L: O.Layer, idx, hq, hd):
    """sum_k |w_down[r,k]| |h~_k| for every slot (routed slots, then the shared one)."""
    out = []
    slots = [(L.down, int(e)) for e in idx]
    if L.shared is not None:
        slots.append((L.shared[2], 0))
    for s, (m, e) in enumerate(slots):
        ht = np.abs(hq[s].astype(np.float64) * np.repeat(O.f16_array_to_f64(hd[s]), 32))
        out.append(_abs_dense(m, e) @ ht)
    return out


def output_bound(L: O.Layer, idx, p, hq, hd) -> np.ndarray:
    """B_r for one token given its routing and quantized h per slot."""
    b = slot_bounds(L, idx, hq, hd)
    w = list(p) + ([1.0] if L.shared is not None else [])
    return sum(wi * bi for wi, bi in zip(w, b))


def check_output(y_gpu, y_ref, bound, what=""):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref)
    worst = np.max(err / np.maximum(bound, 1e-300))
    rel = np.linalg.norm(y_gpu - y_ref) / max(np.linalg.norm(y_ref), 1e-300)
    assert np.all(err <= ELEM * bound), f"{what}: max |err|/B = {worst:.3g} > {ELEM}"
    assert rel <= REL_L2, f"{what}: relative L2 {rel:.3g} > {REL_L2}"
    return worst, rel
