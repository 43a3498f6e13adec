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


def requant_bound(L: O.Layer, idx, p, hq_a, hd_a, hq_b, hd_b) -> np.ndarray:
    """D_r = sum_slot p_slot sum_k |w_down[r,k]| |h~a_k - h~b_k|: how far the
    down projection and combine of two quantized h (the GPU's and the oracle's
    own) can move y apart, in exact arithmetic."""
    slots = [(L.down, int(e)) for e in idx]
    if L.shared is not None:
        slots.append((L.shared[2], 0))
    w = list(p) + ([1.0] if L.shared is not None else [])
    D = np.zeros(L.H)
    for s, (m, e) in enumerate(slots):
        ta = hq_a[s].astype(np.float64) * np.repeat(O.f16_array_to_f64(hd_a[s]), 32)
        tb = hq_b[s].astype(np.float64) * np.repeat(O.f16_array_to_f64(hd_b[s]), 32)
        dh = np.abs(ta - tb)
        nz = np.nonzero(dh)[0]
        if nz.size:  # only the columns where the two differ
            codes = O.unpack(m.fmt, m.rows, m.cols, m.codes[e])[:, nz]
            sv = O.scale_values(m.fmt, m.scales[e]).reshape(m.rows, m.cols // 32)[:, nz // 32]
            D += w[s] * (np.abs(sv * m.cb[e].astype(np.float64)[codes]) @ dh[nz])
    return D


def check_independent(y_gpu, y_ora, bound, requant, what=""):
    """y against the independent fp64 oracle: the teacher-forced bound widened
    by requant_bound (the part of the difference that comes from the two sides
    quantizing their own h)."""
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ora)
    lim = ELEM * bound + requant
    worst = np.max(err / np.maximum(lim, 1e-300))
    rel = np.linalg.norm(y_gpu - y_ora) / max(np.linalg.norm(y_ora), 1e-300)
    rel_lim = REL_L2 + np.linalg.norm(requant) / max(np.linalg.norm(y_ora), 1e-300)
    assert np.all(err <= lim), f"{what}: max |err| / (2e-3 B + D) = {worst:.3g} > 1"
    assert rel <= rel_lim, f"{what}: relative L2 {rel:.3g} > {rel_lim:.3g}"
    return worst, rel


def check_output(y_gpu, y_ref, bound, what=""):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref)
    worst = np.max(err / np.maximum(bound, 1e-300))
    rel = np.linalg.norm(y_gpu - y_ref) / max(np.linalg.norm(y_ref), 1e-300)
    assert np.all(err <= ELEM * bound), f"{what}: max |err|/B = {worst:.3g} > {ELEM}"
    assert rel <= REL_L2, f"{what}: relative L2 {rel:.3g} > {REL_L2}"
    return worst, rel


# Share of h elements whose int8 code may differ between the GPU's
# quantization and the fp64 oracle's own (each side quantizes its own h; the
# GPU's h is checked against the oracle's quantizer bit for bit regardless).
# Decode and q=4 sum exact int32 block partials in fp32: 0.1 %. The prefill's
# tensor-core operands carry code x scale in two bf16 parts (what they leave
# out, with the low x low product, is below 8 * 2^-18 of |w x| per product,
# tests/test_prefill_split_bound.py), so its h differs from the oracle's by a
# few 1e-5 relative and 0.1-0.2 % of the codes flip (measured): 1 %.
FLIPS_DECODE = 1e-3
FLIPS_PREFILL = 1e-2
# Absolute tolerance of h, as a fraction of the token's max |h|: the prefill's
# operand parts leave out up to 8 * 2^-18 (3.1e-5) of |w x| per product
# (tests/test_prefill_split_bound.py), so g and u err by a fraction of
# sum |w x|, i.e. of the largest h rather than of each element.
H_ATOL_DECODE = 2e-6
H_ATOL_PREFILL = 1e-4
# Per-slot output o against the oracle's, as a fraction of the slot's bound
# sum |w x|: the decode's block sums are exact integers (fp32 rounding only);
# the prefill's tensor-core operands leave out at most 8 * 2^-18 (3.1e-5) of
# |w x| per product (the two split residuals, each below 2^-17, and the
# low x low product, below 2^-16), plus fp32 rounding.
O_REL_DECODE = 1e-5
O_REL_PREFILL = 4e-5
PREFILL = dict(flip_frac=FLIPS_PREFILL, h_atol=H_ATOL_PREFILL, o_rel=O_REL_PREFILL)


def check_token(L, cfg, x_row, y, g, partials, flip_frac=FLIPS_DECODE, h_atol=H_ATOL_DECODE,
                o_rel=O_REL_DECODE):
    """Stage-by-stage parity of one token's decode intermediates g (one
    column's view of the debug buffers) and output y against the oracle.
    Returns the independent oracle output, the bound B and whether the GPU's
    quantized h equals the oracle's."""
    H, I, k = cfg["H"], cfg["I"], cfg["k"]
    ns = k + (1 if cfg["shared_fmt"] else 0)
    yo, tr = O.ffn_decode(L, x_row, trace=True, partials=partials)
    np.testing.assert_array_equal(g["xq"], tr["xq"])
    np.testing.assert_array_equal(g["xd"], tr["xd"])
    np.testing.assert_array_equal(g["logits"], tr["logits"])
    np.testing.assert_array_equal(g["idx"], tr["idx"])
    np.testing.assert_allclose(g["p"], tr["p"], rtol=2e-6)
    h = g["h"].reshape(ns, I)
    np.testing.assert_allclose(h, tr["h"][:ns], rtol=2e-4, atol=h_atol * np.abs(tr["h"][:ns]).max())
    # quantization decision: the oracle's quantizer on the GPU's h, bit for bit
    hq = g["hq"].reshape(ns, I)
    hd = g["hd"].reshape(ns, I // 32)
    for s in range(ns):
        hh = h[s]
        if L.signs_h is not None:
            hh = O.h32_f32(hh, L.signs_h)
        q, d = O.q8(hh)
        np.testing.assert_array_equal(hq[s], q)
        np.testing.assert_array_equal(hd[s], d)
    # independent quantization differs at most by one step, on rare elements
    diff = np.abs(hq.astype(int) - tr["hq"][:ns].astype(int))
    assert diff.max() <= 1 and (diff > 0).sum() <= max(2, flip_frac * diff.size)
    # teacher-forced down projection: bit-exact partials, tight y
    yt, tt = O.ffn_decode(L, x_row, trace=True, partials=partials, force_hq=hq, force_hd=hd)
    if partials:
        np.testing.assert_array_equal(g["S_gate"].reshape(ns, I, H // 32), tr["S_gate"][:ns])
        np.testing.assert_array_equal(g["S_up"].reshape(ns, I, H // 32), tr["S_up"][:ns])
        np.testing.assert_array_equal(g["S_down"].reshape(ns, H, I // 32), tt["S_down"][:ns])
    B = output_bound(L, tr["idx"], tr["p"], hq, hd)
    o = g["o"].reshape(ns, H)
    for s, bs in enumerate(slot_bounds(L, tr["idx"], hq, hd)):
        err = np.abs(o[s] - tt["o"][s])
        assert np.all(err <= o_rel * bs), f"o[{s}]: max err/bound {np.max(err / bs):.3g}"
    check_output(y, yt, B, "y (teacher-forced)")
    same_q = np.array_equal(hq, tr["hq"][:ns]) and np.array_equal(hd, tr["hd"][:ns])
    # and against the independent oracle output
    D = requant_bound(L, tr["idx"], tr["p"], hq, hd, tr["hq"][:ns], tr["hd"][:ns])
    check_independent(y, yo, B, D, "y (independent)")
    return yo, B, same_q


def column_view(g, cfg, c):
    """The debug buffers of column c of a multi-column call, shaped like a
    single-token decode's."""
    H, I, E, k = cfg["H"], cfg["I"], cfg["E"], cfg["k"]
    ns = k + (1 if cfg["shared_fmt"] else 0)
    per = dict(xq=H, xd=H // 32, logits=E, idx=k, p=k, h=ns * I, hq=ns * I, hd=ns * I // 32,
               o=ns * H, S_gate=ns * I * H // 32, S_up=ns * I * H // 32, S_down=ns * H * I // 32)
    return {n: v[c * per[n]:(c + 1) * per[n]] for n, v in g.items()}
