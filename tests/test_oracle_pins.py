"""Pins of the CPU oracle against facts that do not come from the oracle itself:
hand-derived bytes and values (tests/golden), library routines (numpy float16,
torch bfloat16, scipy's Hadamard matrix and softmax), closed forms, invariants
and brute force on tiny inputs. CPU only."""
import os

import numpy as np
import pytest
import scipy.linalg
import scipy.special
import torch

import oracle as O
from oracle import workload as W
from bit_codebook_quantized_dequant_gb300 import synth as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                yield [s.strip() for s in line.split("|")]


# ----------------------------------------------------------------- number formats
def test_f16_conversion_matches_numpy():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 6, 4000),
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9, 2.0 ** -24, 2.0 ** -25,
                  3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 6.1e-5, 1e-4, 1e-2],
                 dtype=np.float32)])
    # exact ties of the fp16 grid: odd multiples of half an fp16 ulp
    ties = (np.arange(1, 400, 2, dtype=np.float64) * 2.0 ** -11 + 1.0).astype(np.float32)
    vals = np.concatenate([vals, ties, -ties])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([O.f32_to_f16(v) for v in vals], dtype=np.uint16)
    np.testing.assert_array_equal(got, ref)
    back = O.f16_array_to_f64(ref)
    np.testing.assert_array_equal(back, ref.view(np.float16).astype(np.float64))


def test_bf16_conversion_matches_torch():
    rng = np.random.default_rng(2)
    vals = (rng.standard_normal(5000) * 10.0 ** rng.integers(-20, 20, 5000)).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([O.f32_to_bf16(v) for v in vals], dtype=np.uint16)
    np.testing.assert_array_equal(got, ref)
    # the generator's vectorized conversion agrees with the same library rounding
    np.testing.assert_array_equal(S.f32_to_bf16_bits(vals), ref)


def test_scale_values():
    e8 = np.array([127, 120, 114, 0, 254], dtype=np.uint8)
    np.testing.assert_array_equal(O.scale_values(4, e8), [1.0, 2.0 ** -7, 2.0 ** -13, 2.0 ** -127,
                                                         2.0 ** 127])
    f16 = np.array([0x3C00, 0x068E, 0x211F, 0x0001, 0xBC00], dtype=np.uint16)
    np.testing.assert_array_equal(O.scale_values(2, f16), f16.view(np.float16).astype(np.float64))


# ----------------------------------------------------------------- packing
@pytest.mark.parametrize("fmt", [2, 3, 4, 24])
def test_pack_roundtrip_and_sizes(fmt):
    for rows, cols in [(1, 32), (3, 128), (17, 256), (5, 4096)]:
        c = S.codes(7, fmt * 100 + rows, S.code_bits(fmt), rows, cols)
        p = O.pack(fmt, c)
        nb = rows * cols // 32
        cb, sb = O.packed_bytes(fmt, rows, cols)
        assert cb == nb * {2: 8, 3: 12, 4: 16, 24: 12}[fmt]
        assert cb + sb == nb * {2: 10, 3: 14, 4: 17, 24: 14}[fmt]
        assert p.size == cb
        np.testing.assert_array_equal(O.unpack(fmt, rows, cols, p), c)


def test_pack_golden_bytes():
    n = 0
    for fmt, expr, hexbytes in _golden_lines("pack_patterns.txt"):
        c = np.array([[eval(expr, {"j": j}) for j in range(32)]], dtype=np.uint8)
        assert O.pack(int(fmt), c).tobytes().hex() == hexbytes, (fmt, expr)
        n += 1
    assert n >= 9


def test_packed24_bytes_against_a_96_bit_integer():
    """Packed24: each block equals sum_j code_j * 8^j written as a 12-byte
    little-endian integer (Python integers, not the oracle's bit loop), for
    random codes over several blocks and rows."""
    c = S.codes(9, 2424, 3, 7, 256)
    p = O.pack(24, c).reshape(7, 8, 12)
    for r in range(7):
        for b in range(8):
            v = sum(int(c[r, 32 * b + j]) << (3 * j) for j in range(32))
            assert p[r, b].tobytes() == v.to_bytes(12, "little")
    with pytest.raises(RuntimeError):
        bad = np.zeros((1, 32), dtype=np.uint8)
        bad[0, 3] = 8
        O.pack(24, bad)


def test_pack_rejects_out_of_range_codes():
    c = np.zeros((1, 32), dtype=np.uint8)
    c[0, 5] = 4
    with pytest.raises(RuntimeError):
        O.pack(2, c)


def test_generator_distributions():
    cb = S.codebook(3, 11, 4)
    assert cb.size == 16 and np.all(np.diff(cb.astype(int)) > 0)
    assert cb.min() >= -127 and cb.max() <= 127
    c = S.codes(3, 12, 3, 64, 256)
    counts = np.bincount(c.ravel(), minlength=8)
    assert counts.size == 8 and counts.min() > 0.8 * c.size / 8
    sc = S.scales_f16(3, 13, 100000).view(np.float16).astype(np.float64)
    assert sc.min() >= 1e-4 * (1 - 1e-3) and sc.max() <= 1e-2 * (1 + 1e-3)
    assert abs(np.median(np.log10(sc)) + 3.0) < 0.15      # log-uniform median near 1e-3
    e = S.scales_e8m0(3, 14, 10000).astype(int) - 127
    assert e.min() == -13 and e.max() == -7
    x = S.bf16_bits_to_f32(S.normal_bf16(3, 15, 200000)).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    # rows drawn alone equal the same rows drawn with the whole matrix
    np.testing.assert_array_equal(S.codes_rows(3, 12, 3, 256, 10, 5), c[10:15])
    np.testing.assert_array_equal(S.tokens(3, S.WORKLOADS["tiny-decode"], 3, start=4),
                                  S.tokens(3, S.WORKLOADS["tiny-decode"], 8)[4:7])


# ----------------------------------------------------------------- Q8
def test_q8_zero_block_and_single_value():
    q, d = O.q8(np.zeros(64, np.float32))
    assert np.all(q == 0) and np.all(d == 0)
    v = np.zeros(32, np.float32)
    v[5] = -3.25
    q, d = O.q8(v)
    assert q[5] == -127 and np.all(np.delete(q, 5) == 0)
    assert d[0] == np.float16(np.float32(3.25) / np.float32(127.0)).view(np.uint16)


def test_q8_ties_go_to_even():
    # amax = 15.875 -> d = 0.125 exactly (fp16 0x3000), 1/d = 8, so v*8 = k + 0.5 exactly
    v = np.zeros(32, np.float32)
    v[0] = 15.875
    halves = [0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, 126.5]
    for i, h in enumerate(halves):
        v[1 + i] = h / 8.0
    q, d = O.q8(v)
    assert d[0] == 0x3000
    assert q[0] == 127
    assert list(q[1:1 + len(halves)]) == [0, 2, 2, 4, 0, -2, -2, 126]


def test_q8_matches_library_rounding_on_random_blocks():
    rng = np.random.default_rng(4)
    v = (rng.standard_normal(32 * 500) * 10.0 ** rng.integers(-4, 4, 32 * 500)).astype(np.float32)
    q, d = O.q8(v)
    vb = v.reshape(-1, 32)
    amax = np.abs(vb).max(axis=1)
    dd = (amax / np.float32(127.0)).astype(np.float32).astype(np.float16)
    np.testing.assert_array_equal(d, dd.view(np.uint16))
    r = (np.float32(1.0) / dd.astype(np.float32)).astype(np.float32)
    qq = np.clip(np.rint((vb * r[:, None]).astype(np.float32)), -127, 127).astype(np.int8)
    np.testing.assert_array_equal(q.reshape(-1, 32), qq)
    # dequantized error is within half a step of every block
    err = np.abs(q.reshape(-1, 32) * dd.astype(np.float64)[:, None] - vb)
    assert np.all(err <= 0.5 * dd.astype(np.float64)[:, None] * (1 + 1e-3) + 1e-30)


# ----------------------------------------------------------------- H32
def test_h32_is_sylvester_hadamard():
    eye = np.eye(32)
    M = np.stack([O.h32_f64(eye[j], None) for j in range(32)], axis=1)
    np.testing.assert_array_equal(M, scipy.linalg.hadamard(32))
    np.testing.assert_array_equal(M @ M, 32 * np.eye(32))
    Mf = np.stack([O.h32_f32(eye[j].astype(np.float32), None) for j in range(32)], axis=1)
    np.testing.assert_array_equal(Mf, M)


def test_h32_signs_and_rotation_invariance():
    rng = np.random.default_rng(5)
    s = S.signs(9, 1, 4)
    D = np.array([[-1.0 if (int(s[b]) >> i) & 1 else 1.0 for i in range(32)] for b in range(4)])
    x = rng.standard_normal(128)
    w = rng.standard_normal(128)
    hx = O.h32_f64(x, s)
    Hm = scipy.linalg.hadamard(32)
    ref = np.concatenate([Hm @ (D[b] * x[32 * b:32 * b + 32]) for b in range(4)])
    np.testing.assert_allclose(hx, ref, rtol=0, atol=1e-12)
    hw = O.h32_f64(w, s)
    assert abs(hx @ hw - 32.0 * (x @ w)) <= 1e-10 * 32 * np.abs(x) @ np.abs(w)
    # fp32 butterfly is exact on small integers and equals the matrix form
    xi = rng.integers(-1000, 1000, 128).astype(np.float32)
    np.testing.assert_array_equal(O.h32_f32(xi, s), O.h32_f64(xi.astype(np.float64), s))
    # twice without signs: 32 x input
    np.testing.assert_array_equal(O.h32_f32(O.h32_f32(xi, None), None), 32 * xi)


# ----------------------------------------------------------------- router
def test_router_exact_on_integer_inputs():
    rng = np.random.default_rng(6)
    H, E = 1024, 8
    xi = rng.integers(-8, 9, H).astype(np.float32)
    wi = rng.integers(-8, 9, (E, H)).astype(np.float32)
    lg = O.router_logits(S.f32_to_bf16_bits(xi), S.f32_to_bf16_bits(wi))[0]
    exact = wi.astype(np.int64) @ xi.astype(np.int64)
    np.testing.assert_array_equal(lg.astype(np.int64), exact)


def test_router_order_golden():
    n = 0
    for H, entries, expect in _golden_lines("router_order.txt"):
        H = int(H)
        x = np.zeros(H, np.float32)
        w = np.zeros(H, np.float32)
        for ent in entries.split():
            k, xv, wv = ent.split(":")
            x[int(k)] = float(xv)
            w[int(k)] = float(wv)
        lg = O.router_logits(S.f32_to_bf16_bits(x), S.f32_to_bf16_bits(w)[None, :])
        assert lg[0, 0] == np.float32(float(expect)), (H, entries)
        n += 1
    assert n == 3


def test_router_within_fp32_bound_of_fp64():
    cfg = S.WORKLOADS["decode-b1"]
    seed = S.workload_seed("decode-b1")
    wr = S.router_weights(seed, 0, cfg)[:32]
    x = S.tokens(seed, cfg, 2)
    lg = O.router_logits(x, wr)
    xf = S.bf16_bits_to_f32(x).astype(np.float64)
    wf = S.bf16_bits_to_f32(wr).astype(np.float64)
    ref = xf @ wf.T
    bound = (cfg["H"] // 32 + 5) * 2.0 ** -24 * (np.abs(xf) @ np.abs(wf).T)
    assert np.all(np.abs(lg - ref) <= bound)


# ----------------------------------------------------------------- top-k
def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(7)
    for trial in range(200):
        E = int(rng.integers(2, 40))
        k = int(rng.integers(1, E + 1))
        l = rng.integers(-3, 4, E).astype(np.float32)       # many ties
        if trial % 3 == 0:
            l = rng.standard_normal(E).astype(np.float32)
        idx, p = O.topk(l, k)
        order = np.lexsort((np.arange(E), -l.astype(np.float64)))
        np.testing.assert_array_equal(idx, order[:k])
        sm = scipy.special.softmax(l.astype(np.float64))
        np.testing.assert_allclose(p, sm[order[:k]], rtol=1e-14)


def test_topk_nan_ranks_last_and_signed_zero_ties():
    l = np.array([np.nan, 0.0, -0.0, -1.0], dtype=np.float32)
    idx, _ = O.topk(l, 4)
    assert list(idx) == [1, 2, 3, 0]


# ----------------------------------------------------------------- block mat-vec
def _dense(m: O.Matrix, e: int, codes: np.ndarray) -> np.ndarray:
    """Dequantized matrix from the generator's codes (not the oracle's unpack)."""
    sv = O.scale_values(m.fmt, m.scales[e]).reshape(m.rows, m.cols // 32)
    return np.repeat(sv, 32, axis=1) * m.cb[e].astype(np.float64)[codes]


@pytest.mark.parametrize("name", ["gate", "down", "sgate"])
def test_matvec_equals_dense_brute_force(name):
    cfg = dict(S.WORKLOADS["decode-b1"])
    cfg.update(H=256, I=128)
    seed = 11
    m = W.matrix(seed, 0, cfg, name, [3] if name != "sgate" else [0])
    e = 3 if name != "sgate" else 0
    codes = S.expert_codes(seed, 0, name, e, cfg)
    rng = np.random.default_rng(8)
    v = rng.standard_normal(m.cols).astype(np.float32)
    q, d = O.q8(v)
    out, Sp = O.matvec(m, e, q, d, partials=True)
    xdeq = q.astype(np.float64) * np.repeat(O.f16_array_to_f64(d), 32)
    ref = _dense(m, e, codes) @ xdeq
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-15)
    ci = m.cb[e].astype(np.int64)[codes].reshape(m.rows, -1, 32)
    Sref = (ci * q.astype(np.int64).reshape(1, -1, 32)).sum(-1)
    np.testing.assert_array_equal(Sp, Sref)


# ----------------------------------------------------------------- FFN
def _brute_ffn(cfg, seed, L, x, idx_p):
    """The whole FFN from dense dequantized matrices (numpy), with the pinned
    quantizer, rotation and router as building blocks."""
    H, I, k = cfg["H"], cfg["I"], cfg["k"]
    xf = S.bf16_bits_to_f32(x)
    if L.signs_x is not None:
        xf = O.h32_f32(xf, L.signs_x)
    xq, xd = O.q8(xf)
    xdeq = xq.astype(np.float64) * np.repeat(O.f16_array_to_f64(xd), 32)
    idx, p = idx_p
    experts = [("gate", "up", "down", e, p_) for e, p_ in zip(idx, p)]
    if cfg["shared_fmt"]:
        experts.append(("sgate", "sup", "sdown", 0, 1.0))
    y = np.zeros(H)
    hqs = []
    for gn, un, dn, e, w in experts:
        mats = [L.shared[i] if gn == "sgate" else (L.gate, L.up, L.down)[i] for i in range(3)]
        Wg = _dense(mats[0], e, S.expert_codes(seed, 0, gn, e, cfg))
        Wu = _dense(mats[1], e, S.expert_codes(seed, 0, un, e, cfg))
        Wd = _dense(mats[2], e, S.expert_codes(seed, 0, dn, e, cfg))
        g = Wg @ xdeq
        u = Wu @ xdeq
        h = (g * u / (1.0 + np.exp(-g))).astype(np.float32)
        if L.signs_h is not None:
            h = O.h32_f32(h, L.signs_h)
        hq, hd = O.q8(h)
        hqs.append(hq)
        hdeq = hq.astype(np.float64) * np.repeat(O.f16_array_to_f64(hd), 32)
        y += w * (Wd @ hdeq)
    return y, np.stack(hqs)


@pytest.mark.parametrize("variant", ["tiny", "tiny-shared", "tiny-h32", "tiny-p24"])
def test_ffn_decode_equals_brute_force(variant):
    cfg = dict(S.WORKLOADS["tiny-decode"])
    if variant == "tiny-shared":
        cfg.update(shared_fmt=4, k=3)
    if variant == "tiny-p24":  # down projections in the Packed24 layout
        cfg.update(fmt_down=24)
    if variant == "tiny-h32":
        cfg.update(h32=True, fmt_gu=4, fmt_down=4)
    seed = 21
    x = S.tokens(seed, cfg, 3)
    for t in range(3):
        L = W.layer(seed, 0, cfg, range(cfg["E"]))
        y, tr = O.ffn_decode(L, x[t], trace=True)
        lg = O.router_logits(x[t], L.router)[0]
        idx_p = O.topk(lg, cfg["k"])
        np.testing.assert_array_equal(tr["idx"], idx_p[0])
        ref, hq_ref = _brute_ffn(cfg, seed, L, x[t], idx_p)
        if np.array_equal(tr["hq"][:hq_ref.shape[0]], hq_ref):
            np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-14 * np.abs(ref).max())
        else:  # an fp32 rounding of h landed on the other side of a step: rare
            assert np.abs(tr["hq"][:hq_ref.shape[0]].astype(int) - hq_ref).max() <= 1


def test_expert_relabelling_invariance():
    cfg = S.WORKLOADS["tiny-decode"]
    seed = 22
    L = W.layer(seed, 0, cfg, range(cfg["E"]))
    x = S.tokens(seed, cfg, 2)
    perm = np.random.default_rng(9).permutation(cfg["E"])   # new id of old expert e: perm[e]
    L2 = W.layer(seed, 0, cfg, range(cfg["E"]))
    L2.router = L.router[np.argsort(perm)]
    for mname in ("gate", "up", "down"):
        m, m2 = getattr(L, mname), getattr(L2, mname)
        for field in ("codes", "scales", "cb"):
            setattr(m2, field, {int(perm[e]): v for e, v in getattr(m, field).items()})
    for t in range(2):
        y1, t1 = O.ffn_decode(L, x[t], trace=True)
        y2, t2 = O.ffn_decode(L2, x[t], trace=True)
        np.testing.assert_array_equal(perm[t1["idx"]], t2["idx"])
        np.testing.assert_array_equal(y1, y2)


def test_teacher_forcing_replaces_quantized_h():
    cfg = S.WORKLOADS["tiny-decode"]
    seed = 23
    L = W.layer(seed, 0, cfg, range(cfg["E"]))
    x = S.tokens(seed, cfg, 1)[0]
    y, tr = O.ffn_decode(L, x, trace=True)
    y2 = O.ffn_decode(L, x, force_hq=tr["hq"], force_hd=tr["hd"])
    np.testing.assert_array_equal(y, y2)
    hq = tr["hq"].copy()
    hq[0, 0] = hq[0, 0] + (1 if hq[0, 0] < 127 else -1)
    y3 = O.ffn_decode(L, x, force_hq=hq, force_hd=tr["hd"])
    assert not np.array_equal(y, y3)


def test_prefill_and_q4_are_per_token_decode():
    cfg = dict(S.WORKLOADS["tiny-decode"])
    cfg.update(dense=True, shared_fmt=4)
    seed = 24
    L = W.layer(seed, 0, cfg, range(cfg["E"]))
    x = S.tokens(seed, cfg, 4)
    yp = O.ffn_prefill(L, x)
    dense = W.dense(seed, 0, cfg)
    y4, yd = O.ffn_verify_q4(L, dense, x)
    for t in range(4):
        yt = O.ffn_decode(L, x[t])
        np.testing.assert_array_equal(yp[t], yt)
        np.testing.assert_array_equal(y4[t], yt)
        xq, xd = O.q8(S.bf16_bits_to_f32(x[t]))
        xdeq = xq.astype(np.float64) * np.repeat(O.f16_array_to_f64(xd), 32)
        Wd = _dense(dense, 0, S.expert_codes(seed, 0, "dense", 0, cfg))
        np.testing.assert_allclose(yd[t], Wd @ xdeq, rtol=1e-11, atol=1e-15)


# ----------------------------------------------------------------- RMSNorm
def test_rmsnorm_order_golden():
    n = 0
    for H, entries, expect in _golden_lines("rmsnorm_order.txt"):
        r = np.zeros(int(H), np.float32)
        for ent in entries.split():
            k, v = ent.split(":")
            r[int(k)] = np.float32(float(v))
        a = O.rmsnorm_bf16(r)
        for ent in expect.split():
            k, hx = ent.split(":")
            assert int(a[int(k)]) == int(hx, 16), (k, hex(int(a[int(k)])), hx)
        n += 1
    assert n == 1


def test_rmsnorm_bf16():
    a = O.rmsnorm_bf16(np.ones(4096, np.float32))
    assert np.all(a == 0x3F80)                      # 1 / sqrt(1 + 1e-6) rounds to bf16 1.0
    rng = np.random.default_rng(10)
    for scale in (1e-3, 1.0, 300.0):
        r = (rng.standard_normal(4096) * scale).astype(np.float32)
        a = S.bf16_bits_to_f32(O.rmsnorm_bf16(r)).astype(np.float64)
        r64 = r.astype(np.float64)
        ref = r64 / np.sqrt(np.mean(r64 ** 2) + 1e-6)
        ulp = 2.0 ** (np.floor(np.log2(np.abs(ref) + 1e-300)) - 7)
        assert np.all(np.abs(a - ref) <= ulp * 0.5001 + 1e-5 * np.abs(ref))


# ----------------------------------------------------------------- codebook quantizer
def _recoverable(fmt, rows=64, cols=256, seed=3):
    """Weights built from a known sorted codebook, codes and block scales, with
    one entry of magnitude 127 in every block (so that max|w| = 127 d)."""
    rng = np.random.default_rng(seed)
    K = 1 << fmt
    inner = np.sort(rng.choice(np.arange(-120, 121), K - 2, replace=False))
    cb = np.concatenate([[-127], inner, [127]]).astype(np.int8)
    codes = rng.integers(0, K, size=(rows, cols)).astype(np.uint8)
    codes[:, ::32] = np.where(rng.random((rows, cols // 32)) < 0.5, 0, K - 1)
    if fmt == 4:
        e = rng.integers(-20, -5, size=(rows, cols // 32))
        d = np.ldexp(1.0, e).astype(np.float32)
        sc = (e + 127).astype(np.uint8)
    else:
        d = np.float16(rng.uniform(1e-4, 1e-2, size=(rows, cols // 32))).astype(np.float32)
        sc = d.astype(np.float16).view(np.uint16)
    w = cb.astype(np.float32)[codes] * np.repeat(d, 32, axis=1)
    return w, cb, codes, sc


@pytest.mark.parametrize("fmt", [2, 3, 4])
def test_quantizer_recovers_a_known_codebook(fmt):
    w, cb, codes, sc = _recoverable(fmt)
    c2, s2, cb2 = O.quantize_expert(fmt, w)
    np.testing.assert_array_equal(cb2, cb)
    np.testing.assert_array_equal(s2, sc)
    np.testing.assert_array_equal(c2, codes)


@pytest.mark.parametrize("fmt", [2, 3, 4])
def test_quantizer_scales_codes_against_numpy(fmt):
    rng = np.random.default_rng(20 + fmt)
    w = (rng.standard_normal((48, 512)) * 0.02).astype(np.float32)
    w[3, 32:64] = 0.0  # an all-zero block
    codes, sc, cb = O.quantize_expert(fmt, w)
    m = np.abs(w).reshape(48, 16, 32).max(axis=2)
    if fmt == 4:
        e = sc.astype(np.int64) - 127
        d = np.ldexp(1.0, e)
        pos = m > 0
        assert np.all(127.0 * d >= m)                                  # |v| <= 127
        assert np.all((127.0 * d / 2 < m)[pos & (e > -127)])           # smallest such power
        assert np.all(e[~pos] == -127)
    else:
        ref = (m.astype(np.float32) / np.float32(127.0)).astype(np.float16)   # numpy RNE
        np.testing.assert_array_equal(sc, ref.view(np.uint16))
        d = ref.astype(np.float64)
    # codebook: 2^fmt sorted int8 entries
    assert cb.size == 1 << fmt and np.all(np.diff(cb.astype(int)) >= 0)
    # every code is the nearest entry to v = w / d in fp32, ties to the lower index
    df = np.repeat(d.astype(np.float32), 32, axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        v = np.where(df == 0, np.float32(0), w / df).astype(np.float32)
    dist = np.abs(v[..., None] - cb.astype(np.float32)[None, None, :])
    np.testing.assert_array_equal(codes, np.argmin(dist, axis=2))


def test_quantizer_lloyd_steps_golden():
    """A block whose codebook moves under the Lloyd steps, each step derived by
    hand (tests/golden/quantizer_lloyd.txt): pins the mid-quantile start, the
    nearest-entry cells with ties to the lower entry, and the half-up mean."""
    vals = {}
    for line in open(os.path.join(GOLDEN, "quantizer_lloyd.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split(":", 1)
            vals[k] = v.split()
    w = np.array([float(t) for t in vals["w"]], np.float32)[None, :]
    codes, sc, cb = O.quantize_expert(2, w)
    assert sc.ravel().tolist() == [int(vals["scale"][0], 16)]
    assert cb.astype(int).tolist() == [int(t) for t in vals["codebook"]]
    assert codes.ravel().tolist() == [int(t) for t in vals["codes"]]


def test_quantizer_ties_go_to_the_lower_entry():
    # codebook {-127, -1, 1, 127}; zeros sit exactly between -1 and 1
    fmt, rows, cols = 2, 8, 256
    K = 4
    cb = np.array([-127, -1, 1, 127], np.int8)
    rng = np.random.default_rng(5)
    codes = rng.integers(0, K, size=(rows, cols)).astype(np.uint8)
    codes[:, ::32] = 3
    d = np.float32(2.0 ** -10)
    w = cb.astype(np.float32)[codes] * d
    zero = rng.random((rows, cols)) < 0.01
    zero[:, ::32] = False
    w[zero] = 0.0
    c2, _, cb2 = O.quantize_expert(fmt, w)
    np.testing.assert_array_equal(cb2, cb)
    assert np.all(c2[zero] == 1)          # |0 - (-1)| == |0 - 1|: the lower index
    np.testing.assert_array_equal(c2[~zero], codes[~zero])
