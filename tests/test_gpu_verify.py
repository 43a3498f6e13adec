"""GPU parity of moe_ffn_verify_q4 (four columns, each routed independently,
every expert's weights read once for all the columns that select it) against
the oracle: per column the same stage-by-stage checks as the decode, the dense
projection within the output tolerance, and bitwise agreement with four
separate decodes (the kernel takes the same fp32 operations in the same order
for a column whatever other columns share its experts)."""
import numpy as np
import pytest
import torch

import oracle as O
import bit_codebook_quantized_dequant_gb300 as M
from bit_codebook_quantized_dequant_gb300 import synth as S
from bit_codebook_quantized_dequant_gb300.workload import (Debug, Workspace, build_layer,
                                                           to_dev_u16)
from oracle import workload as W
from _parity import check_output, check_token, column_view, host_layer_for

pytestmark = pytest.mark.gpu


def _cfg(name, **over):
    c = dict(S.WORKLOADS[name])
    c.update(over)
    return c


def _verify(dl, ws, X, partials=False, with_dense=True, dbg=True):
    cfg = dl.cfg
    H = cfg["H"]
    d = Debug(cfg, 4, partials) if dbg else None
    y = torch.zeros(4 * H, dtype=torch.float32, device="cuda")
    dm = dl.dense if with_dense else None
    yd = torch.full((4 * dm.rows,) if dm is not None else (16,), 7.0, dtype=torch.float32,
                    device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_ffn_verify_q4(dl.desc(), dm.desc() if dm is not None else None, to_dev_u16(X), y,
                        yd if dm is not None else None, ws.ptr, ws.nbytes, st,
                        d.struct if d is not None else None)
    torch.cuda.synchronize()
    assert st.item() == 0, M.STATUS.get(st.item())
    return (y.cpu().numpy().reshape(4, H), yd.cpu().numpy(),
            d.numpy() if d is not None else None)


def _decode(dl, ws1, x_row):
    y = torch.zeros(dl.cfg["H"], dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_ffn_decode(dl.desc(), to_dev_u16(x_row), y, ws1.ptr, ws1.nbytes, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return y.cpu().numpy()


def _abs_weights(Dm: O.Matrix):
    codes = O.unpack(Dm.fmt, Dm.rows, Dm.cols, Dm.codes[0])
    sv = O.scale_values(Dm.fmt, Dm.scales[0]).reshape(Dm.rows, Dm.cols // 32)
    return np.abs(np.repeat(sv, 32, axis=1) * Dm.cb[0].astype(np.float64)[codes])


def _dense_bound(Wabs, xq, xd):
    xt = np.abs(xq.astype(np.float64) * np.repeat(O.f16_array_to_f64(xd), 32))
    return Wabs @ xt


def _check_batch(dl, seed, cfg, X, partials, ws, ws1, L=None, dense=None):
    """One q=4 call on the 4 columns of X, checked column by column (L: an
    oracle layer holding the columns' experts; dense: (matrix, |W|) of the
    dense projection, built when not given)."""
    y, yd, g = _verify(dl, ws, X, partials)
    if L is None:
        L = host_layer_for(seed, 0, cfg, X)
    for c in range(4):
        check_token(L, cfg, X[c], y[c], column_view(g, cfg, c), partials)
        np.testing.assert_array_equal(y[c], _decode(dl, ws1, X[c]), err_msg=f"column {c}")
    if cfg["dense"]:
        if dense is None:
            Dm = W.dense(seed, 0, cfg)
            dense = (Dm, _abs_weights(Dm))
        Dm, Wabs = dense
        _, yd_ref = O.ffn_verify_q4(L, Dm, X)
        H = cfg["H"]
        for c in range(4):
            B = _dense_bound(Wabs, g["xq"][c * H:(c + 1) * H], g["xd"][c * (H // 32):(c + 1) * (H // 32)])
            check_output(yd[c * Dm.rows:(c + 1) * Dm.rows], yd_ref[c], B, f"y_dense[{c}]")
    return y


@pytest.mark.parametrize("pattern", ["distinct", "all-equal", "pairs"])
@pytest.mark.parametrize("variant", ["cfg0-shared", "cfg0-h32-fp4"])
def test_verify_tiny(variant, pattern):
    over = dict(dense=True)
    if variant == "cfg0-shared":
        over.update(shared_fmt=4, k=3)
    else:
        over.update(h32=True, fmt_gu=4, fmt_down=4)
    cfg = _cfg("tiny-decode", **over)
    seed = S.workload_seed("tiny-decode") + 101 * len(variant)
    dl = build_layer(seed, 0, cfg)
    ws, ws1 = Workspace(dl, 1), Workspace(dl, 0)
    xs = S.tokens(seed, cfg, 12)
    batches = [xs[4 * i:4 * i + 4] for i in range(3)]
    if pattern == "all-equal":
        batches = [np.repeat(b[:1], 4, axis=0) for b in batches[:2]]
    elif pattern == "pairs":
        batches = [b[[0, 1, 0, 2]] for b in batches[:2]]
    for i, X in enumerate(batches):
        _check_batch(dl, seed, cfg, np.ascontiguousarray(X), i == 0, ws, ws1)


def test_verify_config2_sampled_batches():
    cfg = _cfg("verify-q4")
    seed = S.workload_seed("verify-q4")
    dl = build_layer(seed, 0, cfg)
    ws, ws1 = Workspace(dl, 1), Workspace(dl, 0)
    nb = 16  # batches of 4 independently routed columns
    xs = S.tokens(seed, cfg, 4 * nb)
    L = host_layer_for(seed, 0, cfg, xs)
    Dm = W.dense(seed, 0, cfg)
    dense = (Dm, _abs_weights(Dm))
    for b in range(nb):
        _check_batch(dl, seed, cfg, xs[4 * b:4 * b + 4], b == 0, ws, ws1, L, dense)
    # two columns equal: their experts are read once for both
    _check_batch(dl, seed, cfg, np.ascontiguousarray(xs[[4, 5, 4, 6]]), False, ws, ws1, L, dense)


def test_verify_without_dense_and_repeatable():
    cfg = _cfg("verify-q4")
    seed = S.workload_seed("verify-q4")
    dl = build_layer(seed, 0, cfg)
    ws = Workspace(dl, 1)
    X = S.tokens(seed, cfg, 4, start=40)
    ys = []
    for rep in range(3):
        y, yd, _ = _verify(dl, ws, X, with_dense=False, dbg=False)
        assert np.all(yd == 7.0)  # y_dense untouched without a dense matrix
        ys.append(y)
    for rep in range(1, 3):
        np.testing.assert_array_equal(ys[rep], ys[0])
    y, _, _ = _verify(dl, ws, X, with_dense=True, dbg=False)
    np.testing.assert_array_equal(y, ys[0])
    # counters (and routing record copies) are back to zero after every call
    units = 4 * cfg["k"] + 1
    n_ctr = 32 * (4 + units) + 32 * 16 * 4
    ctr = ws.buf[: 4 * n_ctr].view(torch.int32).cpu().numpy()
    assert not ctr.any()
