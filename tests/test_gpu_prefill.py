"""GPU parity of moe_ffn_prefill (expert-grouped, T tokens) against the oracle:
for sampled tokens the same stage-by-stage checks as the decode (bit-exact
xq/xd, logits and indices; h within fp32 tolerance; hq/hd equal to the
oracle's quantizer on the GPU's h; per-slot outputs and y teacher-forced
within the output tolerance), the residual form, and the edge cases (T = 0,
one token, a ragged last tile, a workspace too small)."""
import numpy as np
import pytest
import torch

import oracle as O
import bit_codebook_quantized_dequant_gb300 as M
from bit_codebook_quantized_dequant_gb300 import synth as S
from bit_codebook_quantized_dequant_gb300.workload import (Debug, Workspace, build_layer,
                                                           to_dev_u16)
from _parity import FLIPS_PREFILL, PREFILL, check_output, check_token, column_view, host_layer_for

pytestmark = pytest.mark.gpu


def _cfg(name, **over):
    c = dict(S.WORKLOADS[name])
    c.update(over)
    return c


def _prefill(dl, ws, X, residual=None, dbg=True):
    cfg = dl.cfg
    T, H = X.shape
    d = Debug(cfg, T) if dbg else None
    y = torch.zeros(T * H, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = torch.from_numpy(residual).cuda() if residual is not None else None
    M.moe_ffn_prefill(dl.desc(), to_dev_u16(X), T, r, y, ws.ptr, ws.nbytes, st,
                      d.struct if d is not None else None)
    torch.cuda.synchronize()
    assert st.item() == 0, M.STATUS.get(st.item())
    return y.cpu().numpy().reshape(T, H), (d.numpy() if d is not None else None)


def _check_tokens(dl, seed, cfg, X, sample):
    y, g = _prefill(dl, Workspace(dl, 2, X.shape[0]), X)
    L = host_layer_for(seed, 0, cfg, X[sample])
    for t in sample:
        check_token(L, cfg, X[t], y[t], column_view(g, cfg, t), False, **PREFILL)
    return y


@pytest.mark.parametrize("variant", ["cfg0", "cfg0-shared", "cfg0-h32-fp4"])
def test_prefill_tiny(variant):
    over = {}
    if variant == "cfg0-shared":
        over = dict(shared_fmt=4, k=3)
    elif variant == "cfg0-h32-fp4":
        over = dict(h32=True, fmt_gu=4, fmt_down=4)
    cfg = _cfg("tiny-decode", **over)
    seed = S.workload_seed("tiny-decode") + 31 * len(variant)
    dl = build_layer(seed, 0, cfg)
    T = 300  # several 64-row tiles per expert group and a ragged last one
    X = S.tokens(seed, cfg, T)
    sample = list(range(0, T, 23)) + [T - 1]
    _check_tokens(dl, seed, cfg, X, sample)


def test_prefill_config3_sampled_tokens():
    cfg = _cfg("prefill-h32-fp4")
    seed = S.workload_seed("prefill-h32-fp4")
    dl = build_layer(seed, 0, cfg)
    T = 256
    X = S.tokens(seed, cfg, T)
    _check_tokens(dl, seed, cfg, X, list(range(0, T, 16)) + [T - 1])  # 17 tokens


def test_prefill_matches_decode_and_residual():
    cfg = _cfg("decode-b1")
    seed = S.workload_seed("decode-b1")
    dl = build_layer(seed, 0, cfg)
    T = 70
    X = S.tokens(seed, cfg, T, start=500)
    ws = Workspace(dl, 2, T)
    y, g = _prefill(dl, ws, X)
    # decode of the same tokens: same routing, outputs equal up to fp32 summation order
    ws1 = Workspace(dl, 0)
    L = host_layer_for(seed, 0, cfg, X[[0, 69]])
    for t in (0, 69):
        yd = torch.zeros(cfg["H"], dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        dd = Debug(cfg, 1)
        M.moe_ffn_decode(dl.desc(), to_dev_u16(X[t]), yd, ws1.ptr, ws1.nbytes, st, dd.struct)
        torch.cuda.synchronize()
        gt = column_view(g, cfg, t)
        yo, B, _ = check_token(L, cfg, X[t], y[t], gt, False, **PREFILL)
        gd = dd.numpy()
        np.testing.assert_array_equal(gd["idx"], gt["idx"])
        flips = int((gd["hq"] != gt["hq"]).sum())
        assert flips <= FLIPS_PREFILL * gd["hq"].size  # see FLIPS_PREFILL
        if flips == 0 and np.array_equal(gd["hd"], gt["hd"]):
            check_output(yd.cpu().numpy(), y[t].astype(np.float64), B, "decode vs prefill")
    # residual form: y = residual + FFN(x), rounded once
    res = np.random.default_rng(5).standard_normal((T, cfg["H"])).astype(np.float32)
    y2, _ = _prefill(dl, ws, X, residual=res, dbg=False)
    np.testing.assert_array_equal(y2, (res + y).astype(np.float32))
    # repeated calls on one workspace give the same bits
    y3, _ = _prefill(dl, ws, X, dbg=False)
    np.testing.assert_array_equal(y3, y)


def test_prefill_edge_cases():
    cfg = _cfg("tiny-decode")
    seed = S.workload_seed("tiny-decode") + 3
    dl = build_layer(seed, 0, cfg)
    ws = Workspace(dl, 2, 8)
    y = torch.zeros(8 * cfg["H"], dtype=torch.float32, device="cuda")
    X = to_dev_u16(S.tokens(seed, cfg, 8))
    # T = 0 enqueues nothing
    M.moe_ffn_prefill(dl.desc(), X, 0, None, y, ws.ptr, ws.nbytes)
    # a workspace sized for 8 tokens is too small for 9
    with pytest.raises(M.MoeqError) as ex:
        M.moe_ffn_prefill(dl.desc(), X, 9, None, y, ws.ptr, ws.nbytes)
    assert ex.value.rc == M.CODE["MOEQ_ERR_WORKSPACE"]
    # one token
    Xh = S.tokens(seed, cfg, 1)
    y1, g = _prefill(dl, ws, Xh)
    L = host_layer_for(seed, 0, cfg, Xh)
    check_token(L, cfg, Xh[0], y1[0], column_view(g, cfg, 0), False, **PREFILL)
