"""GPU parity of moe_ffn_prefill at the workloads' full token counts, in the
launch configuration bench.py times (one call of T tokens on the current
stream): T = 2048 with FP4 experts and H32 on x and h, and T = 32512 on a
layer of the 43-layer stack (FP2/FP3 routed experts, FP4 shared expert). On
sampled tokens (first, second, last and 13 spread over the rest) the same stage-by-stage checks
as the smaller prefill tests: bit-exact xq/xd, logits and indices; h, hq/hd,
the per-slot outputs and y against the oracle."""
import numpy as np
import pytest
import torch

import bit_codebook_quantized_dequant_gb300 as M
from bit_codebook_quantized_dequant_gb300 import synth as S
from bit_codebook_quantized_dequant_gb300.workload import Debug, Workspace, build_layer, to_dev_u16
from _parity import PREFILL, check_token, column_view, host_layer_for


def token_rows(dbg: Debug, T: int, sample) -> dict:
    """The sampled tokens' rows of the debug buffers (all token-major),
    gathered on the device and copied to the host; row i of each field is
    token sample[i], shaped like column_view's per-token slices."""
    dev = next(iter(dbg.t.values())).device
    idx = torch.as_tensor(list(sample), dtype=torch.long, device=dev)
    out = {}
    for n, v in dbg.t.items():
        a = v.view(T, -1).index_select(0, idx).cpu().numpy()
        if n in ("xd", "hd"):
            a = a.view(np.uint16)
        out[n] = a
    return out


def test_token_rows_matches_column_view():
    # host-side check of the gathering (CPU tensors with distinct values)
    cfg = dict(S.WORKLOADS["tiny-decode"], shared_fmt=4)
    T = 5
    d = Debug(cfg, T, device="cpu")
    for i, v in enumerate(d.t.values()):
        v.copy_(torch.arange(v.numel(), dtype=torch.float64).remainder(97 + i).to(v.dtype))
    full = d.numpy()
    rows = token_rows(d, T, [4, 0, 2])
    for i, t in enumerate([4, 0, 2]):
        ref = column_view(full, cfg, t)
        for n in full:
            np.testing.assert_array_equal(rows[n][i], ref[n], err_msg=n)


@pytest.mark.gpu
@pytest.mark.parametrize("name,T", [("prefill-h32-fp4", 2048), ("prefill-43-layer-stack", 32512)])
def test_prefill_full_size_sampled_tokens(name, T):
    cfg = dict(S.WORKLOADS[name])
    seed = S.workload_seed(name)
    H = cfg["H"]
    dl = build_layer(seed, 0, cfg)
    X = S.tokens(seed, cfg, T)
    # first, second, last and 13 tokens spread over the rest (16 in all)
    sample = sorted({0, 1, T - 1} | {(T * j) // 14 + 3 for j in range(1, 14)})
    ws = Workspace(dl, 2, T)
    d = Debug(cfg, T)
    y = torch.zeros(T * H, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_ffn_prefill(dl.desc(), to_dev_u16(X), T, None, y, ws.ptr, ws.nbytes, st, d.struct,
                      torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert st.item() == 0, M.STATUS.get(st.item())
    g = token_rows(d, T, sample)
    ys = y.view(T, H).index_select(0, torch.as_tensor(sample, device="cuda")).cpu().numpy()
    L = host_layer_for(seed, 0, cfg, X[sample])
    for i, t in enumerate(sample):
        check_token(L, cfg, X[t], ys[i], {n: v[i] for n, v in g.items()}, False, **PREFILL)
