"""GPU parity of one decode token through a stack of layers
(moe_ffn_stack_decode) on layers shaped like the 43-layer workload, on a few
layers and tokens:
  * the stack entry equals its composition (RMSNorm, decode, fp32 residual
    add) bit for bit;
  * per layer, teacher-forced from the GPU's own RMSNorm output a_l: a_l is the
    oracle's RMSNorm of the GPU's r_l bit for bit, and the layer's decode
    passes the stage-by-stage checks against the oracle;
  * end to end, the oracle's own chain agrees with r_L within the summed
    per-layer output bounds, for tokens whose routing is the same in both."""
import numpy as np
import pytest
import torch

import oracle as O
import bit_codebook_quantized_dequant_gb300 as M
from bit_codebook_quantized_dequant_gb300 import synth as S
from bit_codebook_quantized_dequant_gb300.workload import (Debug, Workspace, build_layer,
                                                           to_dev_u16)
from _parity import ELEM, check_token, host_layer_for

pytestmark = pytest.mark.gpu

NL, NTOK = 3, 4


def test_stack_decode_matches_composition_and_oracle():
    cfg = dict(S.WORKLOADS["prefill-43-layer-stack"])
    seed = S.workload_seed("prefill-43-layer-stack")
    layers = [build_layer(seed, l, cfg) for l in range(NL)]
    descs = [dl.desc() for dl in layers]
    H = cfg["H"]
    X = S.tokens(seed, cfg, NTOK, start=900)
    ws = Workspace(layers[0], 4)
    ws1 = Workspace(layers[0], 0)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    checked = 0
    for t in range(NTOK):
        x = to_dev_u16(X[t])
        r_stack = torch.zeros(H, dtype=torch.float32, device="cuda")
        M.moe_ffn_stack_decode(descs, x, r_stack, ws.ptr, ws.nbytes, st)
        torch.cuda.synchronize()
        assert st.item() == 0
        # the composition, layer by layer, with the intermediates
        r = torch.from_numpy((X[t].astype(np.uint32) << 16).view(np.float32).copy()).cuda()
        a = torch.zeros(H, dtype=torch.int16, device="cuda")
        bound = np.zeros(H)
        routes = []
        for l, dl in enumerate(layers):
            r_host = r.cpu().numpy()
            M.moe_rmsnorm_bf16(r, 1, H, a)
            d = Debug(cfg, 1)
            y = torch.zeros(H, dtype=torch.float32, device="cuda")
            M.moe_ffn_decode(dl.desc(), a, y, ws1.ptr, ws1.nbytes, st, d.struct)
            torch.cuda.synchronize()
            assert st.item() == 0
            a_host = a.cpu().numpy().view(np.uint16)
            np.testing.assert_array_equal(a_host, O.rmsnorm_bf16(r_host))
            L = host_layer_for(seed, l, cfg, a_host[None, :])
            g = d.numpy()
            _, B, _ = check_token(L, cfg, a_host, y.cpu().numpy(), g, False)
            bound += B
            routes.append(g["idx"].copy())
            r = r + y
        np.testing.assert_array_equal(r_stack.cpu().numpy(), r.cpu().numpy())
        # the oracle's own chain
        x0 = (X[t].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        ro = x0.copy()
        same = True
        for l in range(NL):
            ao = O.rmsnorm_bf16(ro.astype(np.float32))
            L = host_layer_for(seed, l, cfg, ao[None, :])
            yo, tr = O.ffn_decode(L, ao, trace=True)
            same &= np.array_equal(tr["idx"], routes[l])
            ro = ro + yo
        if not same:  # fp32 drift moved a routing decision near a tie
            continue
        err = np.abs(r.cpu().numpy().astype(np.float64) - ro)
        assert np.all(err <= ELEM * bound + 1e-6 * np.abs(ro)), \
            f"token {t}: max err/B {np.max(err / bound):.3g}"
        checked += 1
    assert checked >= 2


def test_stack_verify_q4_columns_equal_stack_decode():
    """Four columns through the stack with moe_ffn_stack_verify_q4 (each layer's
    weights read once per call for all columns) equal, column by column and bit
    for bit, moe_ffn_stack_decode of each column, which the test above pins to
    the oracle; columns 1 and 3 are equal, so some units serve two columns."""
    cfg = dict(S.WORKLOADS["prefill-43-layer-stack"])
    seed = S.workload_seed("prefill-43-layer-stack")
    layers = [build_layer(seed, l, cfg) for l in range(NL)]
    descs = [dl.desc() for dl in layers]
    H = cfg["H"]
    X = S.tokens(seed, cfg, 3, start=950)
    X4 = np.stack([X[0], X[1], X[2], X[1]])
    ws4 = Workspace(layers[0], 5)
    ws1 = Workspace(layers[0], 4)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    x4 = to_dev_u16(X4)
    r4 = torch.zeros(4, H, dtype=torch.float32, device="cuda")
    for _ in range(2):  # the second call on the same workspace must repeat the first
        M.moe_ffn_stack_verify_q4(descs, x4, r4, ws4.ptr, ws4.nbytes, st)
        torch.cuda.synchronize()
        assert st.item() == 0
        for c in range(4):
            r1 = torch.zeros(H, dtype=torch.float32, device="cuda")
            M.moe_ffn_stack_decode(descs, to_dev_u16(X4[c]), r1, ws1.ptr, ws1.nbytes, st)
            torch.cuda.synchronize()
            assert st.item() == 0
            np.testing.assert_array_equal(r4[c].cpu().numpy(), r1.cpu().numpy())
