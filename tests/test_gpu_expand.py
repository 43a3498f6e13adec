"""GPU parity of the expand-then-multiply ablation: moe_expand_bf16 against the
oracle's unpacked codes, codebooks and block scales (bf16 of the exact fp32
product, bit for bit), and moe_ffn_decode_expanded against a plain fp64
evaluation of the same definition (bf16 weights, unquantized x, h = silu(g) u,
the oracle's routing)."""
import numpy as np
import pytest
import torch

import oracle as O
import bit_codebook_quantized_dequant_gb300 as M
from bit_codebook_quantized_dequant_gb300 import synth as S
from bit_codebook_quantized_dequant_gb300.workload import (build_layer, expand_layer, to_dev_u16)
from _parity import host_layer_for

pytestmark = pytest.mark.gpu


def _dense_bf16(m: O.Matrix, e: int) -> np.ndarray:
    """bf16 expansion from the oracle's pieces, as float64 (torch's RNE)."""
    codes = O.unpack(m.fmt, m.rows, m.cols, m.codes[e])
    sv = O.scale_values(m.fmt, m.scales[e]).reshape(m.rows, m.cols // 32).astype(np.float32)
    w32 = m.cb[e].astype(np.float32)[codes] * np.repeat(sv, 32, axis=1)
    return torch.from_numpy(w32).to(torch.bfloat16).to(torch.float64).numpy()


def _reference(L: O.Layer, x_bf16):
    x = (x_bf16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    lg = O.router_logits(x_bf16[None, :], L.router)[0]
    idx, p = O.topk(lg, L.k)
    slots = [(L.gate, L.up, L.down, int(e), float(pp)) for e, pp in zip(idx, p)]
    if L.shared is not None:
        slots.append((L.shared[0], L.shared[1], L.shared[2], 0, 1.0))
    y = np.zeros(L.H)
    B = np.zeros(L.H)
    for G, U, D, e, w in slots:
        g = _dense_bf16(G, e) @ x
        u = _dense_bf16(U, e) @ x
        h = g * u / (1.0 + np.exp(-g))
        Wd = _dense_bf16(D, e)
        y += w * (Wd @ h)
        B += w * (np.abs(Wd) @ np.abs(h))
    return y, B, idx


@pytest.mark.parametrize("name", ["tiny-decode", "decode-b1"])
def test_expanded_decode_against_fp64_definition(name):
    cfg = dict(S.WORKLOADS[name])
    if name == "tiny-decode":
        cfg.update(shared_fmt=4, k=3)
    seed = S.workload_seed(name) + 3
    dl = build_layer(seed, 0, cfg)
    Lx, keep = expand_layer(dl)
    H = cfg["H"]
    xs = S.tokens(seed, cfg, 3, start=77)
    L = host_layer_for(seed, 0, cfg, xs)
    # the expansion of every matrix of the experts these tokens use, bit for bit
    dev = {n: t for n, t in zip([n for n in ("gate", "up", "down", "sgate", "sup", "sdown") if n in dl.mats], keep)}
    host = {"gate": L.gate, "up": L.up, "down": L.down}
    if L.shared is not None:
        host.update(sgate=L.shared[0], sup=L.shared[1], sdown=L.shared[2])
    for n, m in host.items():
        for e in sorted(m.codes)[:3]:  # experts the oracle layer holds
            got = dev[n][e * m.rows * m.cols:(e + 1) * m.rows * m.cols].cpu().numpy().view(np.uint16)
            ref = torch.from_numpy(_dense_bf16(m, e).astype(np.float32)).to(torch.bfloat16)
            np.testing.assert_array_equal(got, ref.view(torch.int16).numpy().view(np.uint16).ravel(),
                                          err_msg=f"{n} expert {e}")
    ws_bytes = M.moe_ffn_expanded_workspace(H, cfg["I"], cfg["E"], cfg["k"], 1 if cfg["shared_fmt"] else 0)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for t in range(xs.shape[0]):
        y = torch.zeros(H, dtype=torch.float32, device="cuda")
        M.moe_ffn_decode_expanded(Lx, to_dev_u16(xs[t]), y, ws, ws_bytes, st)
        torch.cuda.synchronize()
        assert st.item() == 0
        yr, B, idx = _reference(L, xs[t])
        np.testing.assert_array_equal(ws[:4 * cfg["k"]].view(torch.int32).cpu().numpy(), idx)
        yg = y.cpu().numpy().astype(np.float64)
        err = np.abs(yg - yr)
        assert np.all(err <= 1e-4 * B + 1e-30), f"max err/B {np.max(err / B):.3g}"
        rel = np.linalg.norm(yg - yr) / np.linalg.norm(yr)
        assert rel <= 1e-5, f"relative L2 {rel:.3g}"
