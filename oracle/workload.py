"""Host-side layers for the oracle, drawn from the seeded generators -- TEST
INFRASTRUCTURE ONLY. Packs with the oracle's own packer; only the experts asked
for are materialized (a full decode layer is 2.3 GB packed)."""
from __future__ import annotations

from typing import Iterable, Optional

import numpy as np

import oracle as O
from bit_codebook_quantized_dequant_gb300 import synth as S


def matrix(seed: int, layer: int, cfg: dict, name: str, experts: Iterable[int],
           E: Optional[int] = None) -> O.Matrix:
    fmt, rows, cols = S.matrix_shape(cfg, name)
    if E is None:
        E = cfg["E"] if name in ("gate", "up", "down") else 1
    m = O.Matrix(fmt=fmt, rows=rows, cols=cols, E=E)
    for e in experts:
        c = S.expert_codes(seed, layer, name, e, cfg)
        m.codes[e] = O.pack(fmt, c)
        m.scales[e] = S.expert_scales(seed, layer, name, e, cfg)
        m.cb[e] = S.expert_codebook(seed, layer, name, e, cfg)
    return m


def layer(seed: int, layer_idx: int, cfg: dict, experts: Iterable[int]) -> O.Layer:
    experts = sorted(set(int(e) for e in experts))
    L = O.Layer(H=cfg["H"], I=cfg["I"], E=cfg["E"], k=cfg["k"],
                router=S.router_weights(seed, layer_idx, cfg),
                gate=matrix(seed, layer_idx, cfg, "gate", experts),
                up=matrix(seed, layer_idx, cfg, "up", experts),
                down=matrix(seed, layer_idx, cfg, "down", experts))
    if cfg["shared_fmt"]:
        L.shared = tuple(matrix(seed, layer_idx, cfg, n, [0]) for n in ("sgate", "sup", "sdown"))
    if cfg["h32"]:
        L.signs_x = S.h32_signs(seed, layer_idx, cfg, "x")
        L.signs_h = S.h32_signs(seed, layer_idx, cfg, "h")
    return L


def dense(seed: int, layer_idx: int, cfg: dict) -> O.Matrix:
    return matrix(seed, layer_idx, cfg, "dense", [0])


def route(seed: int, layer_idx: int, cfg: dict, x_bf16: np.ndarray):
    """Oracle top-k of each row of x (to know which experts to materialize)."""
    wr = S.router_weights(seed, layer_idx, cfg)
    lg = O.router_logits(x_bf16, wr)
    return [O.topk(l, cfg["k"])[0] for l in lg], lg
