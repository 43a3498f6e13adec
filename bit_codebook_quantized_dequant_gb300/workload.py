"""Synthetic layers on the device: seeded codes and scales from the library's
generator twin, packed with moe_pack_expert; codebooks, router weights, tokens
and H32 sign masks drawn on the host by ``synth`` and copied over. PyTorch
only allocates memory here."""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np
import torch

from . import (MoeqDebug, MoeqLayer, MoeqMatrix, moe_ffn_workspace, moe_ffn_workspace_init,
               moe_pack_expert, moeq_packed_bytes, moeq_synth_codes, moeq_synth_scales)
from . import synth as S


CB_STRIDE = 16  # bytes per codebook record (the library reads whole 16-byte records)


def _round(n: int, a: int = 256) -> int:
    return (n + a - 1) // a * a


def to_dev_u16(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).to(device)


def to_dev_u32(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint32).view(np.int32)).to(device)


@dataclass
class DeviceMatrix:
    fmt: int
    rows: int
    cols: int
    E: int
    codes: torch.Tensor
    scales: torch.Tensor
    codebooks: torch.Tensor
    stride_codes: int
    stride_scales: int

    def desc(self) -> MoeqMatrix:
        return MoeqMatrix(self.fmt, self.rows, self.cols, self.E, self.codes.data_ptr(),
                          self.stride_codes, self.scales.data_ptr(), self.stride_scales,
                          self.codebooks.data_ptr(), 1 << S.code_bits(self.fmt), CB_STRIDE)

    @property
    def nbytes(self) -> int:
        cb, sb = moeq_packed_bytes(self.fmt, self.rows, self.cols)
        return self.E * (cb + sb)


def build_matrix(seed: int, layer: int, cfg: dict, name: str, scratch: Optional[torch.Tensor] = None,
                 device="cuda") -> DeviceMatrix:
    fmt, rows, cols = S.matrix_shape(cfg, name)
    E = cfg["E"] if name in ("gate", "up", "down") else 1
    cb, sb = moeq_packed_bytes(fmt, rows, cols)
    scb, ssb = _round(cb), _round(sb)
    codes = torch.empty(E * scb, dtype=torch.uint8, device=device)
    scales = torch.empty(E * ssb, dtype=torch.uint8, device=device)
    if scratch is None or scratch.numel() < rows * cols:
        scratch = torch.empty(rows * cols, dtype=torch.uint8, device=device)
    role = S.MATRIX_ROLES[name]
    nb = cols // 32
    bits = S.code_bits(fmt)
    for e in range(E):
        moeq_synth_codes(seed, S.stream_id(layer, role, e, S.KIND_CODES), bits, rows * cols, scratch)
        sp = scales.data_ptr() + e * ssb
        moeq_synth_scales(seed, S.stream_id(layer, role, e, S.KIND_SCALES), bits, rows * nb, sp)
        moe_pack_expert(fmt, rows, cols, scratch, sp, codes.data_ptr() + e * scb, sp)
    books = np.zeros((E, CB_STRIDE), dtype=np.int8)  # records padded to 16 bytes
    for e in range(E):
        books[e, : 1 << bits] = S.codebook(seed, S.stream_id(layer, role, e, S.KIND_CODEBOOK), bits)
    codebooks = torch.from_numpy(books).to(device)
    return DeviceMatrix(fmt, rows, cols, E, codes, scales, codebooks, scb, ssb)


@dataclass
class DeviceLayer:
    cfg: dict
    seed: int
    layer: int
    router: torch.Tensor
    mats: Dict[str, DeviceMatrix]
    signs_x: Optional[torch.Tensor] = None
    signs_h: Optional[torch.Tensor] = None
    _desc: Optional[MoeqLayer] = field(default=None, repr=False)

    def desc(self) -> MoeqLayer:
        if self._desc is None:
            c = self.cfg
            L = MoeqLayer()
            L.H, L.I, L.E, L.k = c["H"], c["I"], c["E"], c["k"]
            L.router = self.router.data_ptr()
            L.gate = self.mats["gate"].desc()
            L.up = self.mats["up"].desc()
            L.down = self.mats["down"].desc()
            if "sgate" in self.mats:
                L.has_shared = 1
                L.sgate = self.mats["sgate"].desc()
                L.sup = self.mats["sup"].desc()
                L.sdown = self.mats["sdown"].desc()
            if self.signs_x is not None:
                L.h32_signs_x = self.signs_x.data_ptr()
                L.h32_signs_h = self.signs_h.data_ptr()
            self._desc = L
        return self._desc

    @property
    def dense(self) -> Optional[DeviceMatrix]:
        return self.mats.get("dense")

    def weight_bytes(self) -> int:
        return sum(m.nbytes for n, m in self.mats.items() if n != "dense") + self.router.numel() * 2


def build_layer(seed: int, layer: int, cfg: dict, device="cuda") -> DeviceLayer:
    H, I = cfg["H"], cfg["I"]
    scratch = torch.empty(max(H * I, H * H if cfg["dense"] else 0), dtype=torch.uint8, device=device)
    mats = {name: build_matrix(seed, layer, cfg, name, scratch, device) for name in S.layer_roles(cfg)}
    router = to_dev_u16(S.router_weights(seed, layer, cfg), device)
    dl = DeviceLayer(cfg, seed, layer, router, mats)
    if cfg["h32"]:
        dl.signs_x = to_dev_u32(S.h32_signs(seed, layer, cfg, "x"), device)
        dl.signs_h = to_dev_u32(S.h32_signs(seed, layer, cfg, "h"), device)
    del scratch
    return dl


def expand_layer(dl: DeviceLayer, device="cuda"):
    """The layer's packed matrices expanded to bf16 (moe_expand_bf16), as a
    layer descriptor of MOEQ_BF16 matrices for moe_ffn_decode_expanded; returns
    (descriptor, the tensors that hold the weights)."""
    from . import MOEQ_BF16, moe_expand_bf16
    keep = []
    L = MoeqLayer()
    src = dl.desc()
    L.H, L.I, L.E, L.k, L.has_shared = src.H, src.I, src.E, src.k, src.has_shared
    L.router = src.router
    for name in ("gate", "up", "down", "sgate", "sup", "sdown"):
        if name not in dl.mats:
            continue
        m = dl.mats[name]
        out = torch.empty(m.E * m.rows * m.cols, dtype=torch.int16, device=device)
        moe_expand_bf16(m.desc(), 0, m.E, out)
        keep.append(out)
        setattr(L, name, MoeqMatrix(MOEQ_BF16, m.rows, m.cols, m.E, out.data_ptr(), 2 * m.rows * m.cols,
                                    None, 0, None, 0, 0))
    return L, keep


class Workspace:
    """A zeroed workspace for one FFN entry point (mode 0 decode, 1 q4, 2 prefill)."""

    def __init__(self, layer: DeviceLayer, mode: int, T_max: int = 1, device="cuda"):
        self.nbytes = moe_ffn_workspace(layer.desc(), T_max, mode)
        if self.nbytes == 0:
            raise ValueError("invalid layer descriptor for the workspace")
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        moe_ffn_workspace_init(self.buf, self.nbytes)

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()


class Debug:
    """Device buffers for the intermediates of a decode (T = 1) or of a q=4
    verification (T = 4 columns); vectors are (column, slot) pairs."""

    def __init__(self, cfg: dict, T: int = 1, partials: bool = False, device="cuda"):
        H, I, E, k = cfg["H"], cfg["I"], cfg["E"], cfg["k"]
        ns = k + (1 if cfg["shared_fmt"] else 0)
        z = lambda n, dt: torch.zeros(n, dtype=dt, device=device)
        self.t = dict(xq=z(T * H, torch.int8), xd=z(T * H // 32, torch.int16),
                      logits=z(T * E, torch.float32), idx=z(T * k, torch.int32),
                      p=z(T * k, torch.float32), h=z(T * ns * I, torch.float32),
                      hq=z(T * ns * I, torch.int8), hd=z(T * ns * I // 32, torch.int16),
                      o=z(T * ns * H, torch.float32))
        if partials:
            self.t.update(S_gate=z(T * ns * I * H // 32, torch.int32),
                          S_up=z(T * ns * I * H // 32, torch.int32),
                          S_down=z(T * ns * H * I // 32, torch.int32))
        self.struct = MoeqDebug(**{n: v.data_ptr() for n, v in self.t.items()})

    def numpy(self) -> Dict[str, np.ndarray]:
        out = {}
        for n, v in self.t.items():
            a = v.cpu().numpy()
            if n in ("xd", "hd"):
                a = a.view(np.uint16)
            out[n] = a
        return out
