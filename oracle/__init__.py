"""ctypes wrapper of the CPU oracle (oracle.c) -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never calls it.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from dataclasses import dataclass, field
from typing import Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-fPIC", "-shared", "-Wall"]

_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so next to the source with gcc (no CUDA involved)."""
    stale = (not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(os.path.getmtime(_SRC),
                                                                       os.path.getmtime(_HDR)))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = C.CDLL(_LIB)
        _declare(_lib)
    return _lib


P = C.c_void_p


class OrcMatrix(C.Structure):
    _fields_ = [("fmt", C.c_int), ("rows", C.c_int), ("cols", C.c_int),
                ("codes", P), ("scales", P), ("cb", P)]


class OrcLayer(C.Structure):
    _fields_ = [("H", C.c_int), ("I", C.c_int), ("E", C.c_int), ("k", C.c_int),
                ("router", P), ("gate", OrcMatrix), ("up", OrcMatrix), ("down", OrcMatrix),
                ("has_shared", C.c_int), ("sgate", OrcMatrix), ("sup", OrcMatrix),
                ("sdown", OrcMatrix), ("signs_x", P), ("signs_h", P)]


class OrcTrace(C.Structure):
    _fields_ = [(n, P) for n in ("xq", "xd", "logits", "idx", "p", "S_gate", "S_up", "g", "u",
                                 "h", "hq", "hd", "S_down", "o", "force_hq", "force_hd",
                                 "force_idx")]


def _declare(L):
    L.orc_f32_to_f16.restype = C.c_uint16
    L.orc_f32_to_f16.argtypes = [C.c_float]
    L.orc_f16_to_f64.restype = C.c_double
    L.orc_f16_to_f64.argtypes = [C.c_uint16]
    L.orc_f32_to_bf16.restype = C.c_uint16
    L.orc_f32_to_bf16.argtypes = [C.c_float]
    L.orc_bf16_to_f32.restype = C.c_float
    L.orc_bf16_to_f32.argtypes = [C.c_uint16]
    L.orc_packed_bytes.argtypes = [C.c_int, C.c_int, C.c_int, C.POINTER(C.c_size_t),
                                   C.POINTER(C.c_size_t)]
    L.orc_pack.argtypes = [C.c_int, C.c_int, C.c_int, P, P]
    L.orc_unpack.argtypes = [C.c_int, C.c_int, C.c_int, P, P]
    L.orc_scale_value.restype = C.c_double
    L.orc_scale_value.argtypes = [C.c_int, P, C.c_size_t]
    L.orc_q8.argtypes = [P, C.c_int, P, P]
    L.orc_q8.restype = None
    L.orc_h32_f32.argtypes = [P, P, C.c_int, P]
    L.orc_h32_f32.restype = None
    L.orc_h32_f64.argtypes = [P, P, C.c_int, P]
    L.orc_h32_f64.restype = None
    L.orc_router_logit.restype = C.c_float
    L.orc_router_logit.argtypes = [P, P, C.c_int]
    L.orc_router.argtypes = [P, C.c_int, P, C.c_int, C.c_int, P]
    L.orc_router.restype = None
    L.orc_topk.argtypes = [P, C.c_int, C.c_int, P, P]
    L.orc_topk.restype = None
    L.orc_block_partials.argtypes = [C.POINTER(OrcMatrix), C.c_int, C.c_int, P, P]
    L.orc_matvec.argtypes = [C.POINTER(OrcMatrix), C.c_int, P, P, P, P]
    L.orc_ffn_decode.argtypes = [C.POINTER(OrcLayer), P, P, C.POINTER(OrcTrace)]
    L.orc_ffn_verify_q4.argtypes = [C.POINTER(OrcLayer), C.POINTER(OrcMatrix), P, P, P,
                                    C.POINTER(OrcTrace)]
    L.orc_ffn_prefill.argtypes = [C.POINTER(OrcLayer), P, C.c_int, P]
    L.orc_rmsnorm_bf16.argtypes = [P, C.c_int, P]
    L.orc_rmsnorm_bf16.restype = None
    L.orc_quantize_expert.argtypes = [C.c_int, C.c_int, C.c_int, P, P, P, P]


def _p(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _chk(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with status {rc}")


# ---------------------------------------------------------------- conversions
def f32_to_f16(x: float) -> int:
    return int(lib().orc_f32_to_f16(float(x)))


def f16_to_f64(h: int) -> float:
    return float(lib().orc_f16_to_f64(int(h)))


def f16_array_to_f64(h: np.ndarray) -> np.ndarray:
    f = lib().orc_f16_to_f64
    return np.array([f(int(v)) for v in np.asarray(h).ravel()], dtype=np.float64).reshape(
        np.asarray(h).shape)


def f32_to_bf16(x: float) -> int:
    return int(lib().orc_f32_to_bf16(float(x)))


# ---------------------------------------------------------------- packing
BLOCK_BYTES = {2: 8, 3: 12, 4: 16}


def packed_bytes(fmt: int, rows: int, cols: int):
    cb, sb = C.c_size_t(), C.c_size_t()
    _chk(lib().orc_packed_bytes(fmt, rows, cols, C.byref(cb), C.byref(sb)), "packed_bytes")
    return cb.value, sb.value


def pack(fmt: int, codes: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    rows, cols = codes.shape
    nbytes, _ = packed_bytes(fmt, rows, cols)
    out = np.zeros(nbytes, dtype=np.uint8)
    _chk(lib().orc_pack(fmt, rows, cols, _p(codes), _p(out)), "pack")
    return out


def unpack(fmt: int, rows: int, cols: int, packed: np.ndarray) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.zeros((rows, cols), dtype=np.uint8)
    _chk(lib().orc_unpack(fmt, rows, cols, _p(packed), _p(out)), "unpack")
    return out


def scale_values(fmt: int, scales: np.ndarray) -> np.ndarray:
    scales = np.ascontiguousarray(scales)
    f = lib().orc_scale_value
    return np.array([f(fmt, _p(scales), i) for i in range(scales.size)]).reshape(scales.shape)


# ---------------------------------------------------------------- activations
def q8(v: np.ndarray):
    v = np.ascontiguousarray(v, dtype=np.float32).ravel()
    assert v.size % 32 == 0
    q = np.zeros(v.size, dtype=np.int8)
    d = np.zeros(v.size // 32, dtype=np.uint16)
    lib().orc_q8(_p(v), v.size, _p(q), _p(d))
    return q, d


def h32_f32(v: np.ndarray, signs: Optional[np.ndarray]) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32).ravel()
    out = np.zeros_like(v)
    s = None if signs is None else np.ascontiguousarray(signs, dtype=np.uint32)
    lib().orc_h32_f32(_p(v), _p(s), v.size // 32, _p(out))
    return out


def h32_f64(v: np.ndarray, signs: Optional[np.ndarray]) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64).ravel()
    out = np.zeros_like(v)
    s = None if signs is None else np.ascontiguousarray(signs, dtype=np.uint32)
    lib().orc_h32_f64(_p(v), _p(s), v.size // 32, _p(out))
    return out


def router_logits(x_bf16: np.ndarray, wr_bf16: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    w = np.ascontiguousarray(wr_bf16, dtype=np.uint16)
    E, H = w.shape
    T = x.size // H
    out = np.zeros((T, E), dtype=np.float32)
    lib().orc_router(_p(x), T, _p(w), E, H, _p(out))
    return out


def topk(logits: np.ndarray, k: int):
    l = np.ascontiguousarray(logits, dtype=np.float32).ravel()
    idx = np.zeros(k, dtype=np.int32)
    p = np.zeros(k, dtype=np.float64)
    lib().orc_topk(_p(l), l.size, k, _p(idx), _p(p))
    return idx, p


def rmsnorm_bf16(r: np.ndarray) -> np.ndarray:
    r = np.ascontiguousarray(r, dtype=np.float32).ravel()
    a = np.zeros(r.size, dtype=np.uint16)
    lib().orc_rmsnorm_bf16(_p(r), r.size, _p(a))
    return a


# ---------------------------------------------------------------- matrices and layers
@dataclass
class Matrix:
    """One role of a layer on the host: packed code planes, scale planes and
    codebooks per expert (only the experts that were materialized)."""
    fmt: int
    rows: int
    cols: int
    E: int
    codes: Dict[int, np.ndarray] = field(default_factory=dict)
    scales: Dict[int, np.ndarray] = field(default_factory=dict)
    cb: Dict[int, np.ndarray] = field(default_factory=dict)

    def c_struct(self, keep: list) -> OrcMatrix:
        def arr(d):
            a = (P * self.E)()
            for e, v in d.items():
                v = np.ascontiguousarray(v)
                keep.append(v)
                a[e] = v.ctypes.data
            keep.append(a)
            return C.cast(a, P)
        return OrcMatrix(self.fmt, self.rows, self.cols, arr(self.codes), arr(self.scales),
                         arr(self.cb))


@dataclass
class Layer:
    H: int
    I: int
    E: int
    k: int
    router: np.ndarray          # bf16 bits [E, H]
    gate: Matrix
    up: Matrix
    down: Matrix
    shared: Optional[tuple] = None   # (gate, up, down) Matrix with E = 1
    signs_x: Optional[np.ndarray] = None
    signs_h: Optional[np.ndarray] = None

    def c_struct(self, keep: list) -> OrcLayer:
        L = OrcLayer()
        L.H, L.I, L.E, L.k = self.H, self.I, self.E, self.k
        r = np.ascontiguousarray(self.router, dtype=np.uint16)
        keep.append(r)
        L.router = r.ctypes.data
        L.gate = self.gate.c_struct(keep)
        L.up = self.up.c_struct(keep)
        L.down = self.down.c_struct(keep)
        if self.shared is not None:
            L.has_shared = 1
            L.sgate = self.shared[0].c_struct(keep)
            L.sup = self.shared[1].c_struct(keep)
            L.sdown = self.shared[2].c_struct(keep)
        for name in ("signs_x", "signs_h"):
            v = getattr(self, name)
            if v is not None:
                v = np.ascontiguousarray(v, dtype=np.uint32)
                keep.append(v)
                setattr(L, name, v.ctypes.data)
        return L


def matvec(m: Matrix, expert: int, q: np.ndarray, d: np.ndarray, partials: bool = False):
    keep = []
    cm = m.c_struct(keep)
    q = np.ascontiguousarray(q, dtype=np.int8)
    d = np.ascontiguousarray(d, dtype=np.uint16)
    out = np.zeros(m.rows, dtype=np.float64)
    S = np.zeros((m.rows, m.cols // 32), dtype=np.int32) if partials else None
    _chk(lib().orc_matvec(C.byref(cm), expert, _p(q), _p(d), _p(out), _p(S)), "matvec")
    return (out, S) if partials else out


def _trace_arrays(L: Layer, full: bool):
    H, I, E, k = L.H, L.I, L.E, L.k
    n = k + 1
    t = dict(xq=np.zeros(H, np.int8), xd=np.zeros(H // 32, np.uint16),
             logits=np.zeros(E, np.float32), idx=np.zeros(k, np.int32), p=np.zeros(k, np.float64),
             g=np.zeros((n, I)), u=np.zeros((n, I)), h=np.zeros((n, I)),
             hq=np.zeros((n, I), np.int8), hd=np.zeros((n, I // 32), np.uint16),
             o=np.zeros((n, H)))
    if full:
        t.update(S_gate=np.zeros((n, I, H // 32), np.int32), S_up=np.zeros((n, I, H // 32), np.int32),
                 S_down=np.zeros((n, H, I // 32), np.int32))
    return t


def ffn_decode(L: Layer, x_bf16: np.ndarray, trace: bool = False, partials: bool = False,
               force_hq: Optional[np.ndarray] = None, force_hd: Optional[np.ndarray] = None,
               force_idx: Optional[np.ndarray] = None):
    """y (fp64 [H]) for one token; with trace=True also a dict of intermediates."""
    keep = []
    cl = L.c_struct(keep)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16).ravel()
    y = np.zeros(L.H, dtype=np.float64)
    tr = OrcTrace()
    arrays = _trace_arrays(L, partials) if trace else {}
    for name, a in arrays.items():
        setattr(tr, name, a.ctypes.data)
    for name, a, dt in (("force_hq", force_hq, np.int8), ("force_hd", force_hd, np.uint16),
                        ("force_idx", force_idx, np.int32)):
        if a is not None:
            a = np.ascontiguousarray(a, dtype=dt)
            keep.append(a)
            setattr(tr, name, a.ctypes.data)
    _chk(lib().orc_ffn_decode(C.byref(cl), _p(x), _p(y), C.byref(tr)), "ffn_decode")
    return (y, arrays) if trace else y


def ffn_verify_q4(L: Layer, dense: Optional[Matrix], x_bf16: np.ndarray):
    keep = []
    cl = L.c_struct(keep)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16).ravel()
    y = np.zeros((4, L.H), dtype=np.float64)
    yd = np.zeros((4, dense.rows), dtype=np.float64) if dense is not None else None
    cd = C.byref(dense.c_struct(keep)) if dense is not None else None
    _chk(lib().orc_ffn_verify_q4(C.byref(cl), cd, _p(x), _p(y), _p(yd), None), "verify_q4")
    return y, yd


def ffn_prefill(L: Layer, x_bf16: np.ndarray):
    keep = []
    cl = L.c_struct(keep)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    T = x.size // L.H
    y = np.zeros((T, L.H), dtype=np.float64)
    _chk(lib().orc_ffn_prefill(C.byref(cl), _p(x), T, _p(y)), "ffn_prefill")
    return y


def quantize_expert(fmt: int, w: np.ndarray):
    """Codebook quantization of one expert matrix (fp32 [rows, cols]) -> codes
    (uint8 [rows, cols]), scales (fp16 bits uint16 or E8M0 uint8 [rows, cols/32])
    and the codebook (int8 [2^fmt]); see orc_quantize_expert."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, cols = w.shape
    codes = np.zeros((rows, cols), np.uint8)
    scales = np.zeros((rows, cols // 32), np.uint8 if fmt == 4 else np.uint16)
    cb = np.zeros(1 << fmt, np.int8)
    _chk(lib().orc_quantize_expert(fmt, rows, cols, _p(w), _p(codes), _p(scales), _p(cb)), "quantize_expert")
    return codes, scales, cb
