"""Python binding of libmoeq (include/moeq.h, include/moeq_synth.h).

Argument marshalling only: every step of the FFN runs in the CUDA library.
Device buffers are passed as integers (device addresses) or torch tensors;
streams as torch.cuda.Stream, an integer handle or None (current stream).
Importing does not load the library; the first call does, and it raises if the
library is missing or cannot be built -- there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoeq.so")

MOEQ_FP2, MOEQ_FP3, MOEQ_FP4, MOEQ_BF16, MOEQ_FP3_PACKED24 = 2, 3, 4, 16, 24
STATUS = {
    0: "MOEQ_OK", -1: "MOEQ_ERR_ARG", -2: "MOEQ_ERR_SHAPE", -3: "MOEQ_ERR_ALIGN",
    -4: "MOEQ_ERR_FORMAT", -5: "MOEQ_ERR_CODEBOOK_MISSING", -6: "MOEQ_ERR_CODEBOOK_TRUNCATED",
    -7: "MOEQ_ERR_CODEBOOK_MISMATCH", -8: "MOEQ_ERR_CODEBOOK_DUPLICATE", -9: "MOEQ_ERR_WORKSPACE",
    -10: "MOEQ_ERR_CUDA", -11: "MOEQ_ERR_DEVICE_TIMEOUT", -12: "MOEQ_ERR_DEVICE_INDEX",
}
CODE = {v: k for k, v in STATUS.items()}


class MoeqError(RuntimeError):
    def __init__(self, what: str, rc: int):
        super().__init__(f"{what} returned {rc} ({STATUS.get(rc, '?')})")
        self.rc = rc


P = C.c_void_p


class MoeqMatrix(C.Structure):
    _fields_ = [("fmt", C.c_int), ("rows", C.c_int), ("cols", C.c_int), ("num_experts", C.c_int),
                ("codes", P), ("expert_stride_codes", C.c_size_t), ("scales", P),
                ("expert_stride_scales", C.c_size_t), ("codebooks", P), ("cb_len", C.c_int),
                ("cb_stride", C.c_int)]


class MoeqLayer(C.Structure):
    _fields_ = [("H", C.c_int), ("I", C.c_int), ("E", C.c_int), ("k", C.c_int), ("router", P),
                ("gate", MoeqMatrix), ("up", MoeqMatrix), ("down", MoeqMatrix),
                ("has_shared", C.c_int), ("sgate", MoeqMatrix), ("sup", MoeqMatrix),
                ("sdown", MoeqMatrix), ("h32_signs_x", P), ("h32_signs_h", P)]


class MoeqDebug(C.Structure):
    _fields_ = [(n, P) for n in ("xq", "xd", "logits", "idx", "p", "h", "hq", "hd", "o", "S_gate",
                                 "S_up", "S_down", "trace")] + [("trace_cap", C.c_int),
                                                                ("spin_limit", C.c_int)]


TRACE_EVENTS = {1: "START", 2: "TAKE", 3: "TOPK", 4: "ISSUED", 5: "READY", 6: "DONE",
                7: "EPI_BEGIN", 8: "EPI_END", 9: "SPIN"}


_lib = None
_lock = threading.Lock()


def load(build_if_missing: bool = True):
    """Loads libmoeq.so (building it with nvcc if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        from . import _build
        if build_if_missing and not _build.up_to_date():
            _build.build()
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmoeq.so not found at {LIB_PATH}; run __graft_entry__.build()")
        lib = C.CDLL(LIB_PATH)
        _declare(lib)
        _lib = lib
        return lib


def _declare(L):
    i, sz, u64 = C.c_int, C.c_size_t, C.c_uint64
    sig = {
        "moeq_packed_bytes": (i, [i, i, i, C.POINTER(sz), C.POINTER(sz)]),
        "moeq_validate_layer": (i, [C.POINTER(MoeqLayer)]),
        "moe_ffn_workspace": (sz, [C.POINTER(MoeqLayer), i, i]),
        "moe_ffn_workspace_init": (i, [P, sz, P]),
        "moe_pack_expert": (i, [i, i, i, P, P, P, P, P, P]),
        "moe_route_topk": (i, [P, i, P, i, i, i, P, P, P, P, P]),
        "moe_ffn_decode": (i, [C.POINTER(MoeqLayer), P, P, P, sz, P, C.POINTER(MoeqDebug), P]),
        "moe_ffn_decode_static": (i, [C.POINTER(MoeqLayer), P, P, P, P]),
        "moe_ffn_verify_q4": (i, [C.POINTER(MoeqLayer), C.POINTER(MoeqMatrix), P, P, P, P, sz, P,
                                  C.POINTER(MoeqDebug), P]),
        "moe_ffn_prefill": (i, [C.POINTER(MoeqLayer), P, i, P, P, P, sz, P, C.POINTER(MoeqDebug),
                                P]),
        "moe_ffn_stack_prefill": (i, [P, i, P, i, P, P, sz, P, P]),
        "moe_ffn_stack_decode": (i, [P, i, P, P, P, sz, P, P]),
        "moe_ffn_stack_verify_q4": (i, [P, i, P, P, P, sz, P, P]),
        "moe_quantize_expert": (i, [i, i, i, P, P, P, P, P, sz, P, P]),
        "moe_expand_bf16": (i, [P, i, i, P, P]),
        "moe_ffn_expanded_workspace": (sz, [i, i, i, i, i]),
        "moe_ffn_decode_expanded": (i, [P, P, P, P, sz, P, P]),
        "h32_rotate": (i, [P, P, i, P, P]),
        "moe_rmsnorm_bf16": (i, [P, i, i, P, P]),
        "moeq_version": (C.c_char_p, []),
        "moeq_synth_codes": (i, [u64, u64, i, sz, P, P]),
        "moeq_synth_scales": (i, [u64, u64, i, sz, P, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args


EXPORTED = ["moeq_packed_bytes", "moeq_validate_layer", "moe_ffn_workspace",
            "moe_ffn_workspace_init", "moe_pack_expert", "moe_route_topk", "moe_ffn_decode",
            "moe_ffn_decode_static",
            "moe_ffn_verify_q4", "moe_ffn_prefill", "moe_ffn_stack_prefill", "moe_ffn_stack_decode",
            "moe_ffn_stack_verify_q4", "moe_quantize_expert", "moe_expand_bf16", "moe_ffn_expanded_workspace",
            "moe_ffn_decode_expanded", "h32_rotate",
            "moe_rmsnorm_bf16",
            "moeq_version", "moeq_synth_codes", "moeq_synth_scales"]


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(name, rc):
    if rc != 0:
        raise MoeqError(name, rc)
    return rc


# ------------------------------------------------------------------ C-ABI wrappers
def moeq_packed_bytes(fmt: int, rows: int, cols: int):
    cb, sb = C.c_size_t(), C.c_size_t()
    _check("moeq_packed_bytes", load().moeq_packed_bytes(fmt, rows, cols, C.byref(cb), C.byref(sb)))
    return cb.value, sb.value


def moeq_validate_layer(layer: MoeqLayer) -> int:
    return load().moeq_validate_layer(C.byref(layer))


def moe_ffn_workspace(layer: MoeqLayer, T_max: int, mode: int) -> int:
    return load().moe_ffn_workspace(C.byref(layer), T_max, mode)


def moe_ffn_workspace_init(ws, nbytes: int, stream=None):
    _check("moe_ffn_workspace_init", load().moe_ffn_workspace_init(_ptr(ws), nbytes, _stream(stream)))


def moe_pack_expert(fmt, rows, cols, codes_u8, scales, out_codes, out_scales, dev_status=None,
                    stream=None):
    _check("moe_pack_expert", load().moe_pack_expert(fmt, rows, cols, _ptr(codes_u8), _ptr(scales),
                                                     _ptr(out_codes), _ptr(out_scales),
                                                     _ptr(dev_status), _stream(stream)))


def moe_route_topk(x, T, router, E, H, k, idx, w, logits=None, dev_status=None, stream=None):
    _check("moe_route_topk", load().moe_route_topk(_ptr(x), T, _ptr(router), E, H, k, _ptr(idx),
                                                   _ptr(w), _ptr(logits), _ptr(dev_status),
                                                   _stream(stream)))


def moe_ffn_decode(layer: MoeqLayer, x, y, ws, ws_bytes, dev_status=None, dbg=None, stream=None):
    return _check("moe_ffn_decode", load().moe_ffn_decode(
        C.byref(layer), _ptr(x), _ptr(y), _ptr(ws), ws_bytes, _ptr(dev_status),
        C.byref(dbg) if dbg is not None else None, _stream(stream)))


def moe_ffn_decode_static(layer: MoeqLayer, x, y, dev_status=None, stream=None):
    """moe_ffn_decode with the library's own per-device scratch (no workspace)."""
    return _check("moe_ffn_decode_static", load().moe_ffn_decode_static(
        C.byref(layer), _ptr(x), _ptr(y), _ptr(dev_status), _stream(stream)))


def moe_ffn_verify_q4(layer: MoeqLayer, dense, x, y, y_dense, ws, ws_bytes, dev_status=None,
                      dbg=None, stream=None):
    return _check("moe_ffn_verify_q4", load().moe_ffn_verify_q4(
        C.byref(layer), C.byref(dense) if dense is not None else None, _ptr(x), _ptr(y),
        _ptr(y_dense), _ptr(ws), ws_bytes, _ptr(dev_status),
        C.byref(dbg) if dbg is not None else None, _stream(stream)))


def moe_ffn_prefill(layer: MoeqLayer, x, T, residual, y, ws, ws_bytes, dev_status=None, dbg=None,
                    stream=None):
    return _check("moe_ffn_prefill", load().moe_ffn_prefill(
        C.byref(layer), _ptr(x), T, _ptr(residual), _ptr(y), _ptr(ws), ws_bytes, _ptr(dev_status),
        C.byref(dbg) if dbg is not None else None, _stream(stream)))


def moe_quantize_expert(fmt, rows, cols, w, codes_u8, scales, codebook, ws, ws_bytes, dev_status=None,
                        stream=None):
    return _check("moe_quantize_expert", load().moe_quantize_expert(
        fmt, rows, cols, _ptr(w), _ptr(codes_u8), _ptr(scales), _ptr(codebook), _ptr(ws), ws_bytes,
        _ptr(dev_status), _stream(stream)))


def moe_expand_bf16(matrix: MoeqMatrix, e0, ne, out_bf16, stream=None):
    return _check("moe_expand_bf16", load().moe_expand_bf16(C.byref(matrix), e0, ne, _ptr(out_bf16),
                                                            _stream(stream)))


def moe_ffn_expanded_workspace(H, I, E, k, has_shared) -> int:
    return load().moe_ffn_expanded_workspace(H, I, E, k, has_shared)


def moe_ffn_decode_expanded(layer: MoeqLayer, x, y, ws, ws_bytes, dev_status=None, stream=None):
    return _check("moe_ffn_decode_expanded", load().moe_ffn_decode_expanded(
        C.byref(layer), _ptr(x), _ptr(y), _ptr(ws), ws_bytes, _ptr(dev_status), _stream(stream)))


def moe_ffn_stack_decode(layers, x, r, ws, ws_bytes, dev_status=None, stream=None):
    """layers: a sequence of MoeqLayer (copied into one contiguous array)."""
    arr = (MoeqLayer * len(layers))(*layers)
    return _check("moe_ffn_stack_decode", load().moe_ffn_stack_decode(
        arr, len(layers), _ptr(x), _ptr(r), _ptr(ws), ws_bytes, _ptr(dev_status), _stream(stream)))


def moe_ffn_stack_verify_q4(layers, x, r, ws, ws_bytes, dev_status=None, stream=None):
    """layers: a sequence of MoeqLayer; x [4 x H] bf16, r [4 x H] fp32."""
    arr = (MoeqLayer * len(layers))(*layers)
    return _check("moe_ffn_stack_verify_q4", load().moe_ffn_stack_verify_q4(
        arr, len(layers), _ptr(x), _ptr(r), _ptr(ws), ws_bytes, _ptr(dev_status), _stream(stream)))


def moe_ffn_stack_prefill(layers, x, T, r, ws, ws_bytes, dev_status=None, stream=None):
    """layers: a sequence of MoeqLayer (copied into one contiguous array)."""
    arr = (MoeqLayer * len(layers))(*layers)
    return _check("moe_ffn_stack_prefill", load().moe_ffn_stack_prefill(
        arr, len(layers), _ptr(x), T, _ptr(r), _ptr(ws), ws_bytes, _ptr(dev_status),
        _stream(stream)))


def h32_rotate(inp, out, nblk, signs=None, stream=None):
    _check("h32_rotate", load().h32_rotate(_ptr(inp), _ptr(out), nblk, _ptr(signs), _stream(stream)))


def moe_rmsnorm_bf16(r, T, H, a, stream=None):
    _check("moe_rmsnorm_bf16", load().moe_rmsnorm_bf16(_ptr(r), T, H, _ptr(a), _stream(stream)))


def moeq_version() -> str:
    return load().moeq_version().decode()


def moeq_synth_codes(seed, stream_id, bits, n, out, stream=None):
    _check("moeq_synth_codes", load().moeq_synth_codes(seed, stream_id, bits, n, _ptr(out),
                                                       _stream(stream)))


def moeq_synth_scales(seed, stream_id, bits, n, out, stream=None):
    _check("moeq_synth_scales", load().moeq_synth_scales(seed, stream_id, bits, n, _ptr(out),
                                                         _stream(stream)))
