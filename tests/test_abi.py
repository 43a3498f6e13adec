"""The C-ABI library builds, loads and exports every declared symbol; host-side
descriptor validation returns the documented codes (no GPU work)."""
import ctypes as C
import os
import re

import pytest

import bit_codebook_quantized_dequant_gb300 as M

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in ("moeq.h", "moeq_synth.h"):
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", src, re.M):
            names.add(m.group(1))
    return names


def test_library_exports_every_declared_symbol():
    lib = M.load()
    names = _declared()
    assert {"moe_pack_expert", "moe_route_topk", "moe_ffn_decode", "moe_ffn_verify_q4",
            "moe_ffn_prefill", "h32_rotate"} <= names
    for n in names:
        assert hasattr(lib, n), n
    assert set(M.EXPORTED) == names
    assert M.moeq_version().startswith("moeq")


def test_packed_bytes():
    assert M.moeq_packed_bytes(2, 2048, 4096) == (2048 * 128 * 8, 2048 * 128 * 2)
    assert M.moeq_packed_bytes(3, 4096, 2048) == (4096 * 64 * 12, 4096 * 64 * 2)
    assert M.moeq_packed_bytes(4, 2048, 4096) == (2048 * 128 * 16, 2048 * 128)
    # unpacked bf16 rows: two bytes per weight, no scale plane
    assert M.moeq_packed_bytes(M.MOEQ_BF16, 256, 4096) == (256 * 4096 * 2, 0)
    with pytest.raises(M.MoeqError):
        M.moeq_packed_bytes(5, 1, 32)
    # no packed role takes MOEQ_BF16
    assert M.moeq_validate_layer(_layer(gate=_mat(M.MOEQ_BF16, 256, 256, 16))) == M.CODE["MOEQ_ERR_FORMAT"]


FAKE = 1 << 40  # aligned fake device address: validation never dereferences


def _mat(fmt, rows, cols, E, **kw):
    cb, sb = M.moeq_packed_bytes(fmt, rows, cols)
    d = dict(fmt=fmt, rows=rows, cols=cols, num_experts=E, codes=FAKE, expert_stride_codes=cb,
             scales=FAKE, expert_stride_scales=(sb + 15) // 16 * 16, codebooks=FAKE,
             cb_len=1 << (3 if fmt == M.MOEQ_FP3_PACKED24 else fmt), cb_stride=16)
    d.update(kw)
    return M.MoeqMatrix(**d)


def _layer(**over):
    L = M.MoeqLayer()
    L.H, L.I, L.E, L.k = 256, 256, 16, 2
    L.router = FAKE
    L.gate = _mat(2, 256, 256, 16)
    L.up = _mat(2, 256, 256, 16)
    L.down = _mat(3, 256, 256, 16)
    for k, v in over.items():
        setattr(L, k, v)
    return L


def test_validation_codes():
    assert M.moeq_validate_layer(_layer()) == 0
    assert M.moe_ffn_workspace(_layer(), 1, 0) > 0
    cases = {
        "MOEQ_ERR_CODEBOOK_MISSING": dict(gate=_mat(2, 256, 256, 16, codebooks=None)),
        "MOEQ_ERR_CODEBOOK_TRUNCATED": dict(down=_mat(3, 256, 256, 16, cb_len=4)),
        "MOEQ_ERR_CODEBOOK_MISMATCH": dict(up=_mat(2, 256, 256, 16, cb_len=8)),
        "MOEQ_ERR_CODEBOOK_DUPLICATE": dict(gate=_mat(2, 256, 256, 16, cb_stride=0)),
        "MOEQ_ERR_FORMAT": dict(gate=M.MoeqMatrix(5, 256, 256, 16, FAKE, 1 << 20, FAKE, 1 << 20,
                                                  FAKE, 32, 32)),
        "MOEQ_ERR_SHAPE": dict(H=200),
        "MOEQ_ERR_ALIGN": dict(router=FAKE + 8),
        "MOEQ_ERR_ARG": dict(k=0),
    }
    for code, over in cases.items():
        assert M.moeq_validate_layer(_layer(**over)) == M.CODE[code], code
    assert M.moeq_validate_layer(_layer(k=17)) == M.CODE["MOEQ_ERR_ARG"]
    # codebook records must be 16-byte aligned and strided
    assert M.moeq_validate_layer(_layer(gate=_mat(2, 256, 256, 16, cb_stride=20))) == \
        M.CODE["MOEQ_ERR_ALIGN"]
    assert M.moeq_validate_layer(_layer(gate=_mat(2, 256, 256, 16, codebooks=FAKE + 4))) == \
        M.CODE["MOEQ_ERR_ALIGN"]
    assert M.moe_ffn_workspace(_layer(H=200), 1, 0) == 0
    # a gate/up format mismatch is a format error
    assert M.moeq_validate_layer(_layer(up=_mat(4, 256, 256, 16))) == M.CODE["MOEQ_ERR_FORMAT"]


def test_entry_points_reject_bad_arguments_before_launch():
    lib = M.load()
    L = _layer()
    # NULL x / y and a NULL workspace are rejected synchronously, nothing enqueued
    assert lib.moe_ffn_decode(C.byref(L), None, None, None, 0, None, None, None) == \
        M.CODE["MOEQ_ERR_ARG"]
    assert lib.moe_ffn_decode(C.byref(L), FAKE, FAKE, None, 0, None, None, None) == \
        M.CODE["MOEQ_ERR_WORKSPACE"]
    assert lib.moe_pack_expert(7, 1, 32, FAKE, FAKE, FAKE, FAKE, None, None) == \
        M.CODE["MOEQ_ERR_FORMAT"]
    assert lib.moe_pack_expert(2, 1, 32, FAKE + 4, FAKE, FAKE, FAKE, None, None) == \
        M.CODE["MOEQ_ERR_ALIGN"]
    assert lib.moe_route_topk(FAKE, 1, FAKE, 16, 100, 2, FAKE, FAKE, None, None, None) == \
        M.CODE["MOEQ_ERR_SHAPE"]
    assert lib.moe_route_topk(FAKE, 1, FAKE, 16, 256, 9, FAKE, FAKE, None, None, None) == \
        M.CODE["MOEQ_ERR_ARG"]
    # q=4 verification: dense projection shape, its output and the workspace
    dense_bad = _mat(4, 256, 512, 1)   # cols != H
    dense_ok = _mat(4, 256, 256, 1)
    assert lib.moe_ffn_verify_q4(C.byref(L), C.byref(dense_bad), FAKE, FAKE, FAKE, FAKE, 1 << 30,
                                 None, None, None) == M.CODE["MOEQ_ERR_SHAPE"]
    assert lib.moe_ffn_verify_q4(C.byref(L), C.byref(dense_ok), FAKE, FAKE, None, FAKE, 1 << 30,
                                 None, None, None) == M.CODE["MOEQ_ERR_ARG"]
    assert lib.moe_ffn_verify_q4(C.byref(L), None, FAKE, FAKE, None, FAKE, 16, None, None,
                                 None) == M.CODE["MOEQ_ERR_WORKSPACE"]
    need4 = lib.moe_ffn_workspace(C.byref(L), 4, 1)
    need1 = lib.moe_ffn_workspace(C.byref(L), 1, 0)
    assert need4 > need1 > 0
    # library-owned scratch: a decode shape whose workspace exceeds 160 KiB is
    # rejected before anything is enqueued
    big = _layer(H=4096, I=4096, E=16, k=8)
    big.gate = _mat(2, 4096, 4096, 16)
    big.up = _mat(2, 4096, 4096, 16)
    big.down = _mat(3, 4096, 4096, 16)
    assert lib.moe_ffn_workspace(C.byref(big), 1, 0) > 160 * 1024
    assert lib.moe_ffn_decode_static(C.byref(big), FAKE, FAKE, None, None) == \
        M.CODE["MOEQ_ERR_WORKSPACE"]
    assert lib.moe_ffn_decode_static(C.byref(L), None, FAKE, None, None) == M.CODE["MOEQ_ERR_ARG"]
    # decode stack: layers, then the workspace (decode + a + y for the largest layer)
    assert lib.moe_ffn_stack_decode(None, 1, FAKE, FAKE, FAKE, 1 << 30, None, None) == M.CODE["MOEQ_ERR_ARG"]
    arr = (M.MoeqLayer * 2)(L, L)
    need_s = lib.moe_ffn_workspace(C.byref(L), 1, 4)
    assert need_s > need1
    assert lib.moe_ffn_stack_decode(arr, 2, FAKE, FAKE, FAKE, need_s - 16, None, None) == \
        M.CODE["MOEQ_ERR_WORKSPACE"]
    assert lib.moe_ffn_stack_decode(arr, 2, FAKE + 8, FAKE, FAKE, need_s, None, None) == M.CODE["MOEQ_ERR_ALIGN"]
    # q=4 stack: q=4 workspace + a [4 x H] + y [4 x H] for the largest layer
    assert lib.moe_ffn_stack_verify_q4(None, 1, FAKE, FAKE, FAKE, 1 << 30, None, None) == M.CODE["MOEQ_ERR_ARG"]
    need_q = lib.moe_ffn_workspace(C.byref(L), 1, 5)
    assert need_q == need4 + 8 * L.H + 16 * L.H
    assert lib.moe_ffn_stack_verify_q4(arr, 2, FAKE, FAKE, FAKE, need_q - 16, None, None) == \
        M.CODE["MOEQ_ERR_WORKSPACE"]
    assert lib.moe_ffn_stack_verify_q4(arr, 2, FAKE, FAKE + 4, FAKE, need_q, None, None) == \
        M.CODE["MOEQ_ERR_ALIGN"]
    other = (M.MoeqLayer * 2)(L, _layer(H=2 * L.H))
    assert lib.moe_ffn_stack_verify_q4(other, 2, FAKE, FAKE, FAKE, 1 << 30, None, None) != M.CODE["MOEQ_OK"]
    assert lib.h32_rotate(None, None, 4, None, None) == M.CODE["MOEQ_ERR_ARG"]
    assert lib.moe_rmsnorm_bf16(FAKE, 1, 100, FAKE, None) == M.CODE["MOEQ_ERR_SHAPE"]


def test_packed24_layout_accepted_for_routed_down_only():
    P24 = M.MOEQ_FP3_PACKED24
    assert M.moeq_packed_bytes(P24, 4096, 2048) == M.moeq_packed_bytes(3, 4096, 2048)
    assert M.moeq_validate_layer(_layer(down=_mat(P24, 256, 256, 16))) == 0
    assert M.moeq_validate_layer(_layer(down=_mat(P24, 256, 256, 16, cb_len=16))) == \
        M.CODE["MOEQ_ERR_CODEBOOK_MISMATCH"]
    assert M.moeq_validate_layer(_layer(gate=_mat(P24, 256, 256, 16), up=_mat(P24, 256, 256, 16))) == \
        M.CODE["MOEQ_ERR_FORMAT"]
    sh = _layer(has_shared=1, sgate=_mat(4, 256, 256, 1), sup=_mat(4, 256, 256, 1),
                sdown=_mat(P24, 256, 256, 1))
    assert M.moeq_validate_layer(sh) == M.CODE["MOEQ_ERR_FORMAT"]
    lib = M.load()
    L = _layer(down=_mat(P24, 256, 256, 16))
    need = lib.moe_ffn_workspace(C.byref(L), 8, 2)
    # the prefill's tensor-core GEMM does not decode the layout: rejected before any launch
    assert lib.moe_ffn_prefill(C.byref(L), FAKE, 8, None, FAKE, FAKE, need, None, None, None) == \
        M.CODE["MOEQ_ERR_FORMAT"]
    assert lib.moe_ffn_stack_prefill((M.MoeqLayer * 1)(L), 1, FAKE, 8, FAKE, FAKE, 1 << 40, None, None) == \
        M.CODE["MOEQ_ERR_FORMAT"]
    # nor does the q=4 dense projection
    dense = _mat(P24, 256, 256, 1)
    assert lib.moe_ffn_verify_q4(C.byref(_layer()), C.byref(dense), FAKE, FAKE, FAKE, FAKE, 1 << 30, None,
                                 None, None) == M.CODE["MOEQ_ERR_FORMAT"]


def test_prefill_entry_points_reject_bad_arguments_before_launch():
    lib = M.load()
    L = _layer()
    need = lib.moe_ffn_workspace(C.byref(L), 8, 2)
    assert need > 0

    def prefill(x=FAKE, T=8, residual=None, y=FAKE, ws=FAKE, ws_bytes=need, layer=L):
        return lib.moe_ffn_prefill(C.byref(layer), x, T, residual, y, ws, ws_bytes, None, None, None)

    assert prefill(layer=_layer(k=0)) == M.CODE["MOEQ_ERR_ARG"]       # the layer is validated first
    assert prefill(T=-1) == M.CODE["MOEQ_ERR_SHAPE"]
    assert prefill(T=0, x=None, y=None, ws=None) == 0                 # T = 0 enqueues nothing
    assert prefill(x=None) == M.CODE["MOEQ_ERR_ARG"]
    assert prefill(y=None) == M.CODE["MOEQ_ERR_ARG"]
    assert prefill(x=FAKE + 8) == M.CODE["MOEQ_ERR_ALIGN"]
    assert prefill(residual=FAKE + 4) == M.CODE["MOEQ_ERR_ALIGN"]
    assert prefill(ws_bytes=need - 1) == M.CODE["MOEQ_ERR_WORKSPACE"]
    assert prefill(ws=None) == M.CODE["MOEQ_ERR_WORKSPACE"]
    assert prefill(ws=FAKE + 8) == M.CODE["MOEQ_ERR_WORKSPACE"]
    # a larger T needs a larger workspace
    assert lib.moe_ffn_workspace(C.byref(L), 9, 2) > need

    # the layer stack: every layer validated, one H, workspace for the largest layer + the RMSNorm output
    arr = (M.MoeqLayer * 2)(_layer(), _layer())
    need3 = lib.moe_ffn_workspace(C.byref(L), 8, 3)
    assert need3 > need

    def stack(layers=arr, n=2, x=FAKE, T=8, r=FAKE, ws=FAKE, ws_bytes=need3):
        return lib.moe_ffn_stack_prefill(layers, n, x, T, r, ws, ws_bytes, None, None)

    assert stack(layers=None) == M.CODE["MOEQ_ERR_ARG"]
    assert stack(n=0) == M.CODE["MOEQ_ERR_ARG"]
    assert stack(T=-1) == M.CODE["MOEQ_ERR_SHAPE"]
    assert stack(layers=(M.MoeqLayer * 2)(_layer(), _layer(k=0))) == M.CODE["MOEQ_ERR_ARG"]
    wide = _layer(H=512)
    wide.router = FAKE
    wide.gate, wide.up, wide.down = _mat(2, 256, 512, 16), _mat(2, 256, 512, 16), _mat(3, 512, 256, 16)
    assert M.moeq_validate_layer(wide) == 0
    assert stack(layers=(M.MoeqLayer * 2)(_layer(), wide)) == M.CODE["MOEQ_ERR_SHAPE"]  # one H
    assert stack(T=0, x=None, r=None, ws=None) == 0
    assert stack(r=None) == M.CODE["MOEQ_ERR_ARG"]
    assert stack(x=FAKE + 2) == M.CODE["MOEQ_ERR_ALIGN"]
    assert stack(ws_bytes=need3 - 1) == M.CODE["MOEQ_ERR_WORKSPACE"]


def test_quantizer_and_expansion_reject_bad_arguments_before_launch():
    lib = M.load()
    # moe_quantize_expert: fmt 2, 3 or 4; cols % 32; pointers; alignment; >= 1 KiB of workspace
    def quant(fmt=2, rows=4, cols=64, w=FAKE, codes=FAKE, scales=FAKE, cb=FAKE, ws=FAKE, ws_bytes=1024):
        return lib.moe_quantize_expert(fmt, rows, cols, w, codes, scales, cb, ws, ws_bytes, None, None)

    assert quant(fmt=5) == M.CODE["MOEQ_ERR_FORMAT"]
    assert quant(fmt=M.MOEQ_FP3_PACKED24) == M.CODE["MOEQ_ERR_FORMAT"]   # a layout, not a code width
    assert quant(cols=100) == M.CODE["MOEQ_ERR_SHAPE"]
    assert quant(rows=0) == M.CODE["MOEQ_ERR_SHAPE"]
    assert quant(rows=1 << 16, cols=1 << 15) == M.CODE["MOEQ_ERR_SHAPE"]  # 2^31 weights
    assert quant(w=None) == M.CODE["MOEQ_ERR_ARG"]
    assert quant(cb=None) == M.CODE["MOEQ_ERR_ARG"]
    assert quant(w=FAKE + 4) == M.CODE["MOEQ_ERR_ALIGN"]
    assert quant(ws_bytes=1019) == M.CODE["MOEQ_ERR_WORKSPACE"]
    assert quant(ws=None) == M.CODE["MOEQ_ERR_WORKSPACE"]
    # moe_expand_bf16: a packed matrix, an expert range inside it, an aligned output
    m = _mat(2, 256, 256, 16)
    assert lib.moe_expand_bf16(None, 0, 1, FAKE, None) == M.CODE["MOEQ_ERR_ARG"]
    assert lib.moe_expand_bf16(C.byref(m), 0, 1, None, None) == M.CODE["MOEQ_ERR_ARG"]
    bad = M.MoeqMatrix(5, 256, 256, 16, FAKE, 1 << 20, FAKE, 1 << 20, FAKE, 32, 32)
    assert lib.moe_expand_bf16(C.byref(bad), 0, 1, FAKE, None) == M.CODE["MOEQ_ERR_FORMAT"]
    assert lib.moe_expand_bf16(C.byref(m), 10, 7, FAKE, None) == M.CODE["MOEQ_ERR_ARG"]
    assert lib.moe_expand_bf16(C.byref(m), -1, 1, FAKE, None) == M.CODE["MOEQ_ERR_ARG"]
    assert lib.moe_expand_bf16(C.byref(m), 0, 1, FAKE + 2, None) == M.CODE["MOEQ_ERR_ALIGN"]
    assert lib.moe_expand_bf16(C.byref(m), 3, 0, FAKE, None) == 0   # nothing to expand
    # moe_ffn_expanded_workspace: idx, p, the arrival counter, logits [E], h [(k + shared) x I]
    need = lib.moe_ffn_expanded_workspace(4096, 2048, 256, 6, 1)
    assert need == 3 * 256 + 1024 + 7 * 2048 * 4
    assert lib.moe_ffn_expanded_workspace(4096, 2048, 0, 6, 1) == 0
    assert lib.moe_ffn_expanded_workspace(4096, 2048, 4, 6, 1) == 0    # k > E
    assert lib.moe_ffn_expanded_workspace(4096, 2048, 2048, 6, 1) == 0  # E > 1024

    # moe_ffn_decode_expanded: MOEQ_BF16 matrices of the layer's shapes, no rotation
    def bf(rows, cols, E):
        return M.MoeqMatrix(M.MOEQ_BF16, rows, cols, E, FAKE, 2 * rows * cols, None, 0, None, 0, 0)

    L = _layer(gate=bf(256, 256, 16), up=bf(256, 256, 16), down=bf(256, 256, 16))
    wsb = lib.moe_ffn_expanded_workspace(256, 256, 16, 2, 0)

    def dec(layer=L, x=FAKE, y=FAKE, ws=FAKE, ws_bytes=wsb):
        return lib.moe_ffn_decode_expanded(C.byref(layer), x, y, ws, ws_bytes, None, None)

    assert lib.moe_ffn_decode_expanded(None, FAKE, FAKE, FAKE, wsb, None, None) == M.CODE["MOEQ_ERR_ARG"]
    assert dec(x=None) == M.CODE["MOEQ_ERR_ARG"]
    assert dec(layer=_layer(H=200, gate=bf(256, 200, 16), up=bf(256, 200, 16), down=bf(200, 256, 16))) == \
        M.CODE["MOEQ_ERR_SHAPE"]
    assert dec(layer=_layer(gate=bf(256, 256, 16), up=bf(256, 256, 16), down=bf(256, 256, 16),
                            h32_signs_x=FAKE)) == M.CODE["MOEQ_ERR_FORMAT"]
    assert dec(layer=_layer()) == M.CODE["MOEQ_ERR_FORMAT"]            # packed matrices
    assert dec(layer=_layer(gate=bf(256, 256, 16), up=bf(128, 256, 16), down=bf(256, 256, 16))) == \
        M.CODE["MOEQ_ERR_SHAPE"]
    assert dec(y=FAKE + 4) == M.CODE["MOEQ_ERR_ALIGN"]
    assert dec(ws_bytes=wsb - 1) == M.CODE["MOEQ_ERR_WORKSPACE"]
    assert dec(ws=None) == M.CODE["MOEQ_ERR_WORKSPACE"]
