"""GPU parity of the codebook quantizer (moe_quantize_expert) against the
oracle's: codes, block scales and codebook bit for bit, on seeded Gaussian
weights of the decode layer's matrix shapes and on a matrix built from a known
codebook (which both must recover), then packed and read back."""
import numpy as np
import pytest
import torch

import oracle as O
import bit_codebook_quantized_dequant_gb300 as M

pytestmark = pytest.mark.gpu


def _gpu_quantize(fmt, w):
    rows, cols = w.shape
    wd = torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32)).cuda()
    codes = torch.zeros(rows * cols, dtype=torch.uint8, device="cuda")
    sdt = torch.uint8 if fmt == 4 else torch.int16
    scales = torch.zeros(rows * (cols // 32), dtype=sdt, device="cuda")
    cb = torch.zeros(1 << fmt, dtype=torch.int8, device="cuda")
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_quantize_expert(fmt, rows, cols, wd, codes, scales, cb, ws, ws.numel(), st)
    torch.cuda.synchronize()
    assert st.item() == 0
    s = scales.cpu().numpy()
    return (codes.cpu().numpy().reshape(rows, cols),
            (s if fmt == 4 else s.view(np.uint16)).reshape(rows, cols // 32),
            cb.cpu().numpy())


@pytest.mark.parametrize("fmt,rows,cols", [(2, 2048, 4096), (3, 4096, 2048), (4, 2048, 4096), (2, 37, 96)])
def test_quantizer_matches_oracle_on_gaussian_weights(fmt, rows, cols):
    rng = np.random.default_rng(1000 + 7 * fmt + rows)
    w = (rng.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    w[0, :32] = 0.0   # an all-zero block
    w[1, 5] = 3.0     # one outlier block
    c_ref, s_ref, cb_ref = O.quantize_expert(fmt, w)
    c, s, cb = _gpu_quantize(fmt, w)
    np.testing.assert_array_equal(cb, cb_ref)
    np.testing.assert_array_equal(s, s_ref)
    np.testing.assert_array_equal(c, c_ref)


@pytest.mark.parametrize("fmt", [2, 3, 4])
def test_quantizer_recovers_known_codebook_and_packs(fmt):
    rng = np.random.default_rng(40 + fmt)
    rows, cols, K = 256, 512, 1 << fmt
    cb_true = np.concatenate([[-127], np.sort(rng.choice(np.arange(-120, 121), K - 2, replace=False)),
                              [127]]).astype(np.int8)
    codes_true = rng.integers(0, K, size=(rows, cols)).astype(np.uint8)
    codes_true[:, ::32] = K - 1
    if fmt == 4:
        d = np.ldexp(1.0, rng.integers(-20, -5, size=(rows, cols // 32))).astype(np.float32)
    else:
        d = np.float16(rng.uniform(1e-4, 1e-2, size=(rows, cols // 32))).astype(np.float32)
    w = cb_true.astype(np.float32)[codes_true] * np.repeat(d, 32, axis=1)
    c, s, cb = _gpu_quantize(fmt, w)
    np.testing.assert_array_equal(cb, cb_true)
    np.testing.assert_array_equal(c, codes_true)
    # the quantizer's output packs to the oracle's block layout
    cbytes, sbytes = M.moeq_packed_bytes(fmt, rows, cols)
    out_c = torch.zeros(cbytes, dtype=torch.uint8, device="cuda")
    out_s = torch.zeros(sbytes, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_pack_expert(fmt, rows, cols, torch.from_numpy(c).cuda(),
                      torch.from_numpy(s.view(np.uint8).copy()).cuda(), out_c, out_s, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    np.testing.assert_array_equal(out_c.cpu().numpy(), O.pack(fmt, c).ravel())
