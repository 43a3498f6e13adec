"""GPU parity of the small entry points against the oracle, through the C ABI:
the generator twin, the packer, the H32 rotation, router + top-k, RMSNorm."""
import numpy as np
import pytest
import torch

import oracle as O
import bit_codebook_quantized_dequant_gb300 as M
from bit_codebook_quantized_dequant_gb300 import synth as S
from bit_codebook_quantized_dequant_gb300.workload import to_dev_u16, to_dev_u32

pytestmark = pytest.mark.gpu


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_generator_twin_matches_host(bits):
    seed, stream = S.workload_seed("decode-b1"), S.stream_id(3, S.ROLE_GATE, 77, S.KIND_CODES)
    rows, cols = 37, 256
    out = torch.empty(rows * cols, dtype=torch.uint8, device="cuda")
    M.moeq_synth_codes(seed, stream, bits, rows * cols, out)
    np.testing.assert_array_equal(out.cpu().numpy().reshape(rows, cols),
                                  S.codes(seed, stream, bits, rows, cols))
    n = 1000
    sc = torch.empty(n * 2, dtype=torch.uint8, device="cuda")
    M.moeq_synth_scales(seed, stream + 1, bits, n, sc)
    ref = S.scales(seed, stream + 1, bits, n)
    got = sc.cpu().numpy()[: n * ref.itemsize].view(ref.dtype)
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("fmt,rows,cols", [(2, 2048, 4096), (3, 4096, 2048), (4, 2048, 4096),
                                           (24, 4096, 2048), (2, 3, 128), (3, 5, 256), (4, 1, 128),
                                           (24, 5, 256)])
def test_pack_bit_exact(fmt, rows, cols):
    bits = S.code_bits(fmt)
    codes = S.codes(5, fmt * 1000 + rows, bits, rows, cols)
    scales = S.scales(5, fmt * 1000 + rows + 1, bits, rows * cols // 32)
    cbytes, sbytes = M.moeq_packed_bytes(fmt, rows, cols)
    d_codes = torch.from_numpy(codes).cuda()
    d_scales = torch.from_numpy(scales.view(np.uint8)).cuda()
    out_c = torch.zeros(cbytes, dtype=torch.uint8, device="cuda")
    out_s = torch.zeros(sbytes, dtype=torch.uint8, device="cuda")
    st = _status()
    M.moe_pack_expert(fmt, rows, cols, d_codes, d_scales, out_c, out_s, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    np.testing.assert_array_equal(out_c.cpu().numpy(), O.pack(fmt, codes))
    np.testing.assert_array_equal(out_s.cpu().numpy(), scales.view(np.uint8))


def test_pack_flags_out_of_range_codes():
    codes = np.zeros((2, 128), dtype=np.uint8)
    codes[1, 100] = 4
    out = torch.zeros(2 * 4 * 8, dtype=torch.uint8, device="cuda")
    st = _status()
    M.moe_pack_expert(2, 2, 128, torch.from_numpy(codes).cuda(), None, out, None, st)
    torch.cuda.synchronize()
    assert st.item() == M.CODE["MOEQ_ERR_DEVICE_INDEX"]


def test_h32_rotate_bit_exact():
    rng = np.random.default_rng(3)
    nblk = 1000
    v = (rng.standard_normal(32 * nblk) * 10.0 ** rng.integers(-6, 4, 32 * nblk)).astype(np.float32)
    signs = S.signs(9, 2, nblk)
    d_in = torch.from_numpy(v).cuda()
    d_out = torch.empty_like(d_in)
    M.h32_rotate(d_in, d_out, nblk, to_dev_u32(signs))
    np.testing.assert_array_equal(d_out.cpu().numpy(), O.h32_f32(v, signs))
    M.h32_rotate(d_in, d_in, nblk, None)   # in place, no signs
    np.testing.assert_array_equal(d_in.cpu().numpy(), O.h32_f32(v, None))


@pytest.mark.parametrize("name,T", [("tiny-decode", 13), ("decode-b1", 37)])
def test_route_topk_bit_exact(name, T):
    cfg = S.WORKLOADS[name]
    seed = S.workload_seed(name)
    wr = S.router_weights(seed, 0, cfg)
    x = S.tokens(seed, cfg, T)
    E, H, k = cfg["E"], cfg["H"], cfg["k"]
    idx = torch.zeros(T * k, dtype=torch.int32, device="cuda")
    w = torch.zeros(T * k, dtype=torch.float32, device="cuda")
    lg = torch.zeros(T * E, dtype=torch.float32, device="cuda")
    M.moe_route_topk(to_dev_u16(x), T, to_dev_u16(wr), E, H, k, idx, w, lg)
    ref = O.router_logits(x, wr)
    np.testing.assert_array_equal(lg.cpu().numpy().reshape(T, E), ref)
    gi = idx.cpu().numpy().reshape(T, k)
    gw = w.cpu().numpy().reshape(T, k)
    for t in range(T):
        ri, rp = O.topk(ref[t], k)
        np.testing.assert_array_equal(gi[t], ri)
        np.testing.assert_allclose(gw[t], rp, rtol=2e-6)


def test_route_topk_ties_and_ragged_tail():
    # integer-valued logits with many exact ties; T not a multiple of the 8-token tile
    H, E, k, T = 256, 40, 5, 11
    rng = np.random.default_rng(4)
    x = S.f32_to_bf16_bits(rng.integers(-2, 3, (T, H)).astype(np.float32))
    wr = S.f32_to_bf16_bits(rng.integers(-1, 2, (E, H)).astype(np.float32))
    idx = torch.zeros(T * k, dtype=torch.int32, device="cuda")
    w = torch.zeros(T * k, dtype=torch.float32, device="cuda")
    M.moe_route_topk(to_dev_u16(x), T, to_dev_u16(wr), E, H, k, idx, w)
    ref = O.router_logits(x, wr)
    for t in range(T):
        np.testing.assert_array_equal(idx.cpu().numpy().reshape(T, k)[t], O.topk(ref[t], k)[0])


def test_route_topk_expert_count_not_multiple_of_4():
    # the kernel takes router rows four at a time; E = 37 leaves a partial group
    H, E, k, T = 512, 37, 3, 9
    rng = np.random.default_rng(6)
    x = S.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    wr = S.f32_to_bf16_bits((rng.standard_normal((E, H)) * 0.05).astype(np.float32))
    idx = torch.zeros(T * k, dtype=torch.int32, device="cuda")
    w = torch.zeros(T * k, dtype=torch.float32, device="cuda")
    lg = torch.full((T * E + 8,), 7.0, dtype=torch.float32, device="cuda")
    M.moe_route_topk(to_dev_u16(x), T, to_dev_u16(wr), E, H, k, idx, w, lg)
    ref = O.router_logits(x, wr)
    out = lg.cpu().numpy()
    np.testing.assert_array_equal(out[:T * E].reshape(T, E), ref)
    assert np.all(out[T * E:] == 7.0)  # nothing written past T x E
    for t in range(T):
        np.testing.assert_array_equal(idx.cpu().numpy().reshape(T, k)[t], O.topk(ref[t], k)[0])


def test_rmsnorm_bit_exact():
    rng = np.random.default_rng(5)
    T, H = 19, 4096
    r = (rng.standard_normal((T, H)) * np.array([1e-3, 1.0, 50.0] * 6 + [3.0])[:, None]).astype(np.float32)
    a = torch.zeros(T * H, dtype=torch.int16, device="cuda")
    M.moe_rmsnorm_bf16(torch.from_numpy(r).cuda(), T, H, a)
    got = a.cpu().numpy().view(np.uint16).reshape(T, H)
    for t in range(T):
        np.testing.assert_array_equal(got[t], O.rmsnorm_bf16(r[t]))
