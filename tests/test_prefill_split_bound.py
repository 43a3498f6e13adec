"""The arithmetic behind the prefill's tensor-core operands and the prefill
tolerances of the parity tests, checked exhaustively on the CPU (no GPU, no
oracle): a weight a = cb * ws (int8 codebook value times an fp16 block scale)
and an activation x = q * d (int8 code times its fp16 scale) are exact in fp32
and split into bf16 parts hi = bf16(v), lo = bf16(v - hi). The claims:
  * |lo| < 2^-8 |v|, and what the two parts leave out is below 2^-17 of |v|
    (exhaustive over the int8 codes and the fp16 scales of a range of binades;
    the relative error repeats from binade to binade);
  * with a power-of-two (E8M0) scale the weight is a bf16 value: lo = 0;
  * a_lo x_lo is below 2^-16 of |a x|, a x - (a_hi x_hi + a_hi x_lo + a_lo x_hi)
    below 8 * 2^-18 of |a x| (the sum of the three bounds), and every part
    product is exact in fp32.
bf16 rounding is torch's (round to nearest even); the references are fp64."""
import numpy as np
import torch

TWO_M18 = 2.0 ** -18
TWO_M17 = 2.0 ** -17
TWO_M16 = 2.0 ** -16


def bf16(v32: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest even) and return them as fp32."""
    return torch.from_numpy(v32).to(torch.bfloat16).to(torch.float32).numpy()


def split(v32: np.ndarray):
    hi = bf16(v32)
    lo = bf16((v32 - hi).astype(np.float32))  # v - hi is exact in fp32 (Sterbenz)
    return hi, lo


def fp16_values(lo: float, hi: float) -> np.ndarray:
    """Every positive finite fp16 value in [lo, hi], as fp32."""
    bits = np.arange(1, 0x7C00, dtype=np.uint16)
    v = bits.view(np.float16).astype(np.float32)
    return v[(v >= lo) & (v <= hi)]


def test_weight_parts_leave_out_below_2_pow_minus_17():
    cb = np.arange(-127, 128, dtype=np.float32)
    ws = fp16_values(6e-5, 0.5)  # the generator draws [1e-4, 1e-2]; wider here
    a = (cb[:, None] * ws[None, :]).astype(np.float32)
    a64 = cb.astype(np.float64)[:, None] * ws.astype(np.float64)[None, :]
    assert np.array_equal(a.astype(np.float64), a64)  # cb * ws is exact in fp32
    hi, lo = split(a)
    left = np.abs(a64 - hi.astype(np.float64) - lo.astype(np.float64))
    assert np.all(left < TWO_M17 * np.abs(a64) + (a64 == 0))
    assert np.all(np.abs(lo) < 2.0 ** -8 * np.abs(a64) + (a64 == 0))


def test_power_of_two_scales_make_the_weight_a_bf16_value():
    cb = np.arange(-127, 128, dtype=np.float32)
    ws = np.float32(2.0) ** np.arange(-30, 10, dtype=np.float32)  # E8M0 exponents, wider than -13..-7
    a = (cb[:, None] * ws[None, :]).astype(np.float32)
    hi, lo = split(a)
    assert np.array_equal(hi, a)
    assert not lo.any()


def test_activation_parts_and_three_part_products():
    rng = np.random.default_rng(11)
    q = np.arange(-127, 128, dtype=np.float32)
    d = fp16_values(1e-6, 60.0)
    x = (q[:, None] * d[None, :]).astype(np.float32)
    x64 = q.astype(np.float64)[:, None] * d.astype(np.float64)[None, :]
    assert np.array_equal(x.astype(np.float64), x64)
    xh, xl = split(x)
    assert np.all(np.abs(x64 - xh - xl.astype(np.float64)) < TWO_M17 * np.abs(x64) + (x64 == 0))
    # products of sampled weights and activations
    n = 400_000
    cb = rng.integers(-127, 128, n).astype(np.float32)
    ws = rng.choice(fp16_values(1e-4, 1e-2), n)
    xs = rng.choice(x.ravel(), n)
    a = (cb * ws).astype(np.float32)
    ah, al = split(a)
    xh, xl = split(xs.astype(np.float32))
    exact = a.astype(np.float64) * xs.astype(np.float64)
    parts = [(ah, xh), (ah, xl), (al, xh)]
    kept = np.zeros(n)
    for u, v in parts:
        p32 = (u * v).astype(np.float32)
        p64 = u.astype(np.float64) * v.astype(np.float64)
        assert np.array_equal(p32.astype(np.float64), p64)  # each part product exact in fp32
        kept += p64
    assert np.all(np.abs(exact - kept) < 8 * TWO_M18 * np.abs(exact) + (exact == 0))
    # the fourth (left-out) product alone is below 2^-16 of |a x|
    assert np.all(np.abs(al.astype(np.float64) * xl) < TWO_M16 * np.abs(exact) + (exact == 0))
