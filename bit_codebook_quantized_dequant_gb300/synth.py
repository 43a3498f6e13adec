"""Seeded synthetic inputs for the codebook-quantized MoE FFN.

This module draws the random numbers that stand in for a real checkpoint and
real activations. It holds none of the FFN's arithmetic: no packing, no
quantization, no dot products. Both the CPU oracle (through the tests) and the
CUDA path (through the tests and the benchmark) take their inputs from here, so
that the two sides see the same seeded data.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) used as a counter-based generator. For a
64-bit seed and a 64-bit stream id,

    key       = mix64(seed * GAMMA + stream)
    u64(i)    = mix64(key + (i + 1) * GAMMA)          (all arithmetic mod 2^64)

which is the i-th output of a SplitMix64 sequence started at state ``key``.
Everything drawn from it below is integer-only except the normal deviates, which
are only ever drawn here on the host.

The library carries a CUDA twin of the code and scale generators (the big
configurations need ~100 GB of weights, which are generated on the device);
that twin follows the same published definition and a GPU test checks it
against this module bit for bit.

Distributions (the pages give the formats, not the data; these follow the
workload descriptions of the hot path):
  * codes: uniform over 2^bits values; element e of a [rows x cols] matrix takes
    bits 4*(e % 16) .. +bits of u64(e // 16);
  * fp16 scales: uniform over the fp16 bit patterns between fp16(1e-4) and
    fp16(1e-2), which is log-uniform across binades (piecewise linear inside one);
  * E8M0 scales: exponent e - 127 uniform in [-13, -7];
  * codebooks: 2^bits distinct int8 values from [-127, 127], sorted ascending
    (partial Fisher-Yates over the 255 candidates);
  * x and router weights: N(0, 1) and N(0, 1/H) by Box-Muller in fp64, rounded to
    fp32 and then to bf16 (round to nearest even at each step);
  * H32 sign masks: the low 32 bits of u64(block).
"""
from __future__ import annotations

import numpy as np

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
M1 = 0xBF58476D1CE4E5B9
M2 = 0x94D049BB133111EB

F16_LO = 0x068E  # fp16(1e-4), round to nearest even
F16_HI = 0x211F  # fp16(1e-2)
E8M0_LO = 127 - 13
E8M0_SPAN = 7

# role ids used in stream ids
ROLE_ROUTER = 1
ROLE_GATE = 2
ROLE_UP = 3
ROLE_DOWN = 4
ROLE_SGATE = 5
ROLE_SUP = 6
ROLE_SDOWN = 7
ROLE_DENSE = 8
ROLE_X = 9
ROLE_SIGNS_X = 10
ROLE_SIGNS_H = 11

KIND_CODES = 0
KIND_SCALES = 1
KIND_CODEBOOK = 2
KIND_VALUES = 3


def workload_seed(name: str) -> int:
    """Base seed of a workload preset (position of its name in WORKLOAD_ORDER)."""
    return 0xC0FFEE00 + WORKLOAD_ORDER.index(name)


def stream_id(layer: int, role: int, expert: int = 0, kind: int = 0) -> int:
    """Stream ids: layer in bits 48..63, role in 40..47, expert in 8..39, kind in 0..7."""
    layer, role, expert, kind = int(layer), int(role), int(expert), int(kind)
    return (((layer & 0xFFFF) << 48) | ((role & 0xFF) << 40) | ((expert & 0xFFFFFFFF) << 8)
            | (kind & 0xFF)) & MASK64


def _mix64_py(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * M1) & MASK64
    z = ((z ^ (z >> 27)) * M2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: int) -> int:
    return _mix64_py((seed * GAMMA + stream) & MASK64)


def _mix64_np(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(M1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(M2)
        return z ^ (z >> np.uint64(31))


def u64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Outputs u64(start) .. u64(start + count - 1) of the (seed, stream) sequence."""
    key = np.uint64(stream_key(seed, stream))
    i = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64_np(key + i * np.uint64(GAMMA))


def codes(seed: int, stream: int, bits: int, rows: int, cols: int) -> np.ndarray:
    """Uniform codes, uint8 [rows, cols]; cols must be a multiple of 16."""
    n = rows * cols
    assert cols % 16 == 0
    u = u64(seed, stream, 0, n // 16)
    sh = (np.arange(16, dtype=np.uint64) * np.uint64(4))
    c = (u[:, None] >> sh[None, :]) & np.uint64((1 << bits) - 1)
    return c.astype(np.uint8).reshape(rows, cols)


def codes_rows(seed: int, stream: int, bits: int, cols: int, r0: int, nrows: int) -> np.ndarray:
    """Rows r0 .. r0+nrows-1 of ``codes(...)`` without drawing the others."""
    assert cols % 16 == 0
    per = cols // 16
    u = u64(seed, stream, r0 * per, nrows * per)
    sh = (np.arange(16, dtype=np.uint64) * np.uint64(4))
    c = (u[:, None] >> sh[None, :]) & np.uint64((1 << bits) - 1)
    return c.astype(np.uint8).reshape(nrows, cols)


def scales_f16(seed: int, stream: int, n: int) -> np.ndarray:
    """fp16 bit patterns (uint16 [n]) spread over [fp16(1e-4), fp16(1e-2)]."""
    u = u64(seed, stream, 0, n)
    span = np.uint64(F16_HI - F16_LO + 1)
    return (np.uint64(F16_LO) + (u >> np.uint64(32)) % span).astype(np.uint16)


def scales_e8m0(seed: int, stream: int, n: int) -> np.ndarray:
    """E8M0 exponent bytes (uint8 [n]) with e - 127 in [-13, -7]."""
    u = u64(seed, stream, 0, n)
    return (np.uint64(E8M0_LO) + (u >> np.uint64(32)) % np.uint64(E8M0_SPAN)).astype(np.uint8)


def scales(seed: int, stream: int, bits: int, n: int) -> np.ndarray:
    return scales_e8m0(seed, stream, n) if bits == 4 else scales_f16(seed, stream, n)


def codebook(seed: int, stream: int, bits: int) -> np.ndarray:
    """2^bits distinct int8 values from [-127, 127], sorted ascending."""
    n = 1 << bits
    cand = list(range(-127, 128))
    u = u64(seed, stream, 0, n)
    for j in range(n):
        k = j + int(int(u[j]) % (len(cand) - j))
        cand[j], cand[k] = cand[k], cand[j]
    return np.array(sorted(cand[:n]), dtype=np.int8)


def _normal(seed: int, stream: int, n: int) -> np.ndarray:
    u = u64(seed, stream, 0, 2 * n)
    ua = u[0::2]
    ub = u[1::2]
    u1 = ((ua >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (ub >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    x = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (x >> np.uint64(16)) & np.uint64(1)
    return ((x + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(seed: int, stream: int, n: int, std: float = 1.0) -> np.ndarray:
    z = _normal(seed, stream, n) * std
    return f32_to_bf16_bits(z.astype(np.float32))


def signs(seed: int, stream: int, n: int) -> np.ndarray:
    return (u64(seed, stream, 0, n) & np.uint64(0xFFFFFFFF)).astype(np.uint32)


# ---------------------------------------------------------------------------
# Workload presets. Shapes and formats of the five seeded workloads; values are
# drawn with the generators above, stream ids from ``stream_id``.
# ---------------------------------------------------------------------------
WORKLOADS = {
    "tiny-decode": dict(name="tiny-decode", H=256, I=128, E=16, k=2, fmt_gu=2, fmt_down=3, shared_fmt=None,
            h32=False, T=1, layers=1, dense=False),
    "decode-b1": dict(name="decode-b1", H=4096, I=2048, E=256, k=6, fmt_gu=2, fmt_down=3, shared_fmt=4,
            h32=False, T=1, layers=1, dense=False),
    "verify-q4": dict(name="verify-q4", H=4096, I=2048, E=256, k=6, fmt_gu=2, fmt_down=3, shared_fmt=4,
            h32=False, T=4, layers=1, dense=True),
    # format variants of the decode layer: top-4 routing, and FP2 down projections
    "decode-b1-top4": dict(name="decode-b1-top4", H=4096, I=2048, E=256, k=4, fmt_gu=2, fmt_down=3,
            shared_fmt=4, h32=False, T=1, layers=1, dense=False),
    "decode-b1-fp2down": dict(name="decode-b1-fp2down", H=4096, I=2048, E=256, k=6, fmt_gu=2, fmt_down=2,
            shared_fmt=4, h32=False, T=1, layers=1, dense=False),
    "decode-b1-p24down": dict(name="decode-b1-p24down", H=4096, I=2048, E=256, k=6, fmt_gu=2, fmt_down=24,
            shared_fmt=4, h32=False, T=1, layers=1, dense=False),
    "prefill-h32-fp4": dict(name="prefill-h32-fp4", H=4096, I=2048, E=256, k=6, fmt_gu=4, fmt_down=4,
            shared_fmt=None, h32=True, T=2048, layers=1, dense=False),
    "prefill-43-layer-stack": dict(name="prefill-43-layer-stack", H=4096, I=2048, E=256, k=6, fmt_gu=2, fmt_down=3,
            shared_fmt=4, h32=False, T=32512, layers=43, dense=False),
}
WORKLOAD_ORDER = ("tiny-decode", "decode-b1", "verify-q4", "prefill-h32-fp4", "prefill-43-layer-stack",
                  "decode-b1-top4", "decode-b1-fp2down", "decode-b1-p24down")

# (role, rows-is-I?) for the matrices of a layer: gate/up are [I x H], down [H x I]
MATRIX_ROLES = {
    "gate": ROLE_GATE, "up": ROLE_UP, "down": ROLE_DOWN,
    "sgate": ROLE_SGATE, "sup": ROLE_SUP, "sdown": ROLE_SDOWN, "dense": ROLE_DENSE,
}


# Format code of 3-bit codes in the Packed24 layout (the bit order differs
# from FP3's; the drawn codes, scales and codebooks do not).
FP3_PACKED24 = 24


def code_bits(fmt: int) -> int:
    """Bits per code of a format code."""
    return 3 if fmt == FP3_PACKED24 else fmt


def matrix_shape(cfg: dict, name: str):
    """(fmt, rows, cols) of a role in a preset."""
    H, I = cfg["H"], cfg["I"]
    if name in ("gate", "up"):
        return cfg["fmt_gu"], I, H
    if name == "down":
        return cfg["fmt_down"], H, I
    if name in ("sgate", "sup"):
        return cfg["shared_fmt"], I, H
    if name == "sdown":
        return cfg["shared_fmt"], H, I
    if name == "dense":
        return 4, H, H
    raise KeyError(name)


def layer_roles(cfg: dict):
    roles = ["gate", "up", "down"]
    if cfg["shared_fmt"]:
        roles += ["sgate", "sup", "sdown"]
    if cfg["dense"]:
        roles += ["dense"]
    return roles


def expert_codes(seed, layer, name, expert, cfg):
    fmt, rows, cols = matrix_shape(cfg, name)
    return codes(seed, stream_id(layer, MATRIX_ROLES[name], expert, KIND_CODES), code_bits(fmt), rows, cols)


def expert_scales(seed, layer, name, expert, cfg):
    fmt, rows, cols = matrix_shape(cfg, name)
    return scales(seed, stream_id(layer, MATRIX_ROLES[name], expert, KIND_SCALES), code_bits(fmt),
                  rows * (cols // 32))


def expert_codebook(seed, layer, name, expert, cfg):
    fmt, _, _ = matrix_shape(cfg, name)
    return codebook(seed, stream_id(layer, MATRIX_ROLES[name], expert, KIND_CODEBOOK), code_bits(fmt))


def router_weights(seed, layer, cfg):
    H, E = cfg["H"], cfg["E"]
    return normal_bf16(seed, stream_id(layer, ROLE_ROUTER, 0, KIND_VALUES), E * H,
                       std=1.0 / np.sqrt(H)).reshape(E, H)


def tokens(seed, cfg, count, start=0, layer=0):
    """x for tokens start .. start+count-1 (bf16 bits [count, H]); token t of the
    workload is the same row whatever batch it is drawn in."""
    H = cfg["H"]
    u = u64(seed, stream_id(layer, ROLE_X, 0, KIND_VALUES), 2 * start * H, 2 * count * H)
    ua, ub = u[0::2], u[1::2]
    u1 = ((ua >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (ub >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return f32_to_bf16_bits(z.astype(np.float32)).reshape(count, H)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def selection_gap(seed, cfg, token=0, layer=0) -> float:
    """Workload screening: the absolute gap between the k-th and (k+1)-th
    largest router logits of one token, from the bf16 inputs in fp64 (a plain
    dot product; the decision itself is taken in the kernels' fp32 order)."""
    x = bf16_bits_to_f64(tokens(seed, cfg, 1, start=token, layer=layer)[0])
    w = bf16_bits_to_f64(router_weights(seed, layer, cfg))
    lg = np.sort(w @ x)[::-1]
    k = cfg["k"]
    return float(lg[k - 1] - lg[k])


CONFIG0_MIN_GAP = 1e-3


def config0_seeds(count: int, cfg=None, min_gap: float = CONFIG0_MIN_GAP):
    """Seeds of the tiny decode workload (one token each, token 0 of layer 0):
    consecutive seeds from the workload's base seed, skipping those whose
    rank-k / rank-(k+1) router logit gap is below min_gap."""
    cfg = cfg or WORKLOADS["tiny-decode"]
    out, s = [], workload_seed("tiny-decode")
    while len(out) < count:
        if selection_gap(s, cfg) >= min_gap:
            out.append(s)
        s += 1
    return out


def h32_signs(seed, layer, cfg, which):
    n = (cfg["H"] if which == "x" else cfg["I"]) // 32
    role = ROLE_SIGNS_X if which == "x" else ROLE_SIGNS_H
    return signs(seed, stream_id(layer, role, 0, KIND_VALUES), n)
