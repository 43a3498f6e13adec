"""Benchmark of the codebook-quantized MoE FFN hot path on GB300.

Default workload: batch-1 decode of one MoE FFN layer (hidden 4096, expert
intermediate 2048, 256 routed experts, top-6 + an always-on shared expert;
routed gate/up FP2, routed down FP3, shared expert FP4, bf16 router). One step
decodes one token through moe_ffn_decode (one persistent kernel). Steps cycle
through independently seeded layer replicas (default 8 x 2.3 GB) so that no
step finds its weights in the 129 MB L2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0). Under torchrun every rank decodes its own token
stream on its own GPU (independent problems, no data-path collective): weak
scaling; value = all ranks' tokens / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

WORKLOAD = ("decode-b1: H=4096 I=2048 E=256 top-6 + shared expert; routed gate/up FP2 (10 B/32), "
            "routed down FP3 (14 B/32), shared FP4 (17 B/32), bf16 router")
DECODE_WORKLOAD = "decode-b1"
# the headline line's value is decode b=1 (one layer); the q=4 verification and
# the 32K prefill are reported beside it ("verify_q4", "prefill"), each with its
# roofline fraction
DECODE_METRIC = "MoE-FFN tok/s (decode b=1, q=4 verify, 32K prefill) + % of HBM/TC roofline"


def algorithmic_bytes_decode(cfg: dict) -> int:
    """Packed weight bytes one token reads: router + k routed experts + shared expert."""
    from bit_codebook_quantized_dequant_gb300 import synth as S
    H, I, E, k = cfg["H"], cfg["I"], cfg["E"], cfg["k"]
    per_blk = {2: 10, 3: 14, 4: 17}
    routed = 2 * I * (H // 32) * per_blk[cfg["fmt_gu"]] + H * (I // 32) * per_blk[cfg["fmt_down"]]
    shared = 0
    if cfg["shared_fmt"]:
        shared = 3 * I * (H // 32) * per_blk[cfg["shared_fmt"]]
    return E * H * 2 + k * routed + shared


def algorithmic_bytes_verify(cfg: dict, distinct_experts: float) -> float:
    """Packed weight bytes one q=4 call reads: router, each distinct routed
    expert once, the shared expert and the dense projection once."""
    H, I, E = cfg["H"], cfg["I"], cfg["E"]
    per_blk = {2: 10, 3: 14, 4: 17}
    routed = 2 * I * (H // 32) * per_blk[cfg["fmt_gu"]] + H * (I // 32) * per_blk[cfg["fmt_down"]]
    shared = 3 * I * (H // 32) * per_blk[cfg["shared_fmt"]] if cfg["shared_fmt"] else 0
    dense = H * (H // 32) * per_blk[4] if cfg["dense"] else 0
    return E * H * 2 + distinct_experts * routed + shared + dense


def prefill_flops(cfg: dict, T: int) -> float:
    """Expert FLOPs of a prefill of T tokens: 3 matrices of H x I per routed
    slot and for the shared expert, 2 FLOPs per multiply-add."""
    ns = cfg["k"] + (1 if cfg["shared_fmt"] else 0)
    return 2.0 * T * ns * 3 * cfg["H"] * cfg["I"]


def prefill_launches(cfg: dict) -> int:
    """Kernels one moe_ffn_prefill call launches: route, prep_x, count, place,
    gather, gate/up/down per routed and shared group, combine."""
    return 5 + 3 * (2 if cfg["shared_fmt"] else 1) + 1


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


DEVICE_HEADER = "bit_codebook_quantized_dequant_gb300/csrc/moeq_device.cuh"


def source_sha(source: str) -> str:
    """Hash of a kernel's source file and the device header it includes."""
    h = hashlib.sha256()
    for f in (source, DEVICE_HEADER):
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# Target fractions of each path's roofline (the decode and q=4 lines: 70 % of
# HBM; the tensor-core-bound prefill: 50 % of the bf16 peak).
TARGET_HBM, TARGET_TC = 0.70, 0.50


def _target(roof: dict, target):
    """The target fraction and the gap to it, beside the achieved fraction."""
    roof["target_frac"] = target
    roof["gap_to_target"] = None if target is None else target - roof["frac"]
    return roof


def _traffic(kernel: str, source: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current source of the kernel (its file and the device header); else
    None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(kernel)
    if not ent:
        return None
    return ent["bytes_per_launch"] if ent.get("source_sha") == source_sha(source) else None


class ClockSampler:
    """nvidia-smi samples of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"moeq_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes),
                "reasons": sorted(reasons), "samples": len(sms)}


def rank_token_start(rank: int, ntok: int) -> int:
    """First token of a rank's own stream: ranks decode disjoint token ranges
    (independent problems, no data-path collective)."""
    return rank * ntok


def max_over_ranks(times_ms, dist=None, device=None):
    """Each rank's timed durations -> the maximum over ranks (the job's time)."""
    import torch
    t = torch.tensor([float(x) for x in times_ms], dtype=torch.float64, device=device)
    if dist is not None and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def job_throughput(world: int, units_per_rank: int, ms: float) -> float:
    """Whole-job units per second: all ranks' units over the max-over-ranks time."""
    return world * units_per_rank / (ms * 1e-3)


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def cpu_baseline(name: str, tokens: int, seconds_cap: float = 30.0):
    """The oracle, as it stands, timed on this host (one core) on a bounded
    sample of the workload's tokens. Returns (tokens/s, sample description)."""
    import oracle as O
    from oracle import workload as W
    from bit_codebook_quantized_dequant_gb300 import synth as S
    cfg = S.WORKLOADS[name]
    seed = S.workload_seed(name)
    xs = S.tokens(seed, cfg, tokens)
    experts = set()
    wr = S.router_weights(seed, 0, cfg)
    lg = O.router_logits(xs, wr)
    for t in range(tokens):
        experts.update(int(e) for e in O.topk(lg[t], cfg["k"])[0])
    L = W.layer(seed, 0, cfg, experts)
    done = 0
    t0 = time.perf_counter()
    for t in range(tokens):
        O.ffn_decode(L, xs[t])
        done += 1
        if time.perf_counter() - t0 > seconds_cap:
            break
    dt = time.perf_counter() - t0
    return done / dt, f"{done} tokens of the decode workload (layer 0), oracle single-threaded", dt


def cpu_baseline_prefill(name: str, tokens: int = 8) -> dict:
    """The oracle's prefill, as it stands, timed on this host (one core) on the
    first `tokens` tokens of a prefill workload (one layer). Each token's FFN
    is independent of the others, so the rate holds for all T tokens."""
    import oracle as O
    from oracle import workload as W
    from bit_codebook_quantized_dequant_gb300 import synth as S
    cfg = S.WORKLOADS[name]
    seed = S.workload_seed(name)
    xs = S.tokens(seed, cfg, tokens)
    idx, _ = W.route(seed, 0, cfg, xs)
    L = W.layer(seed, 0, cfg, {int(e) for r in idx for e in r})
    t0 = time.perf_counter()
    O.ffn_prefill(L, xs)
    dt = time.perf_counter() - t0
    return {"value": tokens / dt, "unit": "tok/s", "cores": 1, "kind": "oracle",
            "sample": f"the first {tokens} tokens of the {name} workload (layer 0) through the "
                      "oracle's prefill, single-threaded; each token's FFN is independent of "
                      "the others, so the rate holds for all T tokens"}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    tps, sample, dt = cpu_baseline(DECODE_WORKLOAD, max(1, min(args.steps, 4)))
    line = {"impl": "reference", "metric": DECODE_METRIC, "value": tps,
            "unit": "tok/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 / tps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD},
            "cpu_baseline": {"value": tps, "unit": "tok/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": tps, "unit": "tok/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def capture_steps(step, first, n, stream, chunk=64):
    """CUDA graphs of steps first .. first + n - 1 (chunks of `chunk` steps),
    each step enqueued by step(i, stream)."""
    import torch
    graphs, i = [], first
    while i < first + n:
        m = min(chunk, first + n - i)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(m):
                step(i + j, stream)
        graphs.append(g)
        i += m
    return graphs


def replay(graphs, stream):
    """Replays the graphs on `stream` (a graph launches on the current stream)."""
    import torch
    with torch.cuda.stream(stream):
        for g in graphs:
            g.replay()


def _abs_weights(m, e):
    """|w| of expert e of an oracle matrix, fp32 (a tolerance, not a result; cpu leg)."""
    import oracle as O
    codes = O.unpack(m.fmt, m.rows, m.cols, m.codes[e])
    sv = O.scale_values(m.fmt, m.scales[e]).astype(np.float32).reshape(m.rows, m.cols // 32)
    return np.abs(np.repeat(sv, 32, axis=1) * m.cb[e].astype(np.float32)[codes])


def oracle_parity(L, x_rows, ys, hqs, hds):
    """The oracle (cpu leg) on sampled tokens against the GPU's outputs ys and
    quantized h (hqs, hds: [tokens, slots, I] / [tokens, slots, I/32]):
    |y - y_oracle| <= 2e-3 B + D with B = sum_slot p sum_k |w_down| |h~| (the
    GPU's h~) and D = sum_slot p sum_k |w_down| |h~ - h~_oracle|, and the
    relative L2 error. Returns (ok, worst err / bound, worst relative L2)."""
    import oracle as O
    worst, rel_worst, ok = 0.0, 0.0, True
    for t in range(len(x_rows)):
        yo, tr = O.ffn_decode(L, x_rows[t], trace=True)
        slots = [(L.down, int(e)) for e in tr["idx"]]
        if L.shared is not None:
            slots.append((L.shared[2], 0))
        w = list(tr["p"]) + ([1.0] if L.shared is not None else [])
        B = np.zeros(L.H)
        D = np.zeros(L.H)
        for s, (m, e) in enumerate(slots):
            hg = hqs[t][s].astype(np.float64) * np.repeat(O.f16_array_to_f64(hds[t][s]), 32)
            ho = tr["hq"][s].astype(np.float64) * np.repeat(O.f16_array_to_f64(tr["hd"][s]), 32)
            A = _abs_weights(m, e)
            B += w[s] * (A @ np.abs(hg).astype(np.float32)).astype(np.float64)
            D += w[s] * (A @ np.abs(hg - ho).astype(np.float32)).astype(np.float64) * (1 + 1e-5)
        y = np.asarray(ys[t], dtype=np.float64)
        err = np.abs(y - yo)
        lim = 2e-3 * B + D
        worst = max(worst, float(np.max(err / np.maximum(lim, 1e-300))))
        rel = float(np.linalg.norm(y - yo) / max(np.linalg.norm(yo), 1e-300))
        rel_lim = 1e-4 + float(np.linalg.norm(D) / max(np.linalg.norm(yo), 1e-300))
        rel_worst = max(rel_worst, rel / rel_lim)
        ok = ok and bool(np.all(err <= lim)) and rel <= rel_lim
    return ok, worst, rel_worst


def gpu_decode_rows(dl, ws, x_rows, cfg):
    """Sampled tokens through the decode with its debug outputs: y, hq, hd per token."""
    import torch
    import bit_codebook_quantized_dequant_gb300 as M
    from bit_codebook_quantized_dequant_gb300.workload import Debug, to_dev_u16
    H, I = cfg["H"], cfg["I"]
    ns = cfg["k"] + (1 if cfg["shared_fmt"] else 0)
    ys, hqs, hds = [], [], []
    for t in range(len(x_rows)):
        d = Debug(cfg, 1)
        y = torch.zeros(H, dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        M.moe_ffn_decode(dl.desc(), to_dev_u16(x_rows[t]), y, ws.ptr, ws.nbytes, st, d.struct)
        torch.cuda.synchronize()
        assert st.item() == 0, f"device status {st.item()}"
        g = d.numpy()
        ys.append(y.cpu().numpy())
        hqs.append(g["hq"].reshape(ns, I))
        hds.append(g["hd"].reshape(ns, I // 32))
    return ys, hqs, hds


def decode_parity_after(dl, ws, xs_host, cfg, seed, ntok=4):
    """After the timed steps: the first sampled tokens of the cpu leg (layer 0)
    through the decode once more, against the oracle's outputs."""
    from oracle import workload as W
    x = xs_host[:ntok]
    ys, hqs, hds = gpu_decode_rows(dl, ws, x, cfg)
    idx, _ = W.route(seed, 0, cfg, x)
    L = W.layer(seed, 0, cfg, {int(e) for r in idx for e in r})
    ok, worst, rel = oracle_parity(L, x, ys, hqs, hds)
    return {"tokens": ntok, "layer": 0, "ok": ok, "max_err_over_limit": worst,
            "max_rel_l2_over_limit": rel,
            "check": "y of sampled tokens against the fp64 oracle: |err| <= 2e-3 B + D, relative L2 "
                     "<= 1e-4 + |D|/|y| (B: sum_slot p |w_down| |h~|; D: the same on the difference "
                     "of the GPU's and the oracle's quantized h)"}


def _timed(fn, warmup, steps, stream):
    import torch
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        fn(warmup + i)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def verify_parity_after(dl, ws, X, cfg, seed):
    """After the timed calls: one batch of 4 columns through the q=4 call once
    more, each column and the dense projection against the oracle."""
    import torch
    import oracle as O
    from oracle import workload as W
    import bit_codebook_quantized_dequant_gb300 as M
    from bit_codebook_quantized_dequant_gb300.workload import Debug, to_dev_u16
    H, I = cfg["H"], cfg["I"]
    ns = cfg["k"] + (1 if cfg["shared_fmt"] else 0)
    d = Debug(cfg, 4)
    y = torch.zeros(4 * H, dtype=torch.float32, device="cuda")
    yd = torch.zeros(4 * H, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_ffn_verify_q4(dl.desc(), dl.dense.desc(), to_dev_u16(X), y, yd, ws.ptr, ws.nbytes, st, d.struct)
    torch.cuda.synchronize()
    assert st.item() == 0, f"device status {st.item()}"
    g = d.numpy()
    ys = y.cpu().numpy().reshape(4, H)
    hq = g["hq"].reshape(4, ns, I)
    hd = g["hd"].reshape(4, ns, I // 32)
    idx, _ = W.route(seed, 0, cfg, X)
    L = W.layer(seed, 0, cfg, {int(e) for r in idx for e in r})
    ok, worst, rel = oracle_parity(L, X, list(ys), list(hq), list(hd))
    # dense projection: |err| <= 2e-3 sum |w_dense| |x~| per row
    Dm = W.dense(seed, 0, cfg)
    _, yd_ref = O.ffn_verify_q4(L, Dm, X)
    A = _abs_weights(Dm, 0)
    yd = yd.cpu().numpy().reshape(4, H)[:, :Dm.rows]
    xq, xd = g["xq"].reshape(4, H), g["xd"].reshape(4, H // 32)
    for c in range(4):
        xt = np.abs(xq[c].astype(np.float32) * np.repeat(O.f16_array_to_f64(xd[c]).astype(np.float32), 32))
        bound = 2e-3 * (A @ xt).astype(np.float64)
        err = np.abs(yd[c] - yd_ref[c])
        worst = max(worst, float(np.max(err / np.maximum(bound, 1e-300))))
        ok = ok and bool(np.all(err <= bound))
    return {"batches": 1, "columns": 4, "layer": 0, "ok": ok, "max_err_over_limit": worst,
            "max_rel_l2_over_limit": rel,
            "check": "each column's y against the fp64 oracle as in the decode section; y_dense "
                     "within 2e-3 sum |w| |x~| per row"}


def bench_verify(args, hbm_peak, peak_kind, cpu=False):
    """q=4 verification: 4 columns per call through moe_ffn_verify_q4, cycling
    over --replicas seeded layer replicas (each with its dense projection)."""
    import torch
    import bit_codebook_quantized_dequant_gb300 as M
    from bit_codebook_quantized_dequant_gb300 import synth as S
    from bit_codebook_quantized_dequant_gb300.workload import Workspace, build_layer, to_dev_u16
    name = "verify-q4"
    cfg = S.WORKLOADS[name]
    seed = S.workload_seed(name)
    R = max(1, args.replicas)
    layers = [build_layer(seed, r, cfg) for r in range(R)]
    wss = [Workspace(dl, 1) for dl in layers]
    descs = [dl.desc() for dl in layers]
    dds = [dl.dense.desc() for dl in layers]
    nb = 64
    X = S.tokens(seed, cfg, 4 * nb)
    xs = to_dev_u16(X)
    H = cfg["H"]
    y = torch.zeros(4 * H, dtype=torch.float32, device="cuda")
    yd = torch.zeros(4 * H, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()

    def step(i, s):
        r = i % R
        M.moe_ffn_verify_q4(descs[r], dds[r], xs.data_ptr() + (i % nb) * 4 * H * 2, y, yd,
                            wss[r].ptr, wss[r].nbytes, st, None, s)

    steps = max(args.steps // 4, 50)
    for i in range(args.warmup):
        step(i, stream)
    torch.cuda.synchronize()
    graphs = capture_steps(step, args.warmup, steps, stream)
    replay(graphs, stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    replay(graphs, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    del graphs
    assert st.item() == 0, f"device status {st.item()}"
    parity = None
    if cpu:
        parity = verify_parity_after(layers[0], wss[0], X[:4], cfg, seed)
    # distinct experts per timed call: the (replica, batch) pairs the timed
    # steps used, each weighted by its count (routing outside the timed region)
    uses = {}
    for i in range(args.warmup, args.warmup + steps):
        key = (i % R, i % nb)
        uses[key] = uses.get(key, 0) + 1
    idx = torch.zeros(4 * cfg["k"], dtype=torch.int32, device="cuda")
    w = torch.zeros(4 * cfg["k"], dtype=torch.float32, device="cuda")
    tot = 0
    for (r, b), n in uses.items():
        M.moe_route_topk(xs.data_ptr() + b * 4 * H * 2, 4, layers[r].router, cfg["E"], H,
                         cfg["k"], idx, w)
        tot += n * len(set(idx.cpu().tolist()))
    nd = tot / steps
    per_call = algorithmic_bytes_verify(cfg, nd)
    achieved = per_call / (ms * 1e-3) / 1e9
    out = {"metric": "q=4 verification column-tokens/s", "value": 4.0 / (ms * 1e-3),
           "unit": "column-tok/s", "ms_per_call": ms, "calls": steps,
           "workload": "verify-q4: decode-b1 layer + dense 4096x4096 FP4; 4 independently routed "
                       f"columns per call; {R} replicas cycled",
           "distinct_experts_per_call": nd,
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                        "frac": achieved / hbm_peak,
                        "traffic": _traffic("ffn_kernel<4>",
                                            "bit_codebook_quantized_dequant_gb300/csrc/decode.cu"),
                        "peak_source": f"{peak_kind} hbm_gbs",
                        "algorithmic_bytes_per_launch": per_call},
           "gpu_launches": steps, "launch": "CUDA graph replay",
           "parity_after": parity}
    _target(out["roofline"], TARGET_HBM)
    del layers, wss
    torch.cuda.empty_cache()
    return out


def prefill_parity_after(dl, ws, X_host, X_dev, y, cfg, seed, T):
    """After the timed calls: the prefill once more with its quantized h
    recorded, then sampled tokens' y against the oracle (as in the decode
    section; the prefill's h comes from tensor-core part products)."""
    import torch
    import bit_codebook_quantized_dequant_gb300 as M
    from oracle import workload as W
    H, I = cfg["H"], cfg["I"]
    ns = cfg["k"] + (1 if cfg["shared_fmt"] else 0)
    hq = torch.zeros(T * ns * I, dtype=torch.int8, device="cuda")
    hd = torch.zeros(T * ns * (I // 32), dtype=torch.int16, device="cuda")
    dbg = M.MoeqDebug(hq=hq.data_ptr(), hd=hd.data_ptr())
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_ffn_prefill(dl.desc(), X_dev, T, None, y, ws.ptr, ws.nbytes, st, dbg)
    torch.cuda.synchronize()
    assert st.item() == 0, f"device status {st.item()}"
    sample = [0, T // 2 + 1, T - 1]
    idx_t = torch.as_tensor(sample, dtype=torch.long, device="cuda")
    ys = y.view(T, H).index_select(0, idx_t).cpu().numpy()
    hqs = hq.view(T, ns, I).index_select(0, idx_t).cpu().numpy()
    hds = hd.view(T, ns, I // 32).index_select(0, idx_t).cpu().numpy().view(np.uint16)
    x = X_host[sample]
    idx, _ = W.route(seed, 0, cfg, x)
    L = W.layer(seed, 0, cfg, {int(e) for r in idx for e in r})
    ok, worst, rel = oracle_parity(L, x, list(ys), list(hqs), list(hds))
    del hq, hd
    return {"tokens": sample, "layer": 0, "ok": ok, "max_err_over_limit": worst,
            "max_rel_l2_over_limit": rel,
            "check": "y of sampled tokens against the fp64 oracle as in the decode section"}


def bench_prefill(args, name, T, tc_peak, hbm_peak, peak_kind, cpu=False):
    """Expert-grouped prefill of T tokens through one layer (moe_ffn_prefill)."""
    import torch
    import bit_codebook_quantized_dequant_gb300 as M
    from bit_codebook_quantized_dequant_gb300 import synth as S
    from bit_codebook_quantized_dequant_gb300.workload import Workspace, build_layer, to_dev_u16
    cfg = S.WORKLOADS[name]
    seed = S.workload_seed(name)
    dl = build_layer(seed, 0, cfg)
    ws = Workspace(dl, 2, T)
    X_host = S.tokens(seed, cfg, T)
    X = to_dev_u16(X_host)
    y = torch.zeros(T * cfg["H"], dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    desc = dl.desc()

    def step(i):
        M.moe_ffn_prefill(desc, X, T, None, y, ws.ptr, ws.nbytes, st, None, stream)

    steps = 3
    ms = _timed(step, 3, steps, stream)
    assert st.item() == 0, f"device status {st.item()}"
    fl = prefill_flops(cfg, T)
    tflops = fl / (ms * 1e-3) / 1e12
    wbytes = dl.weight_bytes()
    hbm_gbs = wbytes / (ms * 1e-3) / 1e9
    tensor = {"bound": "tensor", "achieved": tflops, "peak": tc_peak, "unit": "TFLOP/s",
              "frac": tflops / tc_peak,
              "traffic": _traffic(f"prefill {name} gemm",
                                  "bit_codebook_quantized_dequant_gb300/csrc/gemm_tc.cu"),
              "traffic_scope": "DRAM bytes of the gate, up and down tensor-core "
                               "launches of one call (routed experts)",
              "peak_source": f"{peak_kind} bf16_tflops (the prefill contraction runs "
                             "as bf16 part products on the tensor cores)",
              "algorithmic_flops_per_launch": fl}
    hbm = {"bound": "hbm", "achieved": hbm_gbs, "peak": hbm_peak, "unit": "GB/s",
           "frac": hbm_gbs / hbm_peak,
           "traffic": _traffic(f"prefill {name} gemm", "bit_codebook_quantized_dequant_gb300/csrc/gemm_tc.cu"),
           "traffic_scope": "DRAM bytes of the gate, up and down tensor-core launches of one call",
           "peak_source": f"{peak_kind} hbm_gbs",
           "algorithmic_bytes_per_launch": wbytes}
    # the layer's bound: its FLOP per weight byte against the bf16 ridge
    ridge = tc_peak * 1e12 / (hbm_peak * 1e9)
    hbm_bound = fl / wbytes < ridge
    _target(tensor, TARGET_TC)
    _target(hbm, None)  # no HBM target is stated for the prefill
    out = {"metric": "prefill tok/s (one layer)", "value": T / (ms * 1e-3), "unit": "tok/s",
           "ms_per_call": ms, "calls": steps, "tokens": T,
           "workload": name + f": T={T}, one layer, all 256 experts' weights read once",
           "flop_per_weight_byte": fl / wbytes, "ridge_flop_per_byte": ridge,
           "roofline": hbm if hbm_bound else tensor,
           "roofline_other": tensor if hbm_bound else hbm,
           "gpu_launches_per_call": prefill_launches(cfg)}
    if cpu:
        try:
            out["parity_after"] = prefill_parity_after(dl, ws, X_host, X, y, cfg, seed, T)
        except Exception as e:  # reported, not hidden
            out["parity_after"] = {"ok": False, "error": repr(e)}
    del dl, ws
    torch.cuda.empty_cache()
    if cpu:
        try:
            out["cpu_baseline"] = cpu_baseline_prefill(name)
        except Exception as e:  # the GPU numbers stand without it
            out["cpu_baseline"] = {"error": repr(e)}
    return out


def bench_stack(args, T, nlayers, tc_peak, peak_kind):
    """The 43-layer stack of the prefill workload: T tokens through nlayers
    independently seeded layers (moe_ffn_stack_prefill: RMSNorm, FFN and
    residual per layer), all layers resident in HBM."""
    import torch
    import bit_codebook_quantized_dequant_gb300 as M
    from bit_codebook_quantized_dequant_gb300 import synth as S
    from bit_codebook_quantized_dequant_gb300.workload import Workspace, build_layer, to_dev_u16
    name = "prefill-43-layer-stack"
    cfg = S.WORKLOADS[name]
    seed = S.workload_seed(name)
    layers = [build_layer(seed, l, cfg) for l in range(nlayers)]
    descs = [dl.desc() for dl in layers]
    ws = Workspace(layers[0], 3, T)
    X = to_dev_u16(S.tokens(seed, cfg, T))
    r = torch.zeros(T * cfg["H"], dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def step(i):
        M.moe_ffn_stack_prefill(descs, X, T, r, ws.ptr, ws.nbytes, st, stream)

    ms = _timed(step, 1, 1, stream)
    assert st.item() == 0, f"device status {st.item()}"
    r1 = r.clone()
    step(0)
    torch.cuda.synchronize()
    same = bool(torch.equal(r, r1))
    fl = nlayers * prefill_flops(cfg, T)
    tflops = fl / (ms * 1e-3) / 1e12
    wbytes = sum(dl.weight_bytes() for dl in layers)
    out = {"metric": f"prefill tok/s ({nlayers}-layer stack)", "value": T / (ms * 1e-3),
           "unit": "tok/s", "ms_per_call": ms, "calls": 1, "tokens": T, "layers": nlayers,
           "workload": f"{name}: T={T}, {nlayers} independently seeded layers "
                       f"({wbytes / 1e9:.1f} GB resident), RMSNorm + FFN + residual per layer",
           "roofline": {"bound": "tensor", "achieved": tflops, "peak": tc_peak, "unit": "TFLOP/s",
                        "frac": tflops / tc_peak, "traffic": None,
                        "peak_source": f"{peak_kind} bf16_tflops",
                        "algorithmic_flops_per_launch": fl},
           "parity_after": {"repeat_bit_equal": same,
                            "check": "the stack's output after the timed call equals a second "
                                     "call's bit for bit; the stack's oracle parity (chain, "
                                     "teacher-forced per layer) is a GPU test"}}
    del ws, r, r1
    torch.cuda.empty_cache()
    _target(out["roofline"], TARGET_TC)
    dec = bench_stack_decode(args, layers, cfg, seed)
    _target(dec["roofline"], TARGET_HBM)
    torch.cuda.empty_cache()
    dec["verify_q4_stack"] = bench_stack_verify(args, layers, cfg, seed)
    _target(dec["verify_q4_stack"]["roofline"], TARGET_HBM)
    del layers
    torch.cuda.empty_cache()
    return out, dec


def bench_stack_decode(args, layers, cfg, seed):
    """One decode token at a time through the whole stack (moe_ffn_stack_decode:
    RMSNorm, decode and residual per layer), steps replayed from CUDA graphs."""
    import torch
    import bit_codebook_quantized_dequant_gb300 as M
    from bit_codebook_quantized_dequant_gb300 import synth as S
    from bit_codebook_quantized_dequant_gb300.workload import Workspace, to_dev_u16
    nl = len(layers)
    descs = [dl.desc() for dl in layers]
    ws = Workspace(layers[0], 4)
    H = cfg["H"]
    ntok = 16
    xs = to_dev_u16(S.tokens(seed, cfg, ntok, start=4096))
    r = torch.zeros(H, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()

    def step(i, s):
        M.moe_ffn_stack_decode(descs, xs.data_ptr() + (i % ntok) * H * 2, r, ws.ptr, ws.nbytes, st, s)

    warm, steps = 3, 8
    for i in range(warm):
        step(i, stream)
    torch.cuda.synchronize()
    graphs = capture_steps(step, warm, steps, stream, chunk=8)
    replay(graphs, stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    replay(graphs, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    assert st.item() == 0, f"device status {st.item()}"
    r_graph = r.clone()
    step(warm + steps - 1, stream)  # the last timed token again, launched on the stream
    torch.cuda.synchronize()
    same = bool(torch.equal(r, r_graph))
    del graphs
    hbm_peak, _, peak_kind = _peaks()
    per_tok = nl * algorithmic_bytes_decode(cfg)
    achieved = per_tok / (ms * 1e-3) / 1e9
    return {"metric": f"decode tok/s ({nl}-layer stack, b=1)", "value": 1.0 / (ms * 1e-3),
            "unit": "tok/s", "ms_per_token": ms, "tokens_timed": steps, "layers": nl,
            "workload": f"prefill-43-layer-stack layers (decode-b1 shapes), one token through all "
                        f"{nl} layers per step: RMSNorm + decode + fp32 residual per layer",
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": None,
                         "peak_source": f"{peak_kind} hbm_gbs",
                         "algorithmic_bytes_per_launch": per_tok},
            "gpu_launches_per_token": 2 * nl + 1, "launch": "CUDA graph replay",
            "parity_after": {"repeat_bit_equal": same,
                             "check": "the last timed token through the stack again, launched on a "
                                      "stream, equals the graph's output bit for bit; the stack's "
                                      "oracle parity is a GPU test"}}


def bench_stack_verify(args, layers, cfg, seed):
    """q=4 through the whole stack (moe_ffn_stack_verify_q4: four columns,
    each layer's weights read once per call for all of them), calls replayed
    from CUDA graphs; the distinct experts of each (call, layer) are counted
    afterwards by the same columns through the separate entry points, whose
    result must equal the stack's bit for bit."""
    import torch
    import bit_codebook_quantized_dequant_gb300 as M
    from bit_codebook_quantized_dequant_gb300 import synth as S
    from bit_codebook_quantized_dequant_gb300.workload import Debug, Workspace, to_dev_u16
    nl = len(layers)
    descs = [dl.desc() for dl in layers]
    ws = Workspace(layers[0], 5)
    H = cfg["H"]
    nb = 16
    X = S.tokens(seed, cfg, 4 * nb, start=8192)
    xs = to_dev_u16(X)
    r = torch.zeros(4 * H, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()

    def step(i, s):
        M.moe_ffn_stack_verify_q4(descs, xs.data_ptr() + (i % nb) * 4 * H * 2, r, ws.ptr, ws.nbytes, st, s)

    warm, steps = 3, 8
    for i in range(warm):
        step(i, stream)
    torch.cuda.synchronize()
    graphs = capture_steps(step, warm, steps, stream, chunk=8)
    replay(graphs, stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    replay(graphs, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    assert st.item() == 0, f"device status {st.item()}"
    del graphs
    # the timed calls' columns through the composition: distinct experts per
    # (call, layer), and the last call's result against the stack's
    ws1 = Workspace(layers[0], 1)
    d = Debug(cfg, 4)
    a = torch.zeros(4 * H, dtype=torch.int16, device="cuda")
    y = torch.zeros(4 * H, dtype=torch.float32, device="cuda")
    nbytes, ndist = 0.0, []
    for j in range(steps):
        b = (warm + j) % nb
        rc = torch.from_numpy((X[4 * b:4 * b + 4].astype(np.uint32) << 16).view(np.float32).reshape(-1).copy()).cuda()
        for l in range(nl):
            M.moe_rmsnorm_bf16(rc, 4, H, a)
            M.moe_ffn_verify_q4(descs[l], None, a, y, None, ws1.ptr, ws1.nbytes, st, d.struct)
            nd = len(set(d.t["idx"].cpu().tolist()))
            ndist.append(nd)
            nbytes += algorithmic_bytes_verify(cfg, nd)
            rc += y
    torch.cuda.synchronize()
    assert st.item() == 0, f"device status {st.item()}"
    same = bool(torch.equal(rc, r))
    per_call = nbytes / steps
    hbm_peak, _, peak_kind = _peaks()
    achieved = per_call / (ms * 1e-3) / 1e9
    return {"metric": f"q=4 verification column-tok/s ({nl}-layer stack)", "value": 4.0 / (ms * 1e-3),
            "unit": "column-tok/s", "ms_per_call": ms, "calls_timed": steps, "layers": nl,
            "distinct_experts_per_layer_call": float(np.mean(ndist)),
            "workload": f"prefill-43-layer-stack layers (decode-b1 shapes), 4 independently routed "
                        f"columns through all {nl} layers per call: RMSNorm + q=4 FFN (no dense "
                        f"projection) + fp32 residual per layer",
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": None,
                         "peak_source": f"{peak_kind} hbm_gbs",
                         "algorithmic_bytes_per_launch": per_call},
            "gpu_launches_per_call": 2 * nl + 1, "launch": "CUDA graph replay",
            "parity_after": {"composition_bit_equal": same,
                             "check": "the last timed call's columns through RMSNorm, q=4 and the "
                                      "residual as separate calls equal the stack's output bit for "
                                      "bit; per-column equality with the decode stack and its "
                                      "oracle parity are GPU tests"}}


def bench_expanded(args, hbm_peak, peak_kind):
    """The expand-then-multiply ablation: one decode layer expanded to bf16
    (12.9 GB), decoded with moe_ffn_decode_expanded, beside the fused decode
    of the same packed layer on the same tokens; both from CUDA graphs."""
    import torch
    import bit_codebook_quantized_dequant_gb300 as M
    from bit_codebook_quantized_dequant_gb300 import synth as S
    from bit_codebook_quantized_dequant_gb300.workload import Workspace, build_layer, expand_layer, to_dev_u16
    cfg = S.WORKLOADS[DECODE_WORKLOAD]
    seed = S.workload_seed(DECODE_WORKLOAD)
    dl = build_layer(seed, 7, cfg)
    Lx, keep = expand_layer(dl)
    H, I, k = cfg["H"], cfg["I"], cfg["k"]
    ntok = 256
    xs = to_dev_u16(S.tokens(seed, cfg, ntok, start=2048))
    y = torch.zeros(H, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    wsx_b = M.moe_ffn_expanded_workspace(H, I, cfg["E"], k, 1)
    wsx = torch.zeros(wsx_b, dtype=torch.uint8, device="cuda")
    ws = Workspace(dl, 0)
    desc = dl.desc()
    stream = torch.cuda.Stream()

    def fused(i, s):
        M.moe_ffn_decode(desc, xs.data_ptr() + (i % ntok) * H * 2, y, ws.ptr, ws.nbytes, st, None, s)

    def expanded(i, s):
        M.moe_ffn_decode_expanded(Lx, xs.data_ptr() + (i % ntok) * H * 2, y, wsx, wsx_b, st, s)

    out = {}
    steps = 128
    for name, fn in (("fused", fused), ("expanded", expanded)):
        for i in range(5):
            fn(i, stream)
        torch.cuda.synchronize()
        graphs = capture_steps(fn, 5, steps, stream)
        replay(graphs, stream)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        replay(graphs, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        out[name] = e0.elapsed_time(e1) / steps
        del graphs
    assert st.item() == 0, f"device status {st.item()}"
    ns = k + 1
    xbytes = 2 * (2 * ns * I * H + ns * H * I) + cfg["E"] * H * 2
    res = {"metric": "expand-then-multiply ablation: decode us/token, fused vs expanded bf16 GEMV",
           "us_fused": out["fused"] * 1e3, "us_expanded": out["expanded"] * 1e3,
           "fused_speedup": out["expanded"] / out["fused"],
           "bytes_fused": algorithmic_bytes_decode(cfg), "bytes_expanded": xbytes,
           "expanded_hbm_frac": xbytes / (out["expanded"] * 1e-3) / 1e9 / hbm_peak,
           "workload": "one decode-b1 layer (replica 7), 1 layer resident packed (2.3 GB) and expanded "
                       "to bf16 (12.9 GB); 128 tokens per timing, CUDA graph replay",
           "peak_source": f"{peak_kind} hbm_gbs"}
    del keep, dl, ws
    torch.cuda.empty_cache()
    return res


def bench_packed24(args, hbm_peak, peak_kind):
    """Layout A/B on the decode's integer-pipe budget: one decode-b1 layer with
    its routed down projections in FP3's planes and the same codes, scales and
    codebooks in the Packed24 layout (the same bytes); both decoded from CUDA
    graphs on the same tokens, three alternating rounds each."""
    import torch
    import bit_codebook_quantized_dequant_gb300 as M
    from bit_codebook_quantized_dequant_gb300 import synth as S
    from bit_codebook_quantized_dequant_gb300.workload import Workspace, build_layer, to_dev_u16
    cfg3 = S.WORKLOADS[DECODE_WORKLOAD]
    cfg24 = dict(cfg3, fmt_down=S.FP3_PACKED24)
    seed = S.workload_seed(DECODE_WORKLOAD)
    H = cfg3["H"]
    ntok = 256
    xs = to_dev_u16(S.tokens(seed, cfg3, ntok, start=3072))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    arms = {}
    for name, cfg in (("fp3", cfg3), ("packed24", cfg24)):
        dl = build_layer(seed, 6, cfg)
        ws = Workspace(dl, 0)
        y = torch.zeros(H, dtype=torch.float32, device="cuda")
        arms[name] = (dl, ws, y, dl.desc())
    steps = 128
    graphs = {}
    for name, (dl, ws, y, desc) in arms.items():
        def fn(i, s, desc=desc, ws=ws, y=y):
            M.moe_ffn_decode(desc, xs.data_ptr() + (i % ntok) * H * 2, y, ws.ptr, ws.nbytes, st, None, s)
        for i in range(5):
            fn(i, stream)
        torch.cuda.synchronize()
        graphs[name] = capture_steps(fn, 5, steps, stream)
    times = {n: [] for n in arms}
    for _ in range(3):
        for name in arms:
            replay(graphs[name], stream)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            replay(graphs[name], stream)
            e1.record(stream)
            torch.cuda.synchronize()
            times[name].append(e0.elapsed_time(e1) / steps * 1e3)
    del graphs
    assert st.item() == 0, f"device status {st.item()}"
    same = bool(torch.equal(arms["fp3"][2], arms["packed24"][2]))
    us = {n: statistics.median(t) for n, t in times.items()}
    res = {"metric": "Packed24 layout A/B: decode us/token, routed down projections in FP3 planes "
                     "vs the Packed24 bit order (same codes and bytes)",
           "us_fp3": us["fp3"], "us_packed24": us["packed24"],
           "packed24_slowdown": us["packed24"] / us["fp3"], "rounds_us": times,
           "bytes_per_token": algorithmic_bytes_decode(cfg3),
           "hbm_frac_fp3": algorithmic_bytes_decode(cfg3) / (us["fp3"] * 1e-6) / 1e9 / hbm_peak,
           "hbm_frac_packed24": algorithmic_bytes_decode(cfg3) / (us["packed24"] * 1e-6) / 1e9 / hbm_peak,
           "workload": "one decode-b1 layer (replica 6) in each layout; 128 tokens per timing, median "
                       "of 3 alternating rounds, CUDA graph replay",
           "parity_after": {"last_token_bit_equal": same,
                            "check": "the last timed token's y from the two layouts is equal bit for bit"},
           "peak_source": f"{peak_kind} hbm_gbs"}
    del arms
    torch.cuda.empty_cache()
    return res


def run_sections(args, hbm_peak, tc_peak, peak_kind, cpu=False):
    """The q=4 verification and prefill sections named in --sections (cpu: add
    the oracle's prefill rate on the host to each prefill section)."""
    sec = args.sections.split(",")
    out = {}
    if "verify" in sec:
        out["verify_q4"] = bench_verify(args, hbm_peak, peak_kind, cpu)
    pre = []
    if "prefill" in sec or "prefill3" in sec:
        pre.append(bench_prefill(args, "prefill-h32-fp4", args.prefill_tokens or 2048, tc_peak, hbm_peak,
                                 peak_kind, cpu))
    if "prefill" in sec or "prefill4" in sec:
        pre.append(bench_prefill(args, "prefill-43-layer-stack", args.prefill_tokens or 32512, tc_peak,
                                 hbm_peak, peak_kind, cpu))
    if pre:
        out["prefill"] = pre
    if "ablation" in sec:
        out["expand_then_multiply"] = bench_expanded(args, hbm_peak, peak_kind)
        out["packed24_layout"] = bench_packed24(args, hbm_peak, peak_kind)
    if "stack" in sec:
        out["prefill_stack"], out["decode_stack"] = bench_stack(
            args, args.prefill_tokens or 32512, args.stack_layers, tc_peak, peak_kind)
    return out


def run(args):
    import torch
    import bit_codebook_quantized_dequant_gb300 as M
    from bit_codebook_quantized_dequant_gb300 import synth as S
    from bit_codebook_quantized_dequant_gb300.workload import Workspace, build_layer, to_dev_u16

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    if "decode" not in args.sections.split(","):
        # profiling runs of single sections (no headline line)
        M.load()
        hbm_peak, tc_peak, peak_kind = _peaks()
        print(json.dumps(run_sections(args, hbm_peak, tc_peak, peak_kind)))
        return
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    cfg = S.WORKLOADS[DECODE_WORKLOAD]
    seed = S.workload_seed(DECODE_WORKLOAD)
    M.load()
    R = args.replicas
    layers = [build_layer(seed, r, cfg) for r in range(R)]
    wss = [Workspace(dl, 0) for dl in layers]
    ntok = 1024
    xs_host = S.tokens(seed, cfg, ntok, start=rank_token_start(rank, ntok))
    xs = to_dev_u16(xs_host)                      # [ntok, H] resident in HBM
    H = cfg["H"]
    y = torch.zeros(H, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    descs = [dl.desc() for dl in layers]
    stream = torch.cuda.current_stream()
    xbase, xstride = xs.data_ptr(), H * 2

    def step(i, s):
        r = i % R
        M.moe_ffn_decode(descs[r], xbase + (i % ntok) * xstride, y, wss[r].ptr, wss[r].nbytes, st,
                         None, s)

    # W warm-up steps launched on the stream, then the K timed steps replayed
    # from CUDA graphs (captured and replayed once, untimed, before timing)
    stream = torch.cuda.Stream()
    for i in range(args.warmup):
        step(i, stream)
    torch.cuda.synchronize()
    graphs = capture_steps(step, args.warmup, args.steps, stream)
    replay(graphs, stream)
    torch.cuda.synchronize()
    assert st.item() == 0, f"device status {st.item()}"
    if dist:
        dist.barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        torch.cuda.synchronize()
        ev0.record(stream)
        replay(graphs, stream)
        ev1.record(stream)
        torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    assert st.item() == 0, f"device status {st.item()}"
    del graphs

    # end to end through the same entry point with host buffers: per step the
    # token's x from pinned memory to the device, the decode, and y back to
    # pinned memory, on three streams with two buffers each so that the copies
    # of neighbouring steps overlap the decode; captured and replayed like the
    # device-timed steps
    x_pin = torch.from_numpy(xs_host.view(np.int16)).pin_memory()
    y_pin = torch.empty((args.steps, H), dtype=torch.float32).pin_memory()
    xdev = torch.empty((2, H), dtype=torch.int16, device="cuda")
    ydev = torch.empty((2, H), dtype=torch.float32, device="cuda")
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {n: [torch.cuda.Event(), torch.cuda.Event()] for n in ("x", "used", "y", "out")}

    def e2e_chunk(first, n, s):
        s_in.wait_stream(s)
        s_out.wait_stream(s)
        for j in range(n):
            i, b = first + j, (first + j) % 2
            r = i % R
            if j >= 2:
                s_in.wait_event(ev["used"][b])
            with torch.cuda.stream(s_in):
                xdev[b].copy_(x_pin[i % ntok], non_blocking=True)
                ev["x"][b].record(s_in)
            s.wait_event(ev["x"][b])
            if j >= 2:
                s.wait_event(ev["out"][b])
            M.moe_ffn_decode(descs[r], xdev[b], ydev[b], wss[r].ptr, wss[r].nbytes, st, None, s)
            ev["used"][b].record(s)
            ev["y"][b].record(s)
            s_out.wait_event(ev["y"][b])
            with torch.cuda.stream(s_out):
                y_pin[i - args.warmup].copy_(ydev[b], non_blocking=True)
                ev["out"][b].record(s_out)
        s.wait_stream(s_in)
        s.wait_stream(s_out)

    egraphs, i0 = [], args.warmup
    while i0 < args.warmup + args.steps:
        m = min(64, args.warmup + args.steps - i0)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            e2e_chunk(i0, m, stream)
        egraphs.append(g)
        i0 += m
    replay(egraphs, stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    replay(egraphs, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = e0.elapsed_time(e1)
    assert st.item() == 0, f"device status {st.item()}"
    # the end-to-end outputs are those of the device-timed path
    for i in range(min(4, args.steps)):
        step(args.warmup + i, stream)
        torch.cuda.synchronize()
        assert torch.equal(y.cpu(), y_pin[i]), "end-to-end output differs"
    del egraphs

    if dist:
        ms, ms_e2e = max_over_ranks([ms, ms_e2e], dist, device="cuda")
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    hbm_peak, tc_peak, peak_kind = _peaks()
    per_tok = algorithmic_bytes_decode(cfg)
    ms_step = ms / args.steps
    achieved = per_tok / (ms_step * 1e-3) / 1e9
    value = job_throughput(world, args.steps, ms)
    e2e = job_throughput(world, args.steps, ms_e2e)
    cpu = None
    parity_after = None
    if world == 1 and not args.no_cpu_baseline:
        tps, sample, _ = cpu_baseline(DECODE_WORKLOAD, 20)
        cpu = {"value": tps, "unit": "tok/s", "cores": 1, "kind": "oracle", "sample": sample}
        parity_after = decode_parity_after(layers[0], wss[0], xs_host, cfg, seed, ntok=4)
    traffic = _traffic("ffn_kernel<1>", "bit_codebook_quantized_dequant_gb300/csrc/decode.cu")
    wbytes = R * layers[0].weight_bytes()
    extra = {}
    if world == 1:
        del layers, wss
        torch.cuda.empty_cache()
        extra = run_sections(args, hbm_peak, tc_peak, peak_kind, cpu=not args.no_cpu_baseline)
    line = {
        "metric": DECODE_METRIC,
        "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8-dot/fp32",
        "data": "synthetic (seeded SplitMix64 codes, scales, codebooks; x ~ N(0,1) bf16)",
        "config": {"workload": WORKLOAD, "replicas": R,
                   "l2": f"inputs larger than L2: {R} independently seeded layer replicas "
                         f"({wbytes / 1e9:.1f} GB), cycled per step",
                   "tokens_timed": world * args.steps,
                   "token_pool": ntok,
                   "launch": "K steps replayed from CUDA graphs (stream-launched warm-up before)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": traffic,
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "algorithmic_bytes_per_launch": per_tok},
        "gpu_launches": args.steps,
        "e2e": {"value": e2e, "unit": "tok/s", "h2d_bytes_per_step": H * 2,
                "d2h_bytes_per_step": H * 4},
        "clocks": clk.summary(),
        "cpu_baseline": cpu,
        "parity_after": parity_after,
    }
    _target(line["roofline"], TARGET_HBM)
    line.update(extra)
    print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--replicas", type=int, default=8)
    ap.add_argument("--impl", default="moeq", choices=["moeq", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sections", default="decode,verify,prefill,ablation,stack",
                    help="comma list of decode, verify, prefill (= prefill3,prefill4), ablation, stack; "
                         "without decode only the named sections run (profiling)")
    ap.add_argument("--stack-layers", type=int, default=43)
    ap.add_argument("--prefill-tokens", type=int, default=0,
                    help="tokens of the prefill sections (default: the workloads' 2048 and 32512); "
                         "smaller counts for profiling")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run(args)


if __name__ == "__main__":
    main()
