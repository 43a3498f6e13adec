"""Timeline of one decode launch from the kernel's debug trace.

moe_ffn_decode records, when moeq_debug.trace is set, globaltimer events per
CTA and role (compute group 0, producer warp, teardown, compute group 1):
items taken, the routing known, fills issued, fills ready and done by kind,
and the teardown steps (compute ended, the wait for every down item passed,
the combined rows written, the arrival on the done counter). This module runs
a few decode-b1 tokens over seeded layer replicas, traces the last one and
prints per-event statistics across the CTAs (microseconds from the first
event of the launch).

    python -m bit_codebook_quantized_dequant_gb300.timeline [--replicas 4] [--cap 96]
"""
from __future__ import annotations

import argparse

import numpy as np

# event codes of include/moeq.h (MOEQ_TRACE_*)
EV_START, EV_TAKE, EV_TOPK, EV_ISSUED, EV_READY, EV_DONE, EV_EPI_END = 1, 2, 3, 4, 5, 6, 8
ROLE_GROUP0, ROLE_PRODUCER, ROLE_TEARDOWN, ROLE_GROUP1 = 0, 1, 2, 3
# fill kinds of the packed unit word (kind << 28 | slot << 20 | chunk)
KIND = {0: "ROUTER", 1: "SGU", 2: "GU", 3: "SDOWN", 4: "DOWN", 5: "ROUTE", 6: "DENSE", 7: "END", 15: "END"}


def collect(replicas: int = 4, cap: int = 96, warm: int = 11):
    """Decodes warm + 1 tokens, tracing the last; returns (rel_us, event, unit, valid)
    arrays shaped [CTAs, 4 roles, cap]."""
    import torch
    import bit_codebook_quantized_dequant_gb300 as M
    from bit_codebook_quantized_dequant_gb300 import synth as S
    from bit_codebook_quantized_dequant_gb300.workload import Workspace, build_layer, to_dev_u16
    cfg = S.WORKLOADS["decode-b1"]
    seed = S.workload_seed("decode-b1")
    layers = [build_layer(seed, r, cfg) for r in range(replicas)]
    wss = [Workspace(dl, 0) for dl in layers]
    descs = [dl.desc() for dl in layers]
    H = cfg["H"]
    xs = to_dev_u16(S.tokens(seed, cfg, 16))
    y = torch.zeros(H, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    G = torch.cuda.get_device_properties(0).multi_processor_count
    tr = torch.zeros(G * 4 * cap * 2, dtype=torch.int64, device="cuda")
    dbg = M.MoeqDebug()
    dbg.trace = tr.data_ptr()
    dbg.trace_cap = cap
    for i in range(warm + 1):
        M.moe_ffn_decode(descs[i % replicas], xs.data_ptr() + (i % 16) * H * 2, y, wss[i % replicas].ptr,
                         wss[i % replicas].nbytes, st, dbg if i == warm else None)
    torch.cuda.synchronize()
    if st.item() != 0:
        raise RuntimeError(f"device status {st.item()}")
    t = tr.cpu().numpy().reshape(G, 4, cap, 2)
    ts = t[..., 0].astype(np.int64)
    info = t[..., 1].astype(np.int64)
    valid = ts > 0
    rel = (ts - ts[valid].min()) / 1000.0
    return rel, (info >> 32) & 0xffffffff, info & 0xffffffff, valid


def summarize(rel, ev, unit, valid) -> list:
    """Per-event statistics lines."""
    out = []

    def stats(name, vals):
        v = np.asarray(vals, dtype=float)
        if v.size == 0:
            out.append(f"{name:44s} (none)")
            return
        out.append(f"{name:44s} min {v.min():7.2f} p10 {np.percentile(v, 10):7.2f} med {np.median(v):7.2f} "
                   f"p90 {np.percentile(v, 90):7.2f} max {v.max():7.2f} (n={v.size})")

    out.append(f"span first..last event (us): {rel[valid].max():.3f}")
    for code, name in ((EV_TAKE, "producer TAKE"), (EV_TOPK, "producer route known"),
                       (EV_ISSUED, "producer ISSUED")):
        stats(name, rel[:, ROLE_PRODUCER][valid[:, ROLE_PRODUCER] & (ev[:, ROLE_PRODUCER] == code)])
    ready, done = {}, {}
    for role in (ROLE_GROUP0, ROLE_GROUP1):
        m = valid[:, role]
        kinds = (unit[:, role] >> 28) & 15
        for k in np.unique(kinds[m]):
            ready.setdefault(int(k), []).extend(rel[:, role][m & (ev[:, role] == EV_READY) & (kinds == k)])
            done.setdefault(int(k), []).extend(rel[:, role][m & (ev[:, role] == EV_DONE) & (kinds == k)])
    for k in sorted(ready):
        stats(f"READY {KIND.get(k, k)}", ready[k])
        stats(f"DONE  {KIND.get(k, k)}", done.get(k, []))
    # per fill kind: compute time (DONE - READY of the same fill) and the
    # group's idle gap before it (READY - the group's previous DONE)
    busy, idle = {}, {}
    for b in range(rel.shape[0]):
        for role in (ROLE_GROUP0, ROLE_GROUP1):
            prev_done, ready_at = None, None
            for i in range(rel.shape[2]):
                if not valid[b, role, i]:
                    continue
                k = int((unit[b, role, i] >> 28) & 15)
                if ev[b, role, i] == EV_READY:
                    ready_at = rel[b, role, i]
                    if prev_done is not None:
                        idle.setdefault(k, []).append(ready_at - prev_done)
                elif ev[b, role, i] == EV_DONE and ready_at is not None:
                    busy.setdefault(k, []).append(rel[b, role, i] - ready_at)
                    prev_done = rel[b, role, i]
    for k in sorted(busy):
        stats(f"compute time per fill {KIND.get(k, k)}", busy[k])
    for k in sorted(idle):
        stats(f"group idle before a fill {KIND.get(k, k)}", idle[k])
    m = valid[:, ROLE_TEARDOWN]
    e = ev[:, ROLE_TEARDOWN]
    stats("teardown entered (compute ended)", rel[:, ROLE_TEARDOWN][m & (e == EV_START)])
    stats("down-done wait passed (combining CTAs)", rel[:, ROLE_TEARDOWN][m & (e == EV_READY)])
    stats("combined rows written", rel[:, ROLE_TEARDOWN][m & (e == EV_DONE)])
    stats("arrival on the done counter", rel[:, ROLE_TEARDOWN][m & (e == EV_EPI_END)])
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--replicas", type=int, default=4)
    ap.add_argument("--cap", type=int, default=96)
    args = ap.parse_args()
    print("\n".join(summarize(*collect(args.replicas, args.cap))))


if __name__ == "__main__":
    main()
