"""CPU test of the decode timeline summary (bit_codebook_quantized_dequant_gb300.timeline)
on a synthetic trace: event codes, roles and the packed unit kinds are read
as the decode kernel writes them."""
import numpy as np

from bit_codebook_quantized_dequant_gb300 import timeline as T


def _trace():
    G, cap = 4, 8
    rel = np.zeros((G, 4, cap))
    ev = np.zeros((G, 4, cap), np.int64)
    un = np.zeros((G, 4, cap), np.int64)
    valid = np.zeros((G, 4, cap), bool)
    for b in range(G):
        valid[b, T.ROLE_PRODUCER, :2] = True
        ev[b, T.ROLE_PRODUCER, :2] = [T.EV_TAKE, T.EV_TOPK]
        rel[b, T.ROLE_PRODUCER, :2] = [0.5 * b, 8.0 + b]
        # group 0: a GU fill (kind 2) ready at 10, done at 12; group 1: a DOWN fill (kind 4)
        valid[b, T.ROLE_GROUP0, :2] = True
        ev[b, T.ROLE_GROUP0, :2] = [T.EV_READY, T.EV_DONE]
        un[b, T.ROLE_GROUP0, :2] = (2 << 28) | (1 << 20) | 3
        rel[b, T.ROLE_GROUP0, :2] = [10.0, 12.0]
        valid[b, T.ROLE_GROUP1, :3] = True
        ev[b, T.ROLE_GROUP1, :3] = [T.EV_READY, T.EV_DONE, T.EV_READY]
        un[b, T.ROLE_GROUP1, :3] = [(4 << 28) | 7, (4 << 28) | 7, 0xffffffff]  # then an end marker
        rel[b, T.ROLE_GROUP1, :3] = [20.0, 22.0 + b, 23.0]
        valid[b, T.ROLE_TEARDOWN, :2] = True
        ev[b, T.ROLE_TEARDOWN, :2] = [T.EV_START, T.EV_EPI_END]
        rel[b, T.ROLE_TEARDOWN, :2] = [24.0, 25.0 + b]
    return rel, ev, un, valid


def test_timeline_summary_reads_events_by_role_and_kind():
    lines = T.summarize(*_trace())
    text = "\n".join(lines)
    assert lines[0].startswith("span first..last event (us): 28.000")
    get = {l.split(" min")[0].strip(): l for l in lines[1:]}
    assert "min    0.00" in get["producer TAKE"] and "max    1.50" in get["producer TAKE"]
    assert "min    8.00" in get["producer route known"] and "(n=4)" in get["producer route known"]
    assert "min   10.00" in get["READY GU"] and "(n=4)" in get["READY GU"]
    assert "min   22.00" in get["DONE  DOWN"] and "max   25.00" in get["DONE  DOWN"]
    assert "READY END" in text and "(n=4)" in get["READY END"]
    assert "min   25.00" in get["arrival on the done counter"] and "max   28.00" in get["arrival on the done counter"]
    assert "down-done wait passed (combining CTAs)       (none)" in text
