"""Host-side checks of the workload recipe: the tiny decode workload's seed
rule (seeds whose rank-2/3 router logit gap is below 1e-3 are rejected)."""
import numpy as np

import oracle as O
from bit_codebook_quantized_dequant_gb300 import synth as S


def _oracle_gap(seed, cfg):
    # the gap in the precision that takes the decision (fp32 canonical-order logits)
    lg = np.asarray(O.router_logits(S.tokens(seed, cfg, 1), S.router_weights(seed, 0, cfg))[0],
                    dtype=np.float64)
    s = np.sort(lg)[::-1]
    return s[cfg["k"] - 1] - s[cfg["k"]]


def test_config0_seed_rule_rejects_small_gaps():
    cfg = S.WORKLOADS["tiny-decode"]
    base = S.workload_seed("tiny-decode")
    seeds = S.config0_seeds(160, cfg)
    # consecutive seeds, except base + 156, whose rank-2/3 gap is ~3e-5
    assert seeds[:156] == list(range(base, base + 156))
    assert base + 156 not in seeds and seeds[156] == base + 157
    assert _oracle_gap(base + 156, cfg) < 1e-3
    for s in seeds[150:]:
        assert _oracle_gap(s, cfg) >= S.CONFIG0_MIN_GAP - 1e-5


def test_selection_gap_matches_sorted_logits():
    # the screening gap is the k-th minus the (k+1)-th largest logit
    cfg = dict(S.WORKLOADS["tiny-decode"], k=3)
    seed = S.workload_seed("tiny-decode") + 7
    g = S.selection_gap(seed, cfg)
    assert g >= 0 and abs(g - _oracle_gap(seed, cfg)) < 1e-5
