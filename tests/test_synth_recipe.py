"""The input recipe on CPU: the redraw rule leaves every token of the full-size routed
workloads with top-(k+1) selection scores at least 1e-3 apart (so expert ids cannot flip on
rounding), and the prefill workload's per-expert counts are Zipf-skewed (a head of thousands
of tokens, a median of tens)."""
import numpy as np
import pytest

import parity
from block_quantized_moe_router_gb300 import synth


@pytest.mark.parametrize("name", ["tiny", "dec1", "dec8"])
def test_redraw_makes_gaps(name):
    cfg = synth.CONFIGS[name]
    res = parity.gap_safe_resample(cfg, 0)
    inp = synth.make_inputs(cfg, seed=0, resample=res, with_weights=False)
    assert parity.gap_violations(cfg, parity.oracle_route(cfg, inp)["score"]) == []


def test_prefill_counts_are_skewed():
    cfg = synth.CONFIGS["pre4096"]
    res = parity.gap_safe_resample(cfg, 0)
    inp = synth.make_inputs(cfg, seed=0, resample=res, with_weights=False)
    r = parity.oracle_route(cfg, inp)
    assert parity.gap_violations(cfg, r["score"]) == []
    cnt = np.sort(np.bincount(r["ids"].ravel(), minlength=cfg.E))[::-1]
    assert cnt.sum() == cfg.T * cfg.k and cnt[0] <= cfg.T
    assert cnt[0] > 3000 and cnt[9] > 500           # the head
    assert 10 <= np.median(cnt) <= 60                 # a median of tens
    assert cnt[0] > 50 * np.median(cnt)
    assert (cnt > 0).sum() >= cfg.E - 4               # nearly every expert touched
