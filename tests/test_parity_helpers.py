"""The weight-sensitivity closed forms behind the GPU routing-weight bound (tests/parity.py),
checked against central finite differences of the oracle's route (CPU only)."""
import numpy as np
import pytest

import parity
from block_quantized_moe_router_gb300 import synth


@pytest.mark.parametrize("renorm", [True, False])
@pytest.mark.parametrize("scoring", [0, 1, 3, 4, 5])
def test_weight_sensitivity_matches_finite_differences(orc, scoring, renorm):
    rng = np.random.default_rng(100 + scoring)
    T, E, k, V = 5, 12, 4, 20
    cfg = synth.MoeConfig("fd", T=T, H=128, I=128, E=E, k=k, scoring=scoring, renorm=renorm,
                          scaling=2.5 if scoring else 1.0, vocab=V)
    logits = (rng.standard_normal((T, E)) * 1.5).astype(np.float32)
    bias = rng.uniform(-0.05, 0.05, E).astype(np.float32) * (0.1 if scoring == 4 else 1.0)
    kw = dict(T=T, E=E, k=k, scoring=scoring, renorm=renorm, scaling=cfg.scaling)
    if scoring == 5:
        kw.update(tid2eid=np.stack([rng.permutation(E)[:k] for _ in range(V)]).astype(np.int64),
                  token_ids=rng.integers(0, V, T).astype(np.int32), vocab=V)
    elif scoring != 0:
        kw.update(bias=bias)
    ref = orc.route(logits_in=logits, **kw)
    J = parity._weight_sensitivity(cfg, ref)
    h = 1e-3
    J_fd = np.zeros_like(J)
    for i in range(E):
        lp, lm = logits.astype(np.float64).copy(), logits.astype(np.float64).copy()
        lp[:, i] += h
        lm[:, i] -= h
        rp = orc.route(logits_in=lp.astype(np.float32), **kw)
        rm = orc.route(logits_in=lm.astype(np.float32), **kw)
        assert np.array_equal(rp["ids"], ref["ids"]) and np.array_equal(rm["ids"], ref["ids"])
        dp = (lp.astype(np.float32) - lm.astype(np.float32)).astype(np.float64)[:, i:i + 1]
        J_fd += np.abs((rp["w"] - rm["w"]) / dp)
    assert np.allclose(J, J_fd, rtol=1e-2, atol=1e-6)
