"""Pins of the oracle's routing (CPU only).

Routing kinds of the spark_model MoE pages: softmax top-K (moe/init.rs `moe_topk_softmax`
handles), sigmoid scoring with a correction bias used for selection only (moe/mod.rs
`correction_bias_dev` field doc), static hash routing through tid2eid (moe/init.rs
`new_with_hash` doc), softmax + bias routing over the real and zero-computation experts
(moe/mod.rs, `moe_topk_softmax_bias` handles, `router_logits_n` field doc).  Checked against brute force over every k-subset, closed forms and the
weight-sum invariant.
"""
import itertools
import math

import numpy as np
import pytest

from block_quantized_moe_router_gb300 import synth


def _bf16(a):
    import torch
    return synth.bf16_bits(torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16))


def _brute_topk(v, k):
    """Best k-subset by brute force: the one whose minimum beats every unselected score."""
    E = len(v)
    best = None
    for sub in itertools.combinations(range(E), k):
        rest = [e for e in range(E) if e not in sub]
        if not rest or min(v[list(sub)]) > max(v[rest]):
            assert best is None, "ties in test data"
            best = set(sub)
    return best


def _score(scoring, l):
    if scoring == 0:
        return l
    if scoring == 1:
        return 1 / (1 + np.exp(-l))
    if scoring == 4:
        p = np.exp(l - l.max())
        return p / p.sum()                  # softmax probability (the bias is added on top)
    return np.sqrt(np.log1p(np.exp(l)))   # sqrt(softplus)


@pytest.mark.parametrize("scoring", [0, 1, 3, 4])
@pytest.mark.parametrize("E,k", [(6, 2), (8, 3), (10, 4), (5, 5)])
def test_topk_matches_brute_force(orc, scoring, E, k):
    rng = np.random.default_rng(E * 10 + k + scoring)
    T = 6
    logits = rng.standard_normal((T, E)).astype(np.float32) * 2
    bias = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    r = orc.route(T=T, E=E, k=k, scoring=scoring, renorm=True, scaling=2.5 if scoring else 1.0,
                  logits_in=logits, bias=bias)
    for t in range(T):
        l = logits[t].astype(np.float64)
        v = l if scoring == 0 else _score(scoring, l) + bias
        assert set(r["ids"][t]) == _brute_topk(v, k)
        # descending selection score
        sel = v[r["ids"][t]]
        assert np.all(np.diff(sel) < 0)


def test_softmax_weights_closed_form(orc):
    rng = np.random.default_rng(3)
    T, E, k = 5, 16, 4
    logits = rng.standard_normal((T, E)).astype(np.float32)
    r = orc.route(T=T, E=E, k=k, scoring=0, renorm=True, logits_in=logits)
    r_nr = orc.route(T=T, E=E, k=k, scoring=0, renorm=False, logits_in=logits)
    for t in range(T):
        l = logits[t].astype(np.float64)
        ids = r["ids"][t]
        # renormalised top-k of softmax == softmax over the selected logits
        sm_sel = np.exp(l[ids]) / np.exp(l[ids]).sum()
        assert np.allclose(r["w"][t], sm_sel, rtol=0, atol=1e-15)
        p = np.exp(l - l.max()) / np.exp(l - l.max()).sum()
        assert np.allclose(r_nr["w"][t], p[ids], rtol=0, atol=1e-15)
        assert abs(r["w"][t].sum() - 1.0) < 1e-12


def test_sigmoid_bias_selects_but_does_not_weight(orc):
    E, k = 4, 2
    logits = np.array([[2.0, 1.0, 0.0, -1.0]], np.float32)
    bias = np.array([0.0, 0.0, 0.5, 0.0], np.float32)
    r = orc.route(T=1, E=E, k=k, scoring=1, renorm=True, scaling=2.5, logits_in=logits, bias=bias)
    # scores: s = sigmoid(l) = .881, .731, .5, .269; +bias: .881, .731, 1.0, .269
    assert list(r["ids"][0]) == [2, 0]
    s = 1 / (1 + np.exp(-np.array([0.0, 2.0])))
    assert np.allclose(r["w"][0], s / s.sum() * 2.5, atol=1e-15)
    r_nr = orc.route(T=1, E=E, k=k, scoring=1, renorm=False, scaling=1.0, logits_in=logits, bias=bias)
    assert np.allclose(r_nr["w"][0], s, atol=1e-15)


def test_sqrt_softplus_weights_closed_form(orc):
    rng = np.random.default_rng(21)
    T, E, k = 6, 24, 5
    logits = (rng.standard_normal((T, E)) * 3).astype(np.float32)
    logits[0, 3] = 45.0   # deep in the linear tail of softplus
    bias = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    r = orc.route(T=T, E=E, k=k, scoring=3, renorm=True, scaling=1.5, logits_in=logits, bias=bias)
    for t in range(T):
        s = np.sqrt(np.log1p(np.exp(logits[t].astype(np.float64))))
        ids = r["ids"][t]
        assert np.allclose(r["w"][t], s[ids] / s[ids].sum() * 1.5, rtol=0, atol=1e-14)
    assert 3 in r["ids"][0] and abs(np.sqrt(45.0) - np.sqrt(np.log1p(np.exp(45.0)))) < 1e-12


def test_sqrt_softplus_special_values(orc):
    # softplus(l) = a when l = ln(e^a - 1): a = 1, 4, 9 give scores 1, 2, 3 -> weights 1:2:3
    a = np.array([1.0, 4.0, 9.0])
    l = np.log(np.expm1(a))
    logits = np.array([[l[0], -5.0, l[2], l[1], -7.0]], np.float32)
    r = orc.route(T=1, E=5, k=3, scoring=3, renorm=True, scaling=1.0, logits_in=logits)
    assert list(r["ids"][0]) == [2, 3, 0]
    assert np.allclose(r["w"][0], [3 / 6, 2 / 6, 1 / 6], rtol=0, atol=1e-6)
    # without a bias the ranking is the logit ranking, as for softmax (both are monotone)
    rng = np.random.default_rng(8)
    lg = (rng.standard_normal((16, 40)) * 4).astype(np.float32)
    a = orc.route(T=16, E=40, k=7, scoring=3, logits_in=lg)
    b = orc.route(T=16, E=40, k=7, scoring=0, logits_in=lg)
    assert np.array_equal(a["ids"], b["ids"])


def test_softmax_bias_selects_but_does_not_weight(orc):
    # p = softmax([2, 1, 0, -1]) = .6439, .2369, .0871, .0321; + bias (0, 0, .6, 0) moves
    # expert 2 (.6871) above expert 1 (.2369): top-2 = [2, 0], weighted by p alone
    logits = np.array([[2.0, 1.0, 0.0, -1.0]], np.float32)
    bias = np.array([0.0, 0.0, 0.6, 0.0], np.float32)
    e = [math.exp(v) for v in (2.0, 1.0, 0.0, -1.0)]
    p = [v / sum(e) for v in e]
    r = orc.route(T=1, E=4, k=2, scoring=4, renorm=True, scaling=1.5, logits_in=logits, bias=bias)
    assert list(r["ids"][0]) == [2, 0]
    assert np.allclose(r["w"][0], [p[2] / (p[0] + p[2]) * 1.5, p[0] / (p[0] + p[2]) * 1.5],
                       rtol=0, atol=1e-12)
    r_nr = orc.route(T=1, E=4, k=2, scoring=4, renorm=False, scaling=1.0, logits_in=logits,
                     bias=bias)
    assert np.allclose(r_nr["w"][0], [p[2], p[0]], rtol=0, atol=1e-12)
    # with no bias it is plain softmax top-K
    r0 = orc.route(T=1, E=4, k=2, scoring=4, renorm=False, logits_in=logits)
    r1 = orc.route(T=1, E=4, k=2, scoring=0, renorm=False, logits_in=logits)
    assert np.array_equal(r0["ids"], r1["ids"]) and np.allclose(r0["w"], r1["w"], rtol=0, atol=1e-15)


@pytest.mark.parametrize("scoring,scaling", [(0, 1.0), (1, 2.5), (3, 1.0), (4, 1.5)])
def test_weight_sum_invariant(orc, scoring, scaling):
    rng = np.random.default_rng(11)
    T, E, k = 64, 256, 8
    logits = rng.standard_normal((T, E)).astype(np.float32) * 1.7
    r = orc.route(T=T, E=E, k=k, scoring=scoring, renorm=True, scaling=scaling, logits_in=logits,
                  bias=rng.uniform(-0.1, 0.1, E).astype(np.float32))
    assert np.allclose(r["w"].sum(1), scaling, rtol=0, atol=1e-12)
    for t in range(T):
        assert len(set(r["ids"][t])) == k
        assert r["ids"][t].min() >= 0 and r["ids"][t].max() < E


def test_ties_break_to_lower_index(orc):
    logits = np.array([[1.0, 3.0, 3.0, 2.0, 3.0]], np.float32)
    r = orc.route(T=1, E=5, k=3, scoring=0, logits_in=logits)
    assert list(r["ids"][0]) == [1, 2, 4]


def test_router_gemm_fp64(orc):
    rng = np.random.default_rng(5)
    T, E, H = 3, 7, 64
    x = rng.standard_normal((T, H)).astype(np.float32)
    w = (rng.standard_normal((E, H)) * 0.02).astype(np.float32)
    xb, wb = _bf16(x), _bf16(w)
    r = orc.route(T=T, E=E, k=2, scoring=0, x_bf16=xb, w_router_bf16=wb)
    xf = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    wf = (wb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.allclose(r["logits"], xf @ wf.T, rtol=0, atol=1e-14)


def test_hash_routing_and_bad_ids(orc):
    tid2eid = np.array([[0, 3], [2, 1], [5, 0], [1, -1]], np.int64)   # rows 2 and 3 hold bad ids
    tok = np.array([1, 0, 2, 3, 7], np.int32)                          # token 7 is out of vocab
    r = orc.route(T=5, E=4, k=2, scoring=2, tid2eid=tid2eid, token_ids=tok, vocab=4)
    assert r["ids"].tolist() == [[2, 1], [0, 3], [-1, 0], [1, -1], [-1, -1]]
    assert np.allclose(r["w"], [[.5, .5], [.5, .5], [0, .5], [.5, 0], [0, 0]])
    assert r["status"] == (1 | 2)


def test_nonfinite_logits_rank_last(orc):
    logits = np.array([[np.nan, 0.5, np.inf, -1.0, 0.2]], np.float32)
    r = orc.route(T=1, E=5, k=3, scoring=0, logits_in=logits)
    assert list(r["ids"][0]) == [1, 4, 3]
    assert r["status"] == 4
    r = orc.route(T=1, E=5, k=4, scoring=1, scaling=1.0, logits_in=logits)
    assert list(r["ids"][0])[:3] == [1, 4, 3] and r["w"][0][3] == 0.0


def test_hash_with_sqrtsoftplus_weights(orc):
    """Score-weighted hash routing (scoring 5): the table picks the experts, the router's
    sqrt(softplus) scores weight them.  softplus(l) = a exactly when l = ln(e^a - 1), so the
    scores of a = 1, 4, 9 are 1, 2, 3 and the renormalised weights are 1/6, 2/6, 3/6 (to the
    float32 rounding of the logits, a few 1e-8)."""
    a = np.array([1.0, 4.0, 9.0])
    l = np.log(np.expm1(a))
    E, k = 6, 3
    logits = np.full((4, E), -3.0, np.float32)
    logits[:, 4], logits[:, 1], logits[:, 5] = l[0], l[1], l[2]
    tid2eid = np.array([[4, 1, 5], [5, 4, 1], [1, 9, 5], [4, 1, 5]], np.int64)  # row 2: a bad id
    tok = np.array([0, 1, 2, 3], np.int32)
    logits[3, 1] = np.nan                                   # a non-finite score at a chosen id
    r = orc.route(T=4, E=E, k=k, scoring=5, renorm=True, scaling=2.0, logits_in=logits,
                  tid2eid=tid2eid, token_ids=tok, vocab=4)
    # ids in table order, bad entries dropped
    assert r["ids"].tolist() == [[4, 1, 5], [5, 4, 1], [1, -1, 5], [4, 1, 5]]
    assert np.allclose(r["w"][0], np.array([1, 2, 3]) / 6 * 2.0, rtol=0, atol=1e-6)
    assert np.allclose(r["w"][1], np.array([3, 1, 2]) / 6 * 2.0, rtol=0, atol=1e-6)
    # the dropped pair is left out of the renormalisation: scores 2 and 3 -> 2/5, 3/5
    assert np.allclose(r["w"][2], np.array([2, 0, 3]) / 5 * 2.0, rtol=0, atol=1e-6)
    # a NaN logit weighs 0 and the others renormalise among themselves: 1/4, 3/4
    assert np.allclose(r["w"][3], np.array([1, 0, 3]) / 4 * 2.0, rtol=0, atol=1e-6)
    assert r["status"] == (1 | 4)
    # without renormalisation the weight is the score itself times the scaling
    r_nr = orc.route(T=1, E=E, k=k, scoring=5, renorm=False, scaling=1.5, logits_in=logits[:1],
                     tid2eid=tid2eid, token_ids=tok[:1], vocab=4)
    assert np.allclose(r_nr["w"][0], np.array([1, 2, 3]) * 1.5, rtol=0, atol=1e-6)


def test_hash_sqrtsoftplus_reduces_to_plain_hash(orc):
    """With equal logits every kept pair scores alike, so the weights are the plain hash
    weights scaling / k (the same ids, from the table path that uses no logits), and the
    weights of every token sum to the scaling."""
    rng = np.random.default_rng(21)
    V, E, k, T = 50, 16, 4, 30
    tid2eid = np.stack([rng.permutation(E)[:k] for _ in range(V)]).astype(np.int64)
    tok = rng.integers(0, V, T).astype(np.int32)
    flat = np.full((T, E), 0.7, np.float32)
    a = orc.route(T=T, E=E, k=k, scoring=5, renorm=True, scaling=1.0, logits_in=flat,
                  tid2eid=tid2eid, token_ids=tok, vocab=V)
    b = orc.route(T=T, E=E, k=k, scoring=2, scaling=1.0, tid2eid=tid2eid, token_ids=tok, vocab=V)
    assert np.array_equal(a["ids"], b["ids"])
    assert np.allclose(a["w"], b["w"], rtol=0, atol=1e-15)
    lg = (rng.standard_normal((T, E)) * 2).astype(np.float32)
    c = orc.route(T=T, E=E, k=k, scoring=5, renorm=True, scaling=2.5, logits_in=lg,
                  tid2eid=tid2eid, token_ids=tok, vocab=V)
    assert np.array_equal(c["ids"], b["ids"])
    assert np.allclose(c["w"].sum(1), 2.5, rtol=0, atol=1e-12)
    # the weights follow the logits' order within a token (sqrt(softplus) is increasing)
    for t in range(T):
        lsel = lg[t, c["ids"][t]]
        assert np.array_equal(np.argsort(lsel, kind="stable"), np.argsort(c["w"][t], kind="stable"))
