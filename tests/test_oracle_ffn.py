"""Pins of the oracle's expert FFN + combine (CPU only).

The MoE block of the spark_model pages (moe/mod.rs module doc: gate+up, SiLU, down, then
the top-K weighted sum plus the shared expert) is expanded into a dense masked mixture,
out_t = sum_e gate_te * FFN_e(x_t) + FFN_s(x_t), with every expert dequantized to a dense
fp64 matrix and evaluated with numpy matmuls; the oracle's pair-by-pair loop must agree.
"""
import numpy as np
import pytest
import torch

from block_quantized_moe_router_gb300 import synth


def _np(inp, key):
    return synth.to_numpy_proj(inp.get(key))


def _dense(orc, p, e, N, K):
    sv = 16 if p["fmt"] == 0 else 32
    pk = p["packed"].reshape(-1, N, K // 2)[e]
    sc = p["scales"].reshape(-1, N, K // sv)[e]
    g = 1.0 if p["globals"] is None else float(p["globals"][e])
    return orc.dequant(pk, sc, g, p["fmt"])


def _silu(z):
    return z / (1 + np.exp(-z))


def _dense_mixture(orc, cfg, inp, ids, w, act_mode=0, g1=1.0, g2=1.0):
    x = inp["x"].float().double().numpy()
    if act_mode == 1:
        a = orc.quant_nvfp4(x.astype(np.float32), g1)[2]
    else:
        a = x
    T, H, E = cfg.T, cfg.H, cfg.E
    gate = np.zeros((T, E))
    for t in range(T):
        for j in range(cfg.k):
            if ids[t, j] >= 0:
                gate[t, ids[t, j]] += w[t, j]
    out = np.zeros((T, H))

    def ffn(pg, pu, pd, e, I):
        Wg, Wu, Wd = _dense(orc, pg, e, I, H), _dense(orc, pu, e, I, H), _dense(orc, pd, e, H, I)
        h = _silu(a @ Wg.T) * (a @ Wu.T)
        if act_mode == 1:
            h = orc.quant_nvfp4(h.astype(np.float32), g2)[2]
        return h @ Wd.T

    for e in range(E):
        out += gate[:, e:e + 1] * ffn(_np(inp, "gate"), _np(inp, "up"), _np(inp, "down"), e, cfg.I)
    if cfg.I_shared:
        out += ffn(_np(inp, "sh_gate"), _np(inp, "sh_up"), _np(inp, "sh_down"), 0, cfg.I_shared)
    return out


def _oracle_ffn(orc, cfg, inp, ids, w, act_mode=0, g1=1.0, g2=1.0):
    return orc.moe_ffn(T=cfg.T, E=cfg.E, H=cfg.H, I=cfg.I, k=cfg.k, gate=_np(inp, "gate"),
                       up=_np(inp, "up"), down=_np(inp, "down"), x_bf16=synth.bf16_bits(inp["x"]),
                       ids=ids, w=w, sh_I=cfg.I_shared, sh_gate=_np(inp, "sh_gate"),
                       sh_up=_np(inp, "sh_up"), sh_down=_np(inp, "sh_down"), act_mode=act_mode,
                       g1=g1, g2=g2)


def _route(orc, cfg, inp):
    if cfg.scoring == synth.SCORE_HASH:
        return orc.route(T=cfg.T, E=cfg.E, k=cfg.k, scoring=2, scaling=cfg.scaling,
                         tid2eid=inp["tid2eid"].numpy(), token_ids=inp["token_ids"].numpy(),
                         vocab=cfg.vocab)
    return orc.route(T=cfg.T, E=cfg.E, k=cfg.k, scoring=cfg.scoring, renorm=cfg.renorm,
                     scaling=cfg.scaling, x_bf16=synth.bf16_bits(inp["x"]),
                     w_router_bf16=synth.bf16_bits(inp["w_router"]),
                     bias=None if "bias" not in inp else inp["bias"].numpy())


@pytest.mark.parametrize("act_mode", [0, 1])
def test_tiny_pairwise_equals_dense_mixture(orc, act_mode):
    cfg = synth.CONFIGS["tiny"]
    inp = synth.make_inputs(cfg, seed=0)
    r = _route(orc, cfg, inp)
    out = _oracle_ffn(orc, cfg, inp, r["ids"], r["w"], act_mode)
    ref = _dense_mixture(orc, cfg, inp, r["ids"], r["w"], act_mode)
    assert np.max(np.abs(out - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))
    assert np.max(np.abs(out)) > 0.01  # non-trivial output


def test_sigmoid_mxfp4_mixed_formats_dense(orc):
    cfg = synth.MoeConfig("mix", T=5, H=256, I=128, E=6, k=3, scoring=synth.SCORE_SIGMOID,
                          scaling=2.5, I_shared=256, fmt=synth.FMT_MXFP4, shared_fmt=synth.FMT_NVFP4)
    inp = synth.make_inputs(cfg, seed=3)
    r = _route(orc, cfg, inp)
    out = _oracle_ffn(orc, cfg, inp, r["ids"], r["w"])
    ref = _dense_mixture(orc, cfg, inp, r["ids"], r["w"])
    assert np.max(np.abs(out - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def test_all_experts_selected_is_full_softmax_mixture(orc):
    # special case: top_k == E with softmax routing reduces to the full softmax mixture
    cfg = synth.MoeConfig("full", T=3, H=128, I=128, E=4, k=4, scoring=synth.SCORE_SOFTMAX)
    inp = synth.make_inputs(cfg, seed=4)
    r = _route(orc, cfg, inp)
    l = r["logits"]
    p = np.exp(l - l.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    dense_ids = np.tile(np.arange(4, dtype=np.int32), (3, 1))
    out = _oracle_ffn(orc, cfg, inp, r["ids"], r["w"])
    ref = _oracle_ffn(orc, cfg, inp, dense_ids, p)
    assert np.max(np.abs(out - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_dropped_pairs_contribute_nothing(orc):
    cfg = synth.CONFIGS["tiny"]
    inp = synth.make_inputs(cfg, seed=1)
    r = _route(orc, cfg, inp)
    ids = r["ids"].copy()
    ids[1, 0] = -1
    out = _oracle_ffn(orc, cfg, inp, ids, r["w"])
    ref = _dense_mixture(orc, cfg, inp, ids, r["w"])
    assert np.max(np.abs(out - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def test_linearity_in_routing_weight(orc):
    # out depends linearly on each routing weight (the weighted sum of the block)
    cfg = synth.MoeConfig("lin", T=2, H=128, I=128, E=4, k=2, scoring=synth.SCORE_SOFTMAX)
    inp = synth.make_inputs(cfg, seed=9)
    r = _route(orc, cfg, inp)
    w2 = r["w"].copy()
    w2[0, 1] *= 3.0
    a = _oracle_ffn(orc, cfg, inp, r["ids"], r["w"])
    b = _oracle_ffn(orc, cfg, inp, r["ids"], w2)
    single = r["w"].copy() * 0
    single[0, 1] = r["w"][0, 1]
    c = _oracle_ffn(orc, cfg, inp, r["ids"], single)
    assert np.allclose(b - a, 2.0 * c, rtol=0, atol=1e-12)


@pytest.mark.parametrize("act_mode", [0, 1])
def test_zero_computation_experts_add_the_input(orc, act_mode):
    """Ids in [E, E + Z) are zero-computation experts (moe/mod.rs, the `moe_zero_expert_add`
    handle and `zero_accum_dev` field doc): each adds w * x, x the bf16 token."""
    cfg = synth.CONFIGS["tiny"]
    inp = synth.make_inputs(cfg, seed=4)
    rng = np.random.default_rng(9)
    Z = 3
    ids = np.stack([rng.permutation(cfg.E + Z)[:cfg.k] for _ in range(cfg.T)]).astype(np.int32)
    ids[0] = [cfg.E, cfg.E + 2]          # a token routed to zero experts only
    ids[1, 0] = 1                        # and one with a real expert first
    w = rng.uniform(0.1, 1.0, (cfg.T, cfg.k))
    got = orc.moe_ffn(T=cfg.T, E=cfg.E, H=cfg.H, I=cfg.I, k=cfg.k, gate=_np(inp, "gate"),
                      up=_np(inp, "up"), down=_np(inp, "down"), x_bf16=synth.bf16_bits(inp["x"]),
                      ids=ids, w=w, sh_I=cfg.I_shared, sh_gate=_np(inp, "sh_gate"),
                      sh_up=_np(inp, "sh_up"), sh_down=_np(inp, "sh_down"), act_mode=act_mode,
                      zero_experts=Z)
    real = np.where(ids < cfg.E, ids, -1)
    want = _dense_mixture(orc, cfg, inp, real, w, act_mode=act_mode)
    x = inp["x"].float().double().numpy()
    zw = np.where(ids >= cfg.E, w, 0.0).sum(1, keepdims=True)
    want += zw * x
    assert np.allclose(got, want, rtol=1e-9, atol=1e-12)
    # ids at or beyond E + Z are still dropped
    ids2 = ids.copy()
    ids2[2, 0] = cfg.E + Z
    got2 = orc.moe_ffn(T=cfg.T, E=cfg.E, H=cfg.H, I=cfg.I, k=cfg.k, gate=_np(inp, "gate"),
                       up=_np(inp, "up"), down=_np(inp, "down"), x_bf16=synth.bf16_bits(inp["x"]),
                       ids=ids2, w=w, sh_I=cfg.I_shared, sh_gate=_np(inp, "sh_gate"),
                       sh_up=_np(inp, "sh_up"), sh_down=_np(inp, "sh_down"), act_mode=act_mode,
                       zero_experts=Z)
    real2 = np.where(ids2 < cfg.E, ids2, -1)
    zw2 = np.where((ids2 >= cfg.E) & (ids2 < cfg.E + Z), w, 0.0).sum(1, keepdims=True)
    want2 = _dense_mixture(orc, cfg, inp, real2, w, act_mode=act_mode) + zw2 * x
    assert np.allclose(got2, want2, rtol=1e-9, atol=1e-12)
