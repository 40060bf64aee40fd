"""Helpers for the GPU-vs-oracle parity tests (test infrastructure).

Tolerances (stated by the block's acceptance rule): expert ids bit-exact; routing weights
within 1e-6 * routed_scaling; outputs max|gpu - ref| <= 1e-2 * max|ref| + 1e-3.  Inputs
whose top-(k+1) selection scores come closer than 1e-3 are redrawn (token by token) so that
no near-tie can flip an id.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from block_quantized_moe_router_gb300 import synth

GAP = 1e-3
W_TOL = 1e-6


def oracle_route(cfg, inp):
    Er = cfg.E + cfg.zero_experts
    if cfg.scoring == synth.SCORE_HASH:
        return oracle.route(T=cfg.T, E=Er, k=cfg.k, scoring=2, scaling=cfg.scaling,
                            tid2eid=inp["tid2eid"].numpy(), token_ids=inp["token_ids"].numpy(),
                            vocab=cfg.vocab)
    return oracle.route(T=cfg.T, E=Er, k=cfg.k, scoring=cfg.scoring, renorm=cfg.renorm,
                        scaling=cfg.scaling, x_bf16=synth.bf16_bits(inp["x"]),
                        w_router_bf16=synth.bf16_bits(inp["w_router"]),
                        bias=None if "bias" not in inp else inp["bias"].numpy())


def gap_violations(cfg, score):
    """Tokens whose k+1 best selection scores have an adjacent gap below GAP."""
    k = min(cfg.k + 1, cfg.E)
    top = -np.sort(-score, axis=1)[:, :k]
    gaps = top[:, :-1] - top[:, 1:]
    return [int(t) for t in np.nonzero((gaps < GAP).any(1))[0]]


def gap_safe_resample(cfg, seed, max_rounds=20):
    """Redraw counters that make every token's top-(k+1) scores at least GAP apart."""
    resample = {}
    if cfg.scoring == synth.SCORE_HASH:
        return resample
    for _ in range(max_rounds):
        inp = synth.make_inputs(cfg, seed=seed, resample=resample, with_weights=False)
        bad = gap_violations(cfg, oracle_route(cfg, inp)["score"])
        if not bad:
            return resample
        for t in bad:
            resample[t] = resample.get(t, 0) + 1
    raise RuntimeError("could not separate top-K scores")


def make_case(cfg, seed=0, device="cuda"):
    res = gap_safe_resample(cfg, seed)
    inp = synth.make_inputs(cfg, seed=seed, device=device, resample=res)
    return inp, res


def oracle_ffn(cfg, inp, ids, w, tokens=None):
    """Oracle output for the listed tokens (all when None), fp64 [len(tokens), H]."""
    x = inp["x"]
    if tokens is not None:
        x = x[tokens]
        ids = ids[tokens]
        w = w[tokens]
    npj = lambda key: synth.to_numpy_proj(inp.get(key))
    return oracle.moe_ffn(T=x.shape[0], E=cfg.E, H=cfg.H, I=cfg.I, k=cfg.k, gate=npj("gate"),
                          up=npj("up"), down=npj("down"), x_bf16=synth.bf16_bits(x), ids=ids, w=w,
                          sh_I=cfg.I_shared, sh_gate=npj("sh_gate"), sh_up=npj("sh_up"),
                          sh_down=npj("sh_down"), act_mode=cfg.act, zero_experts=cfg.zero_experts)


def assert_close(gpu: torch.Tensor, ref: np.ndarray, what: str = "out"):
    g = gpu.double().cpu().numpy()
    err = np.abs(g - ref)
    tol = 1e-2 * np.max(np.abs(ref)) + 1e-3
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU values"
    assert err.max() <= tol, f"{what}: max|gpu-ref| {err.max():.3e} > tol {tol:.3e}"
    rel_rms = np.sqrt(np.mean((g - ref) ** 2)) / max(np.sqrt(np.mean(ref ** 2)), 1e-30)
    assert rel_rms < 1e-2, f"{what}: relative RMS error {rel_rms:.3e}"
    return float(err.max()), float(rel_rms)


def assert_routing(cfg, ref, ids, w, gpu_logits=None, inp=None):
    """Ids bit-exact against the fp64 route.  Weights within W_TOL * routed_scaling of the
    oracle's weights -- computed from the GPU's own fp32 logits when those are given, so that
    the check measures the top-K arithmetic and not the fp32 rounding of a long router dot
    product (which the logits check bounds separately)."""
    ids = ids.cpu().numpy()
    w = w.cpu().numpy().astype(np.float64)
    assert np.array_equal(ids, ref["ids"]), "expert ids differ"
    ref_w = ref["w"]
    if gpu_logits is not None and cfg.scoring != synth.SCORE_HASH:
        lg = gpu_logits.float().cpu().numpy()
        r2 = oracle.route(T=cfg.T, E=cfg.E + cfg.zero_experts, k=cfg.k, scoring=cfg.scoring,
                          renorm=cfg.renorm,
                          scaling=cfg.scaling, logits_in=lg,
                          bias=None if inp is None or "bias" not in inp else inp["bias"].numpy())
        assert np.array_equal(r2["ids"], ref["ids"]), "ids from the GPU logits differ"
        ref_w = r2["w"]
    assert np.max(np.abs(w - ref_w)) <= W_TOL * max(cfg.scaling, 1.0), "routing weights differ"
