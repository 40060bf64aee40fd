"""Helpers for the GPU-vs-oracle parity tests (test infrastructure).

Tolerances (stated by the block's acceptance rule): expert ids bit-exact; outputs
max|gpu - ref| <= 1e-2 * max|ref| + 1e-3.  Routing weights are checked twice:
  1. against the oracle's fp64 route (fp64 logits): |w_gpu - w_ref| <= 1e-6 * max(scaling, 1)
     + 2 * J * delta, where delta is the token's largest measured router-logit error
     |l_gpu - l_fp64| and J the sum over the token's logits of |d w / d l| at the fp64 route
     (a closed form per scoring kind, below) -- the first-order propagation of the fp32
     router GEMM's rounding into the weights, doubled to cover second-order terms;
  2. against the oracle's top-K recomputed from the GPU's own fp32 logits:
     |w_gpu - w| <= 1e-6 * max(scaling, 1) -- the top-K arithmetic alone.
Inputs whose top-(k+1) selection scores come closer than 1e-3 are redrawn (token by token) so
that no near-tie can flip an id.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from block_quantized_moe_router_gb300 import synth

GAP = 1e-3
W_TOL = 1e-6
HASH_KINDS = (synth.SCORE_HASH, synth.SCORE_HASH_SQRTSOFTPLUS)


def oracle_route(cfg, inp):
    Er = cfg.E + cfg.zero_experts
    if cfg.scoring == synth.SCORE_HASH:
        return oracle.route(T=cfg.T, E=Er, k=cfg.k, scoring=2, scaling=cfg.scaling,
                            tid2eid=inp["tid2eid"].numpy(), token_ids=inp["token_ids"].numpy(),
                            vocab=cfg.vocab)
    hash_kw = {}
    if cfg.scoring == synth.SCORE_HASH_SQRTSOFTPLUS:
        hash_kw = dict(tid2eid=inp["tid2eid"].cpu().numpy(),
                       token_ids=inp["token_ids"].cpu().numpy(), vocab=cfg.vocab)
    return oracle.route(T=cfg.T, E=Er, k=cfg.k, scoring=cfg.scoring, renorm=cfg.renorm,
                        scaling=cfg.scaling, x_bf16=synth.bf16_bits(inp["x"]),
                        w_router_bf16=synth.bf16_bits(inp["w_router"]),
                        bias=None if "bias" not in inp else inp["bias"].cpu().numpy(), **hash_kw)


def gap_violations(cfg, score):
    """Tokens whose k+1 best selection scores have an adjacent gap below GAP."""
    k = min(cfg.k + 1, cfg.E)
    top = -np.sort(-score, axis=1)[:, :k]
    gaps = top[:, :-1] - top[:, 1:]
    return [int(t) for t in np.nonzero((gaps < GAP).any(1))[0]]


def gap_safe_resample(cfg, seed, max_rounds=20):
    """Redraw counters that make every token's top-(k+1) scores at least GAP apart."""
    resample = {}
    if cfg.scoring in HASH_KINDS:  # the table selects: no score gap to keep
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


def _weight_sensitivity(cfg, ref):
    """J[t, j] = sum_i |d w_tj / d l_ti| at the fp64 route (ref: the oracle's route with its
    fp64 logits).  Closed forms: softmax-type weights w = c p_j / sum p (over the selected
    experts when renormalised, over all otherwise) give 2 c p~_j (1 - p~_j) with p~_j = w_j / c;
    score-type weights w = c s_j / S with s = f(l) give c (f'_j (S - s_j) + s_j sum_{i != j}
    f'_i) / S^2 (renormalised) or c f'_j; f = sigmoid (f' = f (1 - f)) or sqrt(softplus)
    (f' = sigmoid / (2 f)).  Plain hash weights do not depend on the logits."""
    T, k = ref["ids"].shape
    c = cfg.scaling
    if cfg.scoring == synth.SCORE_HASH:
        return np.zeros((T, k))
    if cfg.scoring in (synth.SCORE_SOFTMAX, synth.SCORE_SOFTMAX_BIAS):
        pt = ref["w"] / c
        return 2.0 * c * pt * (1.0 - pt)
    ids = ref["ids"]
    lg = np.take_along_axis(ref["logits"], np.maximum(ids, 0), axis=1)
    sig = 1.0 / (1.0 + np.exp(-lg))
    if cfg.scoring == synth.SCORE_SIGMOID:
        f, fp = sig, sig * (1.0 - sig)
    else:  # sqrt(softplus), also the score-weighted hash kind
        f = np.sqrt(np.log1p(np.exp(lg)))
        fp = sig / (2.0 * f)
    keep = ids >= 0
    f, fp = np.where(keep, f, 0.0), np.where(keep, fp, 0.0)
    if not cfg.renorm:
        return c * fp
    S = f.sum(1, keepdims=True)
    other = fp.sum(1, keepdims=True) - fp
    return c * (fp * (S - f) + f * other) / np.maximum(S, 1e-300) ** 2


def assert_routing(cfg, ref, ids, w, gpu_logits=None, inp=None):
    """Ids bit-exact against the fp64 route.  Weights (1) against the fp64 route within
    W_TOL * max(scaling, 1) + 2 J delta (module docstring), and (2) when the GPU's logits are
    given, against the oracle's top-K of those same fp32 logits within W_TOL * max(scaling, 1)."""
    ids = ids.cpu().numpy()
    w = w.cpu().numpy().astype(np.float64)
    assert np.array_equal(ids, ref["ids"]), "expert ids differ"
    base = W_TOL * max(cfg.scaling, 1.0)
    delta = np.zeros((ids.shape[0], 1))
    if gpu_logits is not None and ref.get("logits") is not None:
        lg = gpu_logits.double().cpu().numpy()
        delta = np.abs(lg - ref["logits"]).max(1, keepdims=True)
    bound = base + 2.0 * _weight_sensitivity(cfg, ref) * delta
    err = np.abs(w - ref["w"])
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), (f"routing weights differ from the fp64 route: |dw| "
                                  f"{err[worst]:.3e} > bound {bound[worst]:.3e} at {worst}")
    if gpu_logits is not None and cfg.scoring != synth.SCORE_HASH:
        lg = gpu_logits.float().cpu().numpy()
        hash_kw = {}
        if cfg.scoring == synth.SCORE_HASH_SQRTSOFTPLUS:
            hash_kw = dict(tid2eid=inp["tid2eid"].cpu().numpy(),
                           token_ids=inp["token_ids"].cpu().numpy(), vocab=cfg.vocab)
        r2 = oracle.route(T=cfg.T, E=cfg.E + cfg.zero_experts, k=cfg.k, scoring=cfg.scoring,
                          renorm=cfg.renorm,
                          scaling=cfg.scaling, logits_in=lg,
                          bias=None if inp is None or "bias" not in inp else inp["bias"].cpu().numpy(),
                          **hash_kw)
        assert np.array_equal(r2["ids"], ref["ids"]), "ids from the GPU logits differ"
        assert np.max(np.abs(w - r2["w"])) <= base, "routing weights differ (GPU logits)"
