"""GPU parity of moe_forward: route + expert FFN in one call through the C ABI.

For a few tokens (T <= 8, T * top_k <= 64, bf16 activations) the whole block -- router GEMV,
top-K (or the hash lookup), gate+up, SiLU * up, down, top-K weighted sum and shared expert --
runs as one persistent launch (the single-launch decode structure of the spark_model MoE
module doc, moe/mod.rs, with the gate fused into the top-K).  Larger batches take moe_route then
moe_ffn_forward.  Ids are bit-exact against the fp64 oracle on gap-safe inputs; weights are
checked against the oracle's top-K of the GPU's own fp32 logits; outputs within
max|gpu - ref| <= 1e-2 * max|ref| + 1e-3.
"""
import dataclasses
import time

import numpy as np
import pytest
import torch

import parity
from block_quantized_moe_router_gb300 import capi, synth
from block_quantized_moe_router_gb300.layer import MoeLayer

pytestmark = pytest.mark.gpu

S = synth
CASES = {
    "tiny": S.CONFIGS["tiny"],
    # H / 128 = 3 K-steps: five of the eight warps have no gate+up work
    "ragged": S.MoeConfig("fw_ragged", T=7, H=384, I=256, E=10, k=3, scoring=S.SCORE_SOFTMAX,
                          I_shared=384),
    "sigmoid_mx": S.MoeConfig("fw_sigmoid_mx", T=5, H=2304, I=384, E=12, k=4,
                              scoring=S.SCORE_SIGMOID, scaling=2.5, I_shared=128,
                              fmt=S.FMT_MXFP4, shared_fmt=S.FMT_NVFP4),
    # 64 routed pairs: the largest dispatch the single launch takes
    "max_pairs": S.MoeConfig("fw_max_pairs", T=8, H=256, I=128, E=40, k=8,
                             scoring=S.SCORE_SIGMOID, scaling=1.5, I_shared=256,
                             fmt=S.FMT_NVFP4, shared_fmt=S.FMT_MXFP4),
    "sqrtsoftplus": S.MoeConfig("fw_sqrtsoftplus", T=3, H=512, I=256, E=24, k=5,
                                scoring=S.SCORE_SQRTSOFTPLUS, scaling=1.5, I_shared=256),
    "hash": S.MoeConfig("fw_hash", T=6, H=256, I=256, E=16, k=4, scoring=S.SCORE_HASH,
                        I_shared=128, fmt=S.FMT_MXFP4, vocab=50),
    "t1_no_renorm": S.MoeConfig("fw_t1", T=1, H=512, I=128, E=16, k=4, scoring=S.SCORE_SOFTMAX,
                                renorm=False),
    # one token with 32-row gate+up tasks (enough of them for two per CTA), MXFP4 routed
    # experts and an NVFP4 shared expert
    "t1_wide": S.MoeConfig("fw_t1_wide", T=1, H=768, I=2048, E=16, k=8, scoring=S.SCORE_SIGMOID,
                           scaling=2.5, I_shared=1024, fmt=S.FMT_MXFP4, shared_fmt=S.FMT_NVFP4),
    "t1_zero_hash": S.MoeConfig("fw_t1_zero_hash", T=1, H=256, I=384, E=12, k=4,
                                scoring=S.SCORE_HASH, I_shared=128, vocab=40, zero_experts=2),
    "many_experts": S.MoeConfig("fw_many_e", T=2, H=512, I=256, E=512, k=8,
                                scoring=S.SCORE_SOFTMAX),
    # softmax + bias routing over real and zero-computation experts (ids >= E add w * x)
    "zero_softmax_bias": S.MoeConfig("fw_zero_sb", T=5, H=512, I=256, E=12, k=4,
                                     scoring=S.SCORE_SOFTMAX_BIAS, renorm=False, scaling=1.5,
                                     I_shared=128, zero_experts=4),
    "zero_softmax_bias_renorm": S.MoeConfig("fw_zero_sbr", T=8, H=256, I=128, E=20, k=6,
                                            scoring=S.SCORE_SOFTMAX_BIAS, zero_experts=6),
    "zero_hash": S.MoeConfig("fw_zero_hash", T=6, H=256, I=256, E=16, k=4, scoring=S.SCORE_HASH,
                             I_shared=128, fmt=S.FMT_MXFP4, vocab=50, zero_experts=3),
    # hash-table ids weighted by the router's sqrt(softplus) scores: the router GEMV still runs
    # in the single launch, the table replaces the top-K
    "hash_sqrt": S.MoeConfig("fw_hash_sqrt", T=6, H=512, I=256, E=16, k=4,
                             scoring=S.SCORE_HASH_SQRTSOFTPLUS, scaling=1.5, I_shared=128,
                             fmt=S.FMT_MXFP4, vocab=50),
    "t1_hash_sqrt": S.MoeConfig("fw_t1_hash_sqrt", T=1, H=256, I=384, E=12, k=6,
                                scoring=S.SCORE_HASH_SQRTSOFTPLUS, renorm=False, vocab=40),
    "fallback_hash_sqrt_tc": S.MoeConfig("fw_hash_sqrt_tc", T=40, H=512, I=256, E=16, k=4,
                                         scoring=S.SCORE_HASH_SQRTSOFTPLUS, scaling=2.0,
                                         I_shared=256, act=S.ACT_NVFP4, vocab=64),
    # the largest top_k (32): one token's 32 picks built by the top-K warp, 64 pairs of two
    # tokens through the general dispatch, then the generic and tensor-core paths
    "max_topk_t1": S.MoeConfig("fw_max_topk_t1", T=1, H=256, I=128, E=64, k=32,
                               scoring=S.SCORE_SIGMOID, scaling=2.0, I_shared=128),
    "max_topk_t2": S.MoeConfig("fw_max_topk_t2", T=2, H=256, I=256, E=48, k=32,
                               scoring=S.SCORE_SOFTMAX),
    # (softmax selection at H 1024: logits spread enough for every token's top 33 to stay
    # 1e-3 apart, which sigmoid scores over 64 experts do not)
    "max_topk_generic": S.MoeConfig("fw_max_topk_generic", T=12, H=1024, I=128, E=64, k=32,
                                    scoring=S.SCORE_SOFTMAX, scaling=2.0, I_shared=128),
    "max_topk_tc": S.MoeConfig("fw_max_topk_tc", T=40, H=1024, I=256, E=64, k=32,
                               scoring=S.SCORE_SOFTMAX, I_shared=256, act=S.ACT_NVFP4),
    # the widest hidden size the single launch takes (H 8192: the router phase's chunk bound,
    # four 16-row output tiles per CTA)
    "max_h_t1": S.MoeConfig("fw_max_h_t1", T=1, H=8192, I=256, E=16, k=4,
                            scoring=S.SCORE_SOFTMAX),
    "max_h_t8": S.MoeConfig("fw_max_h_t8", T=8, H=8192, I=128, E=16, k=4,
                            scoring=S.SCORE_SIGMOID, scaling=2.0, I_shared=128),
    # a hidden size above that bound: a few tokens take moe_route + the generic expert GEMM
    "wide_h_generic": S.MoeConfig("fw_wide_h", T=3, H=8320, I=128, E=8, k=2,
                                  scoring=S.SCORE_SOFTMAX, I_shared=128),
    # more tokens: moe_route + moe_ffn_forward behind the same call
    "fallback_generic": S.MoeConfig("fw_generic", T=20, H=256, I=128, E=16, k=3,
                                    scoring=S.SCORE_SIGMOID, scaling=2.5, I_shared=128),
    "fallback_tc": S.MoeConfig("fw_tc", T=40, H=512, I=256, E=16, k=4, scoring=S.SCORE_SIGMOID,
                               scaling=2.5, I_shared=256, act=S.ACT_NVFP4),
    "fallback_generic_zero": S.MoeConfig("fw_generic_zero", T=20, H=256, I=128, E=12, k=3,
                                         scoring=S.SCORE_SOFTMAX_BIAS, I_shared=128,
                                         zero_experts=4),
    "fallback_tc_zero": S.MoeConfig("fw_tc_zero", T=40, H=512, I=256, E=16, k=4,
                                    scoring=S.SCORE_SOFTMAX_BIAS, renorm=False, scaling=2.0,
                                    I_shared=256, act=S.ACT_NVFP4, zero_experts=4),
}


def _forward(layer, inp, logits_in=None):
    x = inp["x"].cuda()
    tok = inp["token_ids"].cuda() if "token_ids" in inp else None
    out, ids, w, logits = layer.forward(x, token_ids=tok, logits_in=logits_in)
    torch.cuda.synchronize()
    return out, ids, w, logits


def _check(cfg, inp, ref_r, out, ids, w, logits, status, tokens=None):
    assert status == 0
    parity.assert_routing(cfg, ref_r, ids, w, gpu_logits=logits, inp=inp)
    if logits is not None:
        ref_l = ref_r["logits"]
        rel = np.abs(logits.double().cpu().numpy() - ref_l).max() / np.abs(ref_l).max()
        assert rel < 1e-4, f"router logits off by {rel:.2e} (relative)"
    ref = parity.oracle_ffn(cfg, inp, ref_r["ids"], ref_r["w"], tokens=tokens)
    parity.assert_close(out if tokens is None else out[tokens], ref, cfg.name)


@pytest.mark.parametrize("name", list(CASES))
def test_forward_small(cuda_lib, name):
    cfg = CASES[name]
    inp, _ = parity.make_case(cfg, seed=3, device="cpu")
    ref_r = parity.oracle_route(cfg, inp)
    layer = MoeLayer.from_inputs(inp)
    out, ids, w, logits = _forward(layer, inp)
    _check(cfg, inp, ref_r, out, ids, w, logits, int(layer.status.item()))
    layer.close()


@pytest.mark.parametrize("name", ["dec1", "dec8"])
def test_forward_full_size(cuda_lib, name):
    cfg = S.CONFIGS[name]
    inp, _ = parity.make_case(cfg, seed=0, device="cuda")
    ref_r = parity.oracle_route(cfg, inp)
    layer = MoeLayer.from_inputs(inp)
    out, ids, w, logits = _forward(layer, inp)
    _check(cfg, inp, ref_r, out, ids, w, logits, int(layer.status.item()))
    layer.close()


def test_forward_logits_in(cuda_lib):
    cfg = CASES["sigmoid_mx"]
    inp, _ = parity.make_case(cfg, seed=4, device="cpu")
    ref_r = parity.oracle_route(cfg, inp)
    layer = MoeLayer.from_inputs(inp)
    lg = torch.from_numpy(ref_r["logits"].astype(np.float32)).cuda()
    out, ids, w, logits = _forward(layer, inp, logits_in=lg)
    assert logits is None
    parity.assert_routing(cfg, ref_r, ids, w, gpu_logits=lg, inp=inp)
    parity.assert_close(out, parity.oracle_ffn(cfg, inp, ref_r["ids"], ref_r["w"]), "logits_in")
    layer.close()


def test_forward_repeat_and_graph_replay(cuda_lib):
    """Back-to-back launches and CUDA-graph replays on one handle give identical results (the
    device barrier counter carries over from launch to launch)."""
    cfg = CASES["ragged"]
    inp, _ = parity.make_case(cfg, seed=5, device="cpu")
    layer = MoeLayer.from_inputs(inp)
    x = inp["x"].cuda()
    out0, ids0, w0, _ = layer.forward(x)
    outs = [layer.forward(x)[0] for _ in range(5)]
    st = torch.cuda.Stream()
    o = torch.empty_like(out0)
    ids = torch.empty_like(ids0)
    w = torch.empty_like(w0)
    lg = torch.empty((cfg.T, cfg.E), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(st):
        layer.forward(x, out=o, topk_ids=ids, topk_w=w, logits_out=lg)
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            layer.forward(x, out=o, topk_ids=ids, topk_w=w, logits_out=lg)
        o.zero_()
        for _ in range(4):
            g.replay()
    torch.cuda.synchronize()
    for r in outs + [o]:
        assert torch.equal(r, out0)
    assert torch.equal(ids, ids0) and torch.equal(w, w0)
    assert int(layer.status.item()) == 0
    layer.close()


def test_forward_dropped_pairs(cuda_lib):
    cfg = CASES["hash"]
    inp, _ = parity.make_case(cfg, seed=2, device="cpu")
    tab = inp["tid2eid"].clone()
    tok = inp["token_ids"]
    tab[int(tok[1]), 2] = 77     # an id outside [0, E): that pair is dropped
    inp["tid2eid"] = tab
    bad_tok = inp["token_ids"].clone()
    ref_r = parity.oracle_route(cfg, inp)
    layer = MoeLayer.from_inputs(inp)
    out, ids, w, _ = _forward(layer, inp)
    assert int(layer.status.item()) == capi.MOE_DEV_BAD_EXPERT_ID
    parity.assert_routing(cfg, ref_r, ids, w)
    parity.assert_close(out, parity.oracle_ffn(cfg, inp, ref_r["ids"], ref_r["w"]), "dropped")
    # a token id outside the vocabulary drops all of that token's pairs
    bad_tok[0] = cfg.vocab + 5
    inp2 = dict(inp, token_ids=bad_tok)
    ref2 = parity.oracle_route(cfg, inp2)
    layer.status.zero_()
    out2, ids2, w2, _ = _forward(layer, inp2)
    assert int(layer.status.item()) & capi.MOE_DEV_BAD_TOKEN_ID
    parity.assert_routing(cfg, ref2, ids2, w2)
    parity.assert_close(out2, parity.oracle_ffn(cfg, inp2, ref2["ids"], ref2["w"]), "bad token")
    layer.close()


def test_forward_zero_tokens_and_arg_checks(cuda_lib):
    cfg = CASES["tiny"]
    inp, _ = parity.make_case(cfg, seed=0, device="cpu")
    layer = MoeLayer.from_inputs(inp)
    x0 = torch.zeros((0, cfg.H), dtype=torch.bfloat16, device="cuda")
    out0, _, _, _ = layer.forward(x0)
    torch.cuda.synchronize()
    assert out0.shape == (0, cfg.H)
    # a routing descriptor that does not match the weights handle is refused before any launch
    x = inp["x"].cuda()
    d = capi.route_desc(T=cfg.T, E=cfg.E + 1, H=cfg.H, top_k=cfg.k, scoring=cfg.scoring,
                        renormalize=True, routed_scaling=1.0, w_router=layer.w_router)
    with pytest.raises(capi.MoeError) as ei:
        capi.moe_forward(layer.handle, d, capi.MOE_ACT_BF16, 1.0, 1.0, x,
                         torch.empty((cfg.T, cfg.k), dtype=torch.int32, device="cuda"),
                         torch.empty((cfg.T, cfg.k), device="cuda"),
                         torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device="cuda"),
                         layer.workspace(cfg.T),
                         logits_out=torch.empty((cfg.T, cfg.E + 1), device="cuda"))
    assert ei.value.status == capi.MOE_ERR_INVALID_ARG
    layer.close()


HOST_CASES = ["t1_no_renorm", "t1_zero_hash", "max_pairs", "hash_sqrt", "fallback_generic",
              "fallback_tc", "fallback_hash_sqrt_tc"]


@pytest.mark.parametrize("name", HOST_CASES)
def test_forward_host_buffers(cuda_lib, name):
    """moe_forward_host (host buffers in and out, the copies enqueued with the forward) gives
    the oracle's routing and output, and exactly what moe_forward gives on device buffers;
    two slots of pinned buffers used in turn with inputs that differ stay separate."""
    cfg = CASES[name]
    inp, _ = parity.make_case(cfg, seed=7, device="cpu")
    inp2, _ = parity.make_case(cfg, seed=8, device="cpu")
    layer = MoeLayer.from_inputs(inp)
    dev = []
    for case in (inp, inp2):
        out, ids, w, _ = _forward(layer, case)
        dev.append((out.cpu(), ids.cpu(), w.cpu()))
    hash_kind = cfg.scoring in (S.SCORE_HASH, S.SCORE_HASH_SQRTSOFTPLUS)
    slots = []
    for case in (inp, inp2):
        slots.append(dict(
            x=case["x"].to(torch.bfloat16).contiguous().pin_memory(),
            tok=case["token_ids"].contiguous().pin_memory() if hash_kind else None,
            out=torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory(),
            ids=torch.empty((cfg.T, cfg.k), dtype=torch.int32).pin_memory(),
            w=torch.empty((cfg.T, cfg.k), dtype=torch.float32).pin_memory()))
    st = torch.cuda.Stream()
    for _ in range(2):
        for sl in slots:
            layer.forward_host(sl["x"], sl["out"], token_ids_host=sl["tok"],
                               topk_ids_host=sl["ids"], topk_w_host=sl["w"], stream=st)
    st.synchronize()
    assert int(layer.status.item()) == 0
    for sl, (out, ids, w) in zip(slots, dev):
        assert torch.equal(sl["out"], out) and torch.equal(sl["ids"], ids) and torch.equal(sl["w"], w)
    ref_r = parity.oracle_route(cfg, inp)
    parity.assert_routing(cfg, ref_r, slots[0]["ids"], slots[0]["w"], inp=inp)
    parity.assert_close(slots[0]["out"], parity.oracle_ffn(cfg, inp, ref_r["ids"], ref_r["w"]),
                        cfg.name + " host")
    # pageable host memory and no ids / weights requested: same output
    out_p = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16)
    layer.forward_host(inp["x"].to(torch.bfloat16).contiguous(), out_p,
                       token_ids_host=inp["token_ids"].contiguous() if hash_kind else None)
    torch.cuda.synchronize()
    assert torch.equal(out_p, dev[0][0])
    layer.close()


def test_forward_host_arg_checks(cuda_lib):
    cfg = CASES["tiny"]
    inp, _ = parity.make_case(cfg, seed=0, device="cpu")
    layer = MoeLayer.from_inputs(inp)
    x = inp["x"].to(torch.bfloat16).contiguous()
    out = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16)
    d = capi.route_desc(T=cfg.T, E=cfg.E, H=cfg.H, top_k=cfg.k, scoring=cfg.scoring,
                        renormalize=True, routed_scaling=1.0, w_router=layer.w_router)
    need = capi.moe_workspace_size_host(layer.desc, cfg.T, capi.MOE_ACT_BF16)
    assert need >= capi.moe_workspace_size(layer.desc, cfg.T, capi.MOE_ACT_BF16) + 2 * cfg.T * cfg.H * 2
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(capi.MoeError) as ei:
        capi.moe_forward_host(layer.handle, d, capi.MOE_ACT_BF16, 1.0, 1.0, x, out, ws)
    assert ei.value.status == capi.MOE_ERR_WORKSPACE
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    nor = capi.route_desc(T=cfg.T, E=cfg.E, H=cfg.H, top_k=cfg.k, scoring=cfg.scoring,
                          renormalize=True, routed_scaling=1.0)
    with pytest.raises(capi.MoeError) as ei:  # the router must run inside the call
        capi.moe_forward_host(layer.handle, nor, capi.MOE_ACT_BF16, 1.0, 1.0, x, out, ws)
    assert ei.value.status == capi.MOE_ERR_INVALID_ARG
    with pytest.raises(ValueError):  # device tensors are not host buffers
        capi.moe_forward_host(layer.handle, d, capi.MOE_ACT_BF16, 1.0, 1.0, x.cuda(), out, ws)
    # no tokens: a valid no-op
    d0 = capi.route_desc(T=0, E=cfg.E, H=cfg.H, top_k=cfg.k, scoring=cfg.scoring,
                         renormalize=True, routed_scaling=1.0, w_router=layer.w_router)
    capi.moe_forward_host(layer.handle, d0, capi.MOE_ACT_BF16, 1.0, 1.0,
                          torch.empty((0, cfg.H), dtype=torch.bfloat16),
                          torch.empty((0, cfg.H), dtype=torch.bfloat16), ws)
    torch.cuda.synchronize()
    layer.close()


GUARD = 4096


def _guarded(nbytes):
    """A device buffer of nbytes between two 4 KB guard regions filled with 0xA5."""
    buf = torch.full((2 * GUARD + nbytes,), 0xA5, dtype=torch.uint8, device="cuda")
    return buf, buf[GUARD:GUARD + nbytes]


@pytest.mark.parametrize("name", ["t1_zero_hash", "t1_wide", "max_pairs", "fallback_generic_zero",
                                  "fallback_tc_zero", "fallback_hash_sqrt_tc"])
def test_writes_stay_inside_their_buffers(cuda_lib, name):
    """Every kernel of the call writes only inside the buffers it is given: the output, the ids,
    the weights, the router logits and the workspace (sized exactly by moe_workspace_size) each
    sit between guard regions that must come back untouched."""
    cfg = CASES[name]
    inp, _ = parity.make_case(cfg, seed=9, device="cpu")
    layer = MoeLayer.from_inputs(inp)
    T, Er = cfg.T, cfg.E + cfg.zero_experts
    hash_only = cfg.scoring == S.SCORE_HASH
    parts = {"out": (T * cfg.H * 2, torch.bfloat16, (T, cfg.H)),
             "ids": (T * cfg.k * 4, torch.int32, (T, cfg.k)),
             "w": (T * cfg.k * 4, torch.float32, (T, cfg.k)),
             "ws": (capi.moe_workspace_size(layer.desc, T, cfg.act), torch.uint8, None)}
    if not hash_only:
        parts["logits"] = (T * Er * 4, torch.float32, (T, Er))
    bufs, views = {}, {}
    for key, (nbytes, dtype, shape) in parts.items():
        bufs[key], raw = _guarded(nbytes)
        views[key] = raw if shape is None else raw.view(dtype).view(shape)
    tok = inp["token_ids"].cuda() if "token_ids" in inp else None
    d = capi.route_desc(T=T, E=cfg.E, H=cfg.H, top_k=cfg.k, scoring=cfg.scoring,
                        renormalize=cfg.renorm, routed_scaling=cfg.scaling, w_router=layer.w_router,
                        correction_bias=layer.correction_bias, tid2eid=layer.tid2eid,
                        vocab=0 if layer.tid2eid is None else layer.tid2eid.shape[0],
                        token_ids=tok, zero_experts=cfg.zero_experts)
    capi.moe_forward(layer.handle, d, cfg.act, 1.0, 1.0, inp["x"].cuda(), views["ids"], views["w"],
                     views["out"], views["ws"], logits_out=views.get("logits"),
                     dev_status=layer.status)
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    for key, buf in bufs.items():
        assert bool((buf[:GUARD] == 0xA5).all()), f"{key}: written before its start"
        assert bool((buf[GUARD + parts[key][0]:] == 0xA5).all()), f"{key}: written past its end"
    ref_r = parity.oracle_route(cfg, inp)
    parity.assert_close(views["out"], parity.oracle_ffn(cfg, inp, ref_r["ids"], ref_r["w"]), name)
    layer.close()


@pytest.mark.parametrize("name", ["ragged", "t1_no_renorm"])
def test_barrier_wait_runs_out(cuda_lib, name):
    """The few-token kernel's device-wide barrier waits are bounded.  With a 10 ms limit and
    the handle's barrier epoch moved one launch ahead (moe_skew_barrier), no barrier of the
    next launch can complete: the launch must return (well inside a second), set
    MOE_DEV_TIMEOUT, and leave the device usable -- a fresh handle then gives correct results.
    One token (its own kernel instantiation, the top-K warp building the dispatch) and several
    tokens."""
    cfg = CASES[name]
    inp, _ = parity.make_case(cfg, seed=6, device="cpu")
    layer = MoeLayer.from_inputs(inp)
    x = inp["x"].cuda()
    layer.forward(x)
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    capi.moe_set_wait_limit(layer.handle, 20_000_000)  # SM cycles: about 10 ms
    layer.forward(x)                                    # a short limit alone changes nothing
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    capi.moe_skew_barrier(layer.handle)
    t0 = time.perf_counter()
    layer.forward(x)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(layer.status.item()) & capi.MOE_DEV_TIMEOUT
    assert dt < 1.0, f"the timed-out launch took {dt:.3f} s"
    layer.close()
    ref_r = parity.oracle_route(cfg, inp)
    layer = MoeLayer.from_inputs(inp)
    out, ids, w, logits = _forward(layer, inp)
    _check(cfg, inp, ref_r, out, ids, w, logits, int(layer.status.item()))
    layer.close()
