"""End-to-end GPU parity of the MoE block through the C ABI (moe_route + moe_ffn_forward).

Expert FFN per pair -- gate+up, SiLU(gate)*up, down -- and the top-K weighted sum plus the
shared expert (spark_model MoE pages, moe/mod.rs module doc), over NVFP4 / MXFP4 weights
(moe/mod.rs, `experts_scale_kind` doc), with bf16 activations or NVFP4-quantized
activations (the FP4 x FP4 recipe, moe/mod.rs `moe_fused_gate_up_t_k64_fp4` doc).
Tolerance: max|gpu - ref| <= 1e-2 * max|ref| + 1e-3 and relative RMS error < 1e-2.
"""
import dataclasses

import numpy as np
import pytest
import torch

import parity
from block_quantized_moe_router_gb300 import capi, synth
from block_quantized_moe_router_gb300.layer import MoeLayer

pytestmark = pytest.mark.gpu

S = synth
SMALL = {
    "tiny": S.CONFIGS["tiny"],
    "tiny_a4": dataclasses.replace(S.CONFIGS["tiny"], name="tiny_a4", act=S.ACT_NVFP4),
    "ragged": S.MoeConfig("ragged", T=13, H=384, I=256, E=10, k=3, scoring=S.SCORE_SOFTMAX,
                          I_shared=128),
    "ragged_a4": S.MoeConfig("ragged_a4", T=13, H=384, I=256, E=10, k=3, scoring=S.SCORE_SOFTMAX,
                             I_shared=128, act=S.ACT_NVFP4),
    "mx_routed": S.MoeConfig("mx_routed", T=9, H=256, I=384, E=12, k=4, scoring=S.SCORE_SIGMOID,
                             scaling=2.5, I_shared=256, fmt=S.FMT_MXFP4, shared_fmt=S.FMT_NVFP4),
    "mx_shared": S.MoeConfig("mx_shared", T=11, H=256, I=128, E=6, k=2, scoring=S.SCORE_SOFTMAX,
                             I_shared=384, fmt=S.FMT_NVFP4, shared_fmt=S.FMT_MXFP4),
    "mx_all_a4": S.MoeConfig("mx_all_a4", T=40, H=512, I=256, E=16, k=4, scoring=S.SCORE_SIGMOID,
                             scaling=2.5, I_shared=256, fmt=S.FMT_MXFP4, shared_fmt=S.FMT_MXFP4,
                             act=S.ACT_NVFP4),
    "many_tokens": S.MoeConfig("many", T=100, H=256, I=256, E=8, k=2, scoring=S.SCORE_SOFTMAX,
                               I_shared=128),
    "hash_small": S.MoeConfig("hash_small", T=20, H=256, I=128, E=16, k=3, scoring=S.SCORE_HASH,
                              I_shared=128, fmt=S.FMT_MXFP4, vocab=100),
    # few-token path (T <= 8, bf16 activations): fused dispatch, split-K gate+up, down+combine
    "dec_ragged": S.MoeConfig("dec_ragged", T=7, H=384, I=256, E=10, k=3, scoring=S.SCORE_SOFTMAX,
                              I_shared=384),
    "dec_mx": S.MoeConfig("dec_mx", T=5, H=2304, I=384, E=12, k=4, scoring=S.SCORE_SIGMOID,
                          scaling=2.5, I_shared=128, fmt=S.FMT_MXFP4, shared_fmt=S.FMT_NVFP4),
    "dec_mx_shared": S.MoeConfig("dec_mx_shared", T=8, H=256, I=128, E=40, k=8,
                                 scoring=S.SCORE_SIGMOID, scaling=1.5, I_shared=256,
                                 fmt=S.FMT_NVFP4, shared_fmt=S.FMT_MXFP4),
    "dec_hash": S.MoeConfig("dec_hash", T=6, H=256, I=256, E=16, k=4, scoring=S.SCORE_HASH,
                            I_shared=128, fmt=S.FMT_MXFP4, vocab=50),
    "dec_t1": S.MoeConfig("dec_t1", T=1, H=512, I=128, E=16, k=4, scoring=S.SCORE_SOFTMAX,
                          renorm=False),
    # softmax + bias over real and zero-computation experts (routing kernel, then the given ids)
    "dec_zero": S.MoeConfig("dec_zero", T=6, H=256, I=128, E=10, k=3,
                            scoring=S.SCORE_SOFTMAX_BIAS, I_shared=128, zero_experts=3),
    # NVFP4 activations with 256-multiple shapes: tcgen05 block-scaled path
    "tc_small": S.MoeConfig("tc_small", T=40, H=512, I=256, E=16, k=4, scoring=S.SCORE_SIGMOID,
                            scaling=2.5, I_shared=256, act=S.ACT_NVFP4),
    "tc_multi_block": S.MoeConfig("tc_multi_block", T=300, H=768, I=512, E=4, k=2,
                                  scoring=S.SCORE_SOFTMAX, act=S.ACT_NVFP4),
    "tc_shared_wide": S.MoeConfig("tc_shared_wide", T=70, H=256, I=256, E=8, k=2,
                                  scoring=S.SCORE_SOFTMAX, I_shared=512, act=S.ACT_NVFP4),
    "tc_t1": S.MoeConfig("tc_t1", T=1, H=256, I=256, E=8, k=2, scoring=S.SCORE_SOFTMAX,
                         I_shared=256, act=S.ACT_NVFP4),
    # MXFP4 weights on the tensor-core path (E8M0 scales re-expressed as E4M3 powers of two)
    "tc_mx_routed": S.MoeConfig("tc_mx_routed", T=150, H=768, I=512, E=8, k=3,
                                scoring=S.SCORE_SQRTSOFTPLUS, I_shared=256, fmt=S.FMT_MXFP4,
                                shared_fmt=S.FMT_NVFP4, act=S.ACT_NVFP4),
    "tc_mx_hash": S.MoeConfig("tc_mx_hash", T=64, H=512, I=512, E=16, k=6, scoring=S.SCORE_HASH,
                              I_shared=512, fmt=S.FMT_MXFP4, shared_fmt=S.FMT_NVFP4, vocab=500,
                              act=S.ACT_NVFP4),
    # >= 512 routed rows per expert: each expert's weight tiles serve several row blocks
    "tc_many": S.MoeConfig("tc_many", T=1100, H=512, I=256, E=4, k=2, scoring=S.SCORE_SIGMOID,
                          scaling=2.5, I_shared=256, act=S.ACT_NVFP4),
    "tc_many_mx": S.MoeConfig("tc_many_mx", T=1040, H=768, I=512, E=4, k=2,
                             scoring=S.SCORE_SOFTMAX, I_shared=256, fmt=S.FMT_MXFP4,
                             shared_fmt=S.FMT_NVFP4, act=S.ACT_NVFP4),
    # the prefill recipe at reduced size, every row compared: Zipf-skewed counts (the head
    # experts capped at every token, 16 padded 128-row blocks; the tail a partial block each)
    "tc_zipf_all_rows": S.MoeConfig("tc_zipf_all_rows", T=2048, H=768, I=512, E=24, k=8,
                                    scoring=S.SCORE_SIGMOID, scaling=2.5, I_shared=256,
                                    act=S.ACT_NVFP4, zipf_s=1.1),
    # hash-table ids weighted by the router's sqrt(softplus) scores, on the bf16 many-token
    # path and on the tensor-core path
    "hash_sqrt": S.MoeConfig("hash_sqrt", T=20, H=256, I=128, E=16, k=3,
                             scoring=S.SCORE_HASH_SQRTSOFTPLUS, scaling=1.5, I_shared=128,
                             fmt=S.FMT_MXFP4, vocab=100),
    "hash_sqrt_tc": S.MoeConfig("hash_sqrt_tc", T=64, H=512, I=512, E=16, k=6,
                                scoring=S.SCORE_HASH_SQRTSOFTPLUS, I_shared=512,
                                fmt=S.FMT_MXFP4, shared_fmt=S.FMT_NVFP4, vocab=500,
                                act=S.ACT_NVFP4),
}


def _run(cfg, inp, with_logits=False):
    layer = MoeLayer.from_inputs(inp)
    x = inp["x"].cuda()
    tok = inp["token_ids"].cuda() if "token_ids" in inp else None
    ids, w, logits = layer.route(x, token_ids=tok)
    out = layer.ffn(x, ids, w)
    torch.cuda.synchronize()
    status = int(layer.status.item())
    layer.close()
    if with_logits:
        return ids, w, out, status, logits
    return ids, w, out, status


@pytest.mark.parametrize("name", list(SMALL))
def test_small_configs(cuda_lib, name):
    cfg = SMALL[name]
    inp, _ = parity.make_case(cfg, seed=1, device="cpu")
    ref_r = parity.oracle_route(cfg, inp)
    ids, w, out, status, logits = _run(cfg, inp, with_logits=True)
    assert status == 0
    parity.assert_routing(cfg, ref_r, ids, w, gpu_logits=logits, inp=inp)
    ref = parity.oracle_ffn(cfg, inp, ref_r["ids"], ref_r["w"])
    parity.assert_close(out, ref, name)


def covering_tokens(ids, E, per_expert=2, extra=(0, 1)):
    """Tokens such that every routed expert is compared: each expert's first and last token
    (in token order) and, for experts with many rows, per_expert more spread over its tokens;
    plus the `extra` tokens.  Sorted, unique."""
    pick = set(int(t) for t in extra)
    for e in range(E):
        toks = np.nonzero((ids == e).any(1))[0]
        if len(toks) == 0:
            continue
        pick.update([int(toks[0]), int(toks[-1])])
        if len(toks) > 256:
            pick.update(int(t) for t in toks[np.linspace(0, len(toks) - 1, per_expert + 2)[1:-1].astype(int)])
    return sorted(pick)


FULL = {
    "dec1": S.CONFIGS["dec1"],
    "dec8": S.CONFIGS["dec8"],
    "hash64": S.CONFIGS["hash64"],
    "pre4096": S.CONFIGS["pre4096"],
    "pre32768": S.CONFIGS["pre32768"],
}


def last_tokens(ids, E, head=16, extra=(0, 1)):
    """For the largest prefill: the last token of every routed expert (its ragged last 128-row
    block), the first token of the `head` experts with the most tokens, and the `extra` tokens.
    Sorted, unique."""
    pick = set(int(t) for t in extra)
    counts = np.array([(ids == e).any(1).sum() for e in range(E)])
    for e in range(E):
        toks = np.nonzero((ids == e).any(1))[0]
        if len(toks):
            pick.add(int(toks[-1]))
    for e in np.argsort(-counts)[:head]:
        toks = np.nonzero((ids == e).any(1))[0]
        if len(toks):
            pick.add(int(toks[0]))
    return sorted(pick)


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_configs(cuda_lib, name):
    """Full-size workloads: every token for the decode and hash workloads; for the 4096-token
    prefill the first and last token of every routed expert (a few hundred tokens) plus tokens
    spread over the Zipf head's rows; for the 32768-token prefill the last token of every routed
    expert and the first of the largest ones; all rows finite and nonzero."""
    cfg = FULL[name]
    inp, _ = parity.make_case(cfg, seed=0, device="cuda")
    ref_r = parity.oracle_route(cfg, inp)
    ids, w, out, status, logits = _run(cfg, inp, with_logits=True)
    assert status == 0
    parity.assert_routing(cfg, ref_r, ids, w, gpu_logits=logits, inp=inp)
    sample = None
    if cfg.T > 8192:
        sample = last_tokens(ref_r["ids"], cfg.E, extra=(0, 1, cfg.T - 1))
        routed = set(int(e) for e in np.unique(ref_r["ids"]) if 0 <= e < cfg.E)
        assert routed <= set(int(e) for e in np.unique(ref_r["ids"][sample]))  # every expert
    elif cfg.T > 64:
        sample = covering_tokens(ref_r["ids"], cfg.E, per_expert=6, extra=(0, 1, cfg.T - 1))
        assert len(sample) >= cfg.E  # (a few hundred tokens at 4096)
    ref = parity.oracle_ffn(cfg, inp, ref_r["ids"], ref_r["w"], tokens=sample)
    got = out if sample is None else out[sample]
    parity.assert_close(got, ref, name)
    # every output row is finite and the unsampled rows are not left untouched
    assert torch.isfinite(out.float()).all()
    assert (out.float().abs().amax(1) > 0).all()


def test_mxfp4_blocks_far_below_the_largest_scale(cuda_lib):
    """MXFP4 blocks far below their tensor's largest scale: the tensor-core path re-expresses
    E8M0 scales as E4M3 powers of two and flushes blocks more than 2^17 below the largest to
    zero; the few-token path's f16 scale flushes blocks more than 2^27 below.  Rows whose
    every block sits 18, 20 or 28 binades below the largest must still match the oracle (an
    element of a flushed block is below 6 * 2^-17 of the largest block's scale)."""
    cases = [SMALL["tc_mx_routed"],
             S.MoeConfig("mx_flush_dec", T=5, H=512, I=256, E=12, k=4, scoring=S.SCORE_SIGMOID,
                         scaling=2.5, I_shared=128, fmt=S.FMT_MXFP4, shared_fmt=S.FMT_NVFP4),
             S.MoeConfig("mx_flush_generic", T=24, H=256, I=256, E=12, k=4,
                         scoring=S.SCORE_SOFTMAX, fmt=S.FMT_MXFP4)]
    for cfg in cases:
        inp, _ = parity.make_case(cfg, seed=8, device="cpu")
        ref_r = parity.oracle_route(cfg, inp)
        e = int(ref_r["ids"][0, 0])  # an expert that is routed
        for key, drops in (("gate", (18, 20, 28)), ("up", (20, 28, 18)), ("down", (28, 18, 20))):
            sc = inp[key]["scales"].clone()
            bmax = int(sc[e].max())
            n = sc.shape[1]
            for i, d in enumerate(drops):
                rows = slice(i * n // 8, i * n // 8 + n // 16)
                sc[e, rows] = bmax - d
            inp[key] = dict(inp[key], scales=sc)
        ids, w, out, status = _run(cfg, inp)
        assert status == 0
        parity.assert_routing(cfg, ref_r, ids, w)
        parity.assert_close(out, parity.oracle_ffn(cfg, inp, ref_r["ids"], ref_r["w"]), cfg.name)


GIVEN = {
    "decode": S.MoeConfig("given_dec", T=6, H=256, I=128, E=16, k=3, scoring=S.SCORE_SOFTMAX,
                          I_shared=128, zero_experts=2),
    "generic": S.MoeConfig("given_generic", T=20, H=256, I=128, E=16, k=3,
                           scoring=S.SCORE_SOFTMAX, I_shared=128, zero_experts=2),
    "tc": S.MoeConfig("given_tc", T=40, H=512, I=256, E=16, k=3, scoring=S.SCORE_SOFTMAX,
                      I_shared=256, act=S.ACT_NVFP4, zero_experts=2),
}


@pytest.mark.parametrize("name", list(GIVEN))
def test_given_ids_out_of_range(cuda_lib, name):
    """moe_ffn_forward with caller ids: ids outside [-1] + [0, E + Z) are dropped and flagged
    with MOE_DEV_BAD_EXPERT_ID on every path (few-token, bf16 many-token, tensor cores); -1 is
    a silent drop; zero-computation ids add w * x."""
    cfg = GIVEN[name]
    inp, _ = parity.make_case(cfg, seed=7, device="cpu")
    ref_r = parity.oracle_route(cfg, inp)
    ids = ref_r["ids"].copy()
    w = ref_r["w"].astype(np.float32)
    ids[1, 0] = 99          # beyond E + Z
    ids[2, 1] = -5          # negative, not -1
    ids[3, 2] = -1          # the drop marker
    ids[4, 0] = cfg.E + 1   # a zero-computation expert
    layer = MoeLayer.from_inputs(inp)
    x = inp["x"].cuda()
    out = layer.ffn(x, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    assert int(layer.status.item()) == capi.MOE_DEV_BAD_EXPERT_ID
    layer.close()
    parity.assert_close(out, parity.oracle_ffn(cfg, inp, ids, w.astype(np.float64)), name)


DROP = {
    "generic": SMALL["hash_small"],
    "tc": S.MoeConfig("hash_tc", T=50, H=512, I=256, E=16, k=3, scoring=S.SCORE_HASH,
                      I_shared=256, vocab=100, act=S.ACT_NVFP4),
}


@pytest.mark.parametrize("name", list(DROP))
def test_dropped_pairs_and_zero_tokens(cuda_lib, name):
    cfg = DROP[name]
    inp, _ = parity.make_case(cfg, seed=2, device="cpu")
    tab = inp["tid2eid"].clone()
    tok = inp["token_ids"]
    tab[int(tok[3]), 1] = 99     # bad id: that pair is dropped
    inp["tid2eid"] = tab
    ref_r = parity.oracle_route(cfg, inp)
    ids, w, out, status = _run(cfg, inp)
    assert status == capi.MOE_DEV_BAD_EXPERT_ID
    parity.assert_routing(cfg, ref_r, ids, w)
    parity.assert_close(out, parity.oracle_ffn(cfg, inp, ref_r["ids"], ref_r["w"]), "dropped")
    # T == 0 is a no-op through both entry points
    layer = MoeLayer.from_inputs(inp)
    x0 = torch.zeros((0, cfg.H), dtype=torch.bfloat16, device="cuda")
    out0 = layer.ffn(x0, torch.zeros((0, cfg.k), dtype=torch.int32, device="cuda"),
                     torch.zeros((0, cfg.k), device="cuda"))
    torch.cuda.synchronize()
    assert out0.shape == (0, cfg.H)
    layer.close()


def test_quantizer_matches_oracle(cuda_lib):
    import oracle
    rng = np.random.default_rng(0)
    rows, K = 64, 512
    v = rng.standard_normal((rows, K)).astype(np.float32) * rng.uniform(1e-4, 300, (rows, 1)).astype(np.float32)
    v[3, :16] = 0.0                               # all-zero block
    v[4, :16] = [3, -1.5, 0.75, 0.25, 6, 5, -3.5, 0, 1.25, -2.5, 0.5, 1.75, -6, 2, 4, -0.1]
    xb = torch.from_numpy(v).to(torch.bfloat16)
    vb = xb.float().numpy()
    for g in (1.0, 0.25, 8.0):
        packed = torch.zeros((rows, K // 2), dtype=torch.uint8, device="cuda")
        scales = torch.zeros((rows, K // 16), dtype=torch.uint8, device="cuda")
        capi.moe_quantize_act_nvfp4(xb.cuda(), g, packed, scales)
        torch.cuda.synchronize()
        p_ref, s_ref, d_ref = oracle.quant_nvfp4(vb, g)
        assert np.array_equal(scales.cpu().numpy(), s_ref)
        # compare decoded values (a code of -0 and +0 decode alike)
        d_gpu = oracle.dequant(packed.cpu().numpy(), scales.cpu().numpy(), g, 0)
        assert np.array_equal(d_gpu, d_ref)
        # and the raw nibbles wherever the value is nonzero
        nz = d_ref != 0
        codes_gpu = np.stack([packed.cpu().numpy() & 15, packed.cpu().numpy() >> 4], -1).reshape(rows, K)
        codes_ref = np.stack([p_ref & 15, p_ref >> 4], -1).reshape(rows, K)
        assert np.array_equal(codes_gpu[nz], codes_ref[nz])
