"""GPU routing parity through the C ABI (moe_route) against the oracle.

Router GEMM (fp32 logits), softmax / sigmoid+bias / hash top-K (spark_model MoE pages:
moe/init.rs `moe_topk_softmax` and `new_with_hash`; moe/mod.rs `correction_bias_dev` and
`tid2eid_dev` field docs).  Ids bit-exact, weights within 1e-6 * routed_scaling.
"""
import numpy as np
import pytest
import torch

import parity
from block_quantized_moe_router_gb300 import capi, synth

pytestmark = pytest.mark.gpu


def _route_gpu(cfg, inp, logits_in=None):
    T = cfg.T
    ids = torch.full((T, cfg.k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, cfg.k), -7.0, dtype=torch.float32, device="cuda")
    logits = torch.zeros((T, cfg.E), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev = lambda key: inp[key].cuda().contiguous() if key in inp else None
    capi.moe_route(T=T, E=cfg.E, H=cfg.H, top_k=cfg.k, scoring=cfg.scoring,
                   renormalize=cfg.renorm, routed_scaling=cfg.scaling, x=dev("x"),
                   w_router=None if logits_in is not None else dev("w_router"),
                   logits_in=logits_in, logits_out=None if logits_in is not None else logits,
                   correction_bias=dev("bias"), tid2eid=dev("tid2eid"), vocab=cfg.vocab,
                   token_ids=dev("token_ids"), topk_ids=ids, topk_w=w, dev_status=status)
    torch.cuda.synchronize()
    return ids, w, logits, int(status.item())


CASES = {
    "dec1": synth.CONFIGS["dec1"],
    "dec8": synth.CONFIGS["dec8"],
    "ragged": synth.MoeConfig("ragged", T=13, H=96, I=128, E=20, k=3, scoring=synth.SCORE_SOFTMAX),
    "sig_norenorm": synth.MoeConfig("sn", T=9, H=256, I=128, E=40, k=5, scoring=synth.SCORE_SIGMOID,
                                    renorm=False, scaling=1.5),
    "soft_norenorm": synth.MoeConfig("nn", T=17, H=512, I=128, E=64, k=6, scoring=synth.SCORE_SOFTMAX,
                                     renorm=False),
    "max_experts": synth.MoeConfig("mx", T=5, H=2048, I=128, E=512, k=8, scoring=synth.SCORE_SOFTMAX),
    "sqrt_softplus": synth.MoeConfig("sq", T=21, H=1024, I=128, E=96, k=6,
                                     scoring=synth.SCORE_SQRTSOFTPLUS, scaling=1.5),
    "pre4096": synth.CONFIGS["pre4096"],
    # >= 128 tokens, experts a multiple of 128: the tensor-core router GEMM, with a ragged
    # last token block
    "tc_router": synth.MoeConfig("tr", T=300, H=384, I=128, E=128, k=6, scoring=synth.SCORE_SOFTMAX),
    "tc_router_sig": synth.MoeConfig("trs", T=129, H=1152, I=128, E=256, k=8,
                                     scoring=synth.SCORE_SIGMOID, scaling=2.5),
    # >= 128 tokens with experts not a multiple of 128: the shared-memory tiled router GEMM over
    # three 128-token blocks, the last one ragged
    "tiled_router_many": synth.MoeConfig("trm", T=300, H=512, I=128, E=96, k=6,
                                         scoring=synth.SCORE_SOFTMAX),
    # 16500 tokens: 129 token blocks of the tensor-core router, the last one ragged
    "tc_router_many": synth.MoeConfig("trw", T=16500, H=256, I=128, E=256, k=8,
                                      scoring=synth.SCORE_SOFTMAX),
    # hash-table ids, sqrt(softplus) router-score weights (router on the tensor cores, then the
    # hash kernel reads the logits)
    "hash_sqrt": synth.MoeConfig("hs", T=200, H=1024, I=128, E=128, k=6,
                                 scoring=synth.SCORE_HASH_SQRTSOFTPLUS, scaling=2.5, vocab=1000),
    "hash_sqrt_norenorm": synth.MoeConfig("hsn", T=7, H=256, I=128, E=64, k=6,
                                          scoring=synth.SCORE_HASH_SQRTSOFTPLUS, renorm=False,
                                          vocab=30),
}


@pytest.mark.parametrize("name", list(CASES))
def test_router_and_topk(cuda_lib, name):
    cfg = CASES[name]
    res = parity.gap_safe_resample(cfg, seed=0)
    inp = synth.make_inputs(cfg, seed=0, resample=res, with_weights=False)
    ref = parity.oracle_route(cfg, inp)
    ids, w, logits, status = _route_gpu(cfg, inp)
    assert status == 0
    lg = logits.double().cpu().numpy()
    assert np.max(np.abs(lg - ref["logits"])) <= 1e-4 * max(1.0, np.max(np.abs(ref["logits"])))
    parity.assert_routing(cfg, ref, ids, w, gpu_logits=logits, inp=inp)


def test_logits_in_and_nonfinite(cuda_lib):
    cfg = synth.MoeConfig("li", T=6, H=128, I=128, E=33, k=4, scoring=synth.SCORE_SOFTMAX)
    rng = np.random.default_rng(0)
    logits = rng.permuted(np.tile(np.arange(33, dtype=np.float32) * 0.01, (6, 1)), axis=1)
    logits[2, 5] = np.nan
    logits[3, 7] = np.inf
    import oracle
    ref = oracle.route(T=6, E=33, k=4, scoring=0, logits_in=logits)
    ids, w, _, status = _route_gpu(cfg, {}, logits_in=torch.from_numpy(logits).cuda())
    assert status == capi.MOE_DEV_NONFINITE and ref["status"] == capi.MOE_DEV_NONFINITE
    parity.assert_routing(cfg, ref, ids, w)


def test_max_topk_from_logits(cuda_lib):
    # E = 512 experts, top_k = 32: the largest sizes the routing kernel accepts
    cfg = synth.MoeConfig("mk", T=7, H=128, I=128, E=512, k=32, scoring=synth.SCORE_SIGMOID,
                          scaling=2.0)
    rng = np.random.default_rng(1)
    logits = np.stack([rng.permutation(512) for _ in range(7)]).astype(np.float32) * 0.01 - 2.5
    import oracle
    ref = oracle.route(T=7, E=512, k=32, scoring=1, scaling=2.0, logits_in=logits)
    ids, w, _, status = _route_gpu(cfg, {}, logits_in=torch.from_numpy(logits).cuda())
    assert status == 0
    parity.assert_routing(cfg, ref, ids, w)


def test_hash_routing_and_bad_entries(cuda_lib):
    cfg = synth.CONFIGS["hash64"]
    inp = synth.make_inputs(cfg, seed=0, with_weights=False)
    ref = parity.oracle_route(cfg, inp)
    ids, w, _, status = _route_gpu(cfg, inp)
    assert status == 0
    parity.assert_routing(cfg, ref, ids, w)
    # corrupt the table and the token ids: pairs are dropped, bits set, nothing traps
    inp["tid2eid"] = inp["tid2eid"].clone()
    tok = inp["token_ids"].clone()
    inp["tid2eid"][int(tok[0]), 2] = 64
    inp["tid2eid"][int(tok[1]), 0] = -3
    tok[5] = 40000
    inp["token_ids"] = tok
    ref = parity.oracle_route(cfg, inp)
    ids, w, _, status = _route_gpu(cfg, inp)
    assert status == (capi.MOE_DEV_BAD_EXPERT_ID | capi.MOE_DEV_BAD_TOKEN_ID) == ref["status"]
    parity.assert_routing(cfg, ref, ids, w)


def test_zero_tokens_is_noop(cuda_lib):
    cfg = synth.MoeConfig("z", T=0, H=128, I=128, E=8, k=2, scoring=synth.SCORE_SOFTMAX)
    x = torch.zeros((0, 128), dtype=torch.bfloat16, device="cuda")
    wr = torch.zeros((8, 128), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((0, 2), dtype=torch.int32, device="cuda")
    capi.moe_route(T=0, E=8, H=128, top_k=2, scoring=0, renormalize=1, routed_scaling=1.0, x=x,
                   w_router=wr, logits_out=torch.zeros((0, 8), device="cuda"), topk_ids=ids,
                   topk_w=torch.zeros((0, 2), device="cuda"))
    torch.cuda.synchronize()
