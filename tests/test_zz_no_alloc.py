"""moe_ffn_forward_noalloc: the expert FFN for callers that cannot give the library device
memory (a host that freezes its memory plan after start-up, or a plugin interface with no
workspace argument).  The entry point runs on a static 8 MiB device array inside the library.

Checked through the C ABI against the existing entry point, moe_ffn_forward with a caller
workspace, on two calls in a row with different inputs (so a stale array would show), within
the block's output tolerance; and an oversize request must be refused without touching the
output.  This file is collected last so that a run stopping at its first failure has already
run every other test.
"""
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
    "ragged_a4": S.MoeConfig("ragged_a4", T=13, H=384, I=256, E=10, k=3, scoring=S.SCORE_SOFTMAX,
                             I_shared=128, act=S.ACT_NVFP4),
    "dec8": S.CONFIGS["dec8"],
}


def _close(a: torch.Tensor, b: torch.Tensor):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    assert np.all(np.isfinite(a))
    assert np.max(np.abs(a - b)) <= 1e-2 * np.max(np.abs(b)) + 1e-3


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_workspace_entry_point(cuda_lib, name):
    cfg = CASES[name]
    inp = synth.make_inputs(cfg, seed=5, device="cuda")
    layer = MoeLayer.from_inputs(inp)
    xs = [inp["x"].cuda(), torch.flip(inp["x"], dims=[0]).contiguous().cuda() * 0.5]
    for x in xs:  # two calls in a row, different inputs
        ids, w, _ = layer.route(x)
        ref = layer.ffn(x, ids, w)
        out = torch.full_like(ref, float("nan"))
        capi.moe_ffn_forward_noalloc(layer.handle, cfg.T, cfg.act, 1.0, 1.0, x, ids, w, out,
                                     dev_status=layer.status)
        torch.cuda.synchronize()
        assert int(layer.status.item()) == 0
        _close(out, ref)
    layer.close()


def test_noalloc_refuses_oversize_plan(cuda_lib):
    cfg = S.CONFIGS["hash64"]   # 64 tokens need a 9.3 MiB plan, above the 8 MiB array
    inp = synth.make_inputs(cfg, seed=0, device="cuda")
    layer = MoeLayer.from_inputs(inp)
    x = inp["x"].cuda()
    ids, w, _ = layer.route(x, token_ids=inp["token_ids"].cuda())
    out = torch.full((cfg.T, cfg.H), 7.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(capi.MoeError) as ei:
        capi.moe_ffn_forward_noalloc(layer.handle, cfg.T, cfg.act, 1.0, 1.0, x, ids, w, out)
    assert ei.value.status == capi.MOE_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
    # a smaller batch of the same layer fits
    x8 = x[:8].contiguous()
    ids8, w8 = ids[:8].contiguous(), w[:8].contiguous()
    ref = layer.ffn(x8, ids8, w8)
    out8 = torch.empty_like(ref)
    capi.moe_ffn_forward_noalloc(layer.handle, 8, cfg.act, 1.0, 1.0, x8, ids8, w8, out8)
    torch.cuda.synchronize()
    _close(out8, ref)
    layer.close()
