"""The C-ABI library builds, loads without a GPU, exports every symbol include/moe.h declares,
and rejects invalid arguments on the host before launching anything (CPU only)."""
import ctypes
import os
import re

import pytest

from block_quantized_moe_router_gb300 import build, capi

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return capi.load_library()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src))


def test_exports_match_header(lib):
    declared = _declared()
    assert declared == set(capi.EXPORTED)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for s in range(5):
        assert capi.moe_status_string(s).startswith("MOE_")
    assert "unknown" in capi.moe_status_string(99)


def _fake_desc(E=8, H=256, I=128, k=2, Is=0, fmt=0, Z=0):
    fake = 0x1000
    q = capi.moe_qtensor(fake, fake, fake if fmt == 0 else None, fmt)
    sq = q if Is else capi.moe_qtensor(None, None, None, 0)
    return capi.moe_ffn_desc(E, H, I, k, Is, q, q, q, sq, sq, sq, Z)


def test_workspace_size_and_validation(lib):
    n = capi.moe_workspace_size(_fake_desc(), 4, capi.MOE_ACT_BF16)
    n4 = capi.moe_workspace_size(_fake_desc(), 4, capi.MOE_ACT_NVFP4)
    assert n > 0 and n4 > 0
    assert capi.moe_workspace_size(_fake_desc(Is=128), 4, 0) > n
    # more tokens never need less workspace, on every path
    for act in (0, 1):
        sizes = [capi.moe_workspace_size(_fake_desc(H=512, I=256, Is=256), T, act)
                 for T in (1, 8, 9, 64, 1000)]
        assert all(a <= b for a, b in zip(sizes[2:], sizes[3:]))
    assert capi.moe_workspace_size(_fake_desc(k=9, Z=2), 4, 0) > 0  # k <= E + Z is fine
    for bad in [_fake_desc(E=0), _fake_desc(E=513), _fake_desc(k=9), _fake_desc(k=0),
                _fake_desc(H=200), _fake_desc(I=64), _fake_desc(Is=100), _fake_desc(Z=-1),
                _fake_desc(E=510, Z=3)]:
        with pytest.raises(capi.MoeError) as ei:
            capi.moe_workspace_size(bad, 4, 0)
        assert ei.value.status == capi.MOE_ERR_INVALID_ARG
    with pytest.raises(capi.MoeError):
        capi.moe_workspace_size(_fake_desc(), -1, 0)
    with pytest.raises(capi.MoeError):
        capi.moe_workspace_size(_fake_desc(), 4, 7)
    d = _fake_desc()
    d.gate.globals = None  # NVFP4 needs its per-tensor global
    with pytest.raises(capi.MoeError):
        capi.moe_workspace_size(d, 4, 0)


def test_host_workspace_size(lib):
    """The host-buffer entry's workspace is the FFN workspace plus its staging area."""
    for T, act in ((1, 0), (8, 0), (64, 0), (300, 1)):
        d = _fake_desc(H=512, I=256, Is=256, Z=2)
        n = capi.moe_workspace_size(d, T, act)
        nh = capi.moe_workspace_size_host(d, T, act)
        stage = 2 * T * 512 * 2 + 2 * T * 2 * 4 + T * (8 + 2) * 4 + T * 4
        assert n + stage <= nh <= n + stage + 7 * 256
    with pytest.raises(capi.MoeError):
        capi.moe_workspace_size_host(_fake_desc(E=0), 4, 0)
    fake = ctypes.c_void_p(0x1000)
    d = capi.moe_route_desc(4, 8, 256, 2, 0, 1, 1.0, 0x1000, None, None, 0, None, 0)
    assert lib.moe_forward_host(None, ctypes.byref(d), 0, 1.0, 1.0, fake, None, fake, None, None,
                                fake, 1 << 20, None, None) == capi.MOE_ERR_INVALID_ARG


def test_route_rejects_before_launch(lib):
    fake = ctypes.c_void_p(0x1000)

    def call(**kw):
        args = dict(T=4, E=8, H=64, top_k=2, scoring=0, renormalize=1, routed_scaling=1.0,
                    w_router=None, correction_bias=None, tid2eid=None, vocab=0, token_ids=None,
                    zero_experts=0)
        args.update(kw)
        d = capi.moe_route_desc(*[args[f] for f, _ in capi.moe_route_desc._fields_])
        return lib.moe_route(ctypes.byref(d), fake, None, None, fake, fake, None, None)

    assert call(top_k=9) == capi.MOE_ERR_INVALID_ARG
    assert call(E=0) == capi.MOE_ERR_INVALID_ARG
    assert call(T=-1) == capi.MOE_ERR_INVALID_ARG
    assert call(scoring=6, w_router=0x1000) == capi.MOE_ERR_INVALID_ARG
    assert call(scoring=5, w_router=0x1000) == capi.MOE_ERR_INVALID_ARG  # no table, vocab 0
    assert call(scoring=5, w_router=0x1000, vocab=10) == capi.MOE_ERR_INVALID_ARG  # no table
    assert call(zero_experts=-1, w_router=0x1000) == capi.MOE_ERR_INVALID_ARG
    assert call(E=500, zero_experts=13, w_router=0x1000) == capi.MOE_ERR_INVALID_ARG  # E + Z > 512
    assert call(top_k=9, zero_experts=1, w_router=0x1000) == capi.MOE_ERR_INVALID_ARG  # k > E + Z
    assert call() == capi.MOE_ERR_INVALID_ARG               # no logits and no router
    assert call(scoring=2) == capi.MOE_ERR_INVALID_ARG      # hash without a table
    assert call(routed_scaling=float("nan"), w_router=0x1000) == capi.MOE_ERR_INVALID_ARG


def test_ffn_forward_rejects_bad_handle(lib):
    fake = ctypes.c_void_p(0x1000)
    st = lib.moe_ffn_forward(None, 4, 0, 1.0, 1.0, fake, fake, fake, fake, fake, 1 << 20, None, None)
    assert st == capi.MOE_ERR_INVALID_ARG
    assert lib.moe_release_weights(None) == capi.MOE_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    d = _fake_desc(E=0)
    assert lib.moe_prepare_weights(ctypes.byref(d), ctypes.byref(h), None) == capi.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_act_nvfp4(fake, 4, 24, 1.0, fake, fake, None) == capi.MOE_ERR_INVALID_ARG


def test_every_declaration_cites_its_passage():
    """Each entry point's comment names the passage of the pages that defines it (a page of
    the spark_model MoE source: moe/mod.rs, moe/init.rs, qwen3_attention/init.rs) or says that
    the pages have no counterpart."""
    src = open(HEADER).read()
    decls = list(re.finditer(r"\n(moe_status_t|const char\*)\s+(moe_[a-z_0-9]+)\s*\(", src))
    assert {m.group(2) for m in decls} == set(capi.EXPORTED)
    for m in decls:
        before = src[:m.start() + 1]
        # the comment block that ends right before this declaration (or before the previous
        # declaration of a pair that shares one comment)
        end = before.rfind("*/")
        start = before.rfind("/*", 0, end)
        comment = before[start:end]
        between = before[end + 2:]
        assert re.fullmatch(r"\s*(moe_status_t [^;]*;\s*)?", between, flags=re.S), m.group(2)
        assert ("moe/mod.rs" in comment or "moe/init.rs" in comment or
                "qwen3_attention/init.rs" in comment or "no counterpart" in comment), m.group(2)
