"""Pins of the oracle's format tables and activation quantizer (CPU only).

Sources: the weight formats of the spark_model MoE pages (moe/mod.rs, `experts_scale_kind`
field doc: E2M1 + E4M3 per 16 + f32 global, or E2M1 + E8M0 per 32) and the NVFP4 activation
quantizer of the FP4 x FP4 recipe (qwen3_attention/init.rs `quantize_bf16_to_nvfp4` handle).
The tables are checked against the OCP formats' closed forms and against torch's own FP8
conversions (an independent library), the quantizer against hand-worked examples.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_quant_examples.json")


def test_e2m1_table_closed_form(orc):
    e2m1, _, _ = orc.tables()
    for c in range(16):
        s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
        mag = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)   # bias 1, subnormal at e=0
        assert e2m1[c] == (-mag if s else mag), c
    assert sorted(set(np.abs(e2m1))) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def test_e4m3_table_matches_torch_float8(orc):
    _, e4m3, _ = orc.tables()
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(e4m3))
    assert set(np.nonzero(nan)[0]) == {0x7F, 0xFF}
    assert np.array_equal(ref[~nan], e4m3[~nan])
    assert e4m3[0x01] == 2.0 ** -9 and e4m3[0x7E] == 448.0 and e4m3[0x38] == 1.0


def test_e8m0_table(orc):
    _, _, e8m0 = orc.tables()
    for b in range(255):
        assert e8m0[b] == math.ldexp(1.0, b - 127)
    assert math.isnan(e8m0[255]) and e8m0[127] == 1.0
    if hasattr(torch, "float8_e8m0fnu"):
        ref = torch.arange(255, dtype=torch.int32).to(torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
        assert np.array_equal(ref, e8m0[:255])


def test_e2m1_encode_midpoints_and_roundtrip(orc):
    e2m1, _, _ = orc.tables()
    # hand-worked ties (to the even code) and saturation
    for v, want in [(0.25, 0.0), (0.75, 1.0), (1.25, 1.0), (1.75, 2.0), (2.5, 2.0), (3.5, 4.0),
                    (5.0, 4.0), (7.0, 6.0), (100.0, 6.0), (-5.0, -4.0), (0.26, 0.5), (4.9, 4.0)]:
        assert e2m1[orc.e2m1_encode(v)] == want, v
    for c in range(16):
        back = orc.e2m1_encode(e2m1[c])
        assert back == c or (c == 8 and back == 8) or (c == 0 and back == 0)


def test_e4m3_encode_roundtrip_and_rounding(orc):
    _, e4m3, _ = orc.tables()
    for b in range(0x7F):  # every finite non-negative code
        assert orc.e4m3_encode(e4m3[b]) == b
    assert orc.e4m3_encode(1000.0) == 0x7E          # saturates
    assert orc.e4m3_encode(2.0 ** -10) == 0          # tie between 0 and 2^-9 -> even (0)
    assert orc.e4m3_encode(1.5 * 2.0 ** -9) == 2     # tie between m=1 and m=2 -> even (2)
    assert orc.e4m3_encode(1.0625) == 0x38           # tie 1.0 / 1.125 -> even mantissa (1.0)
    assert orc.e4m3_encode(1.1875) == 0x3A           # tie 1.125 / 1.25 -> even mantissa (1.25)
    # against torch's RNE float8 cast on random positive values
    rng = np.random.default_rng(0)
    vals = np.exp(rng.uniform(-12, 6.1, 2000)).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(float(v)) for v in vals], np.uint8)
    assert np.array_equal(ref, got)


@pytest.mark.parametrize("ex", json.load(open(GOLDEN))["examples"], ids=lambda e: e["name"])
def test_quantizer_hand_worked(orc, ex):
    packed, scales, deq = orc.quant_nvfp4(np.array(ex["v"], np.float32)[None, :], g=ex["g"])
    assert int(scales[0, 0]) == ex["scale"]
    assert list(packed[0]) == ex["packed"]
    assert np.array_equal(deq[0], np.array(ex["deq"], np.float64))


def test_quantizer_idempotent_and_dequant_consistent(orc):
    rng = np.random.default_rng(1)
    v = rng.standard_normal((32, 256)).astype(np.float32) * rng.uniform(0.01, 50, (32, 1)).astype(np.float32)
    for g in (1.0, 0.5, 4.0):
        packed, scales, deq = orc.quant_nvfp4(v, g)
        p2, s2, d2 = orc.quant_nvfp4(deq.astype(np.float32), g)
        assert np.array_equal(deq, d2)
        assert np.array_equal(scales, s2)
        # the packed codes decode (through the weight-format dequantizer) to the same values
        assert np.array_equal(orc.dequant(packed, scales, g, 0), deq)
        # per-block error bound: half an E2M1 step at the top of the block's range
        err = np.abs(deq - v).reshape(32, -1, 16).max(-1)
        amax = np.abs(v).reshape(32, -1, 16).max(-1)
        assert np.all(err <= amax / 6 * 1.0625 * 1.0 + 1e-30)


def test_dequant_mxfp4_and_nvfp4_layouts(orc):
    # one row, K = 64: check nibble order, block indexing and the global multiplier
    packed = np.zeros((1, 32), np.uint8)
    packed[0, 0] = 0x21          # k=0 -> code 1 (0.5), k=1 -> code 2 (1.0)
    packed[0, 16] = 0xF7         # k=32 -> 6, k=33 -> -6
    s_nv = np.array([[0x38, 0x40, 0x30, 0x48]], np.uint8)     # 1, 2, 0.5, 4
    d = orc.dequant(packed, s_nv, 0.25, 0)
    assert d[0, 0] == 0.5 * 1 * 0.25 and d[0, 1] == 1.0 * 0.25
    assert d[0, 32] == 6 * 0.5 * 0.25 and d[0, 33] == -6 * 0.5 * 0.25
    s_mx = np.array([[127, 130]], np.uint8)                    # 1, 8
    d = orc.dequant(packed, s_mx, 123.0, 1)                    # global ignored for MXFP4
    assert d[0, 0] == 0.5 and d[0, 1] == 1.0 and d[0, 32] == 48.0 and d[0, 33] == -48.0
