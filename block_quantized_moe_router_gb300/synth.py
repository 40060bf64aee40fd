"""Seeded synthetic inputs for the MoE FFN block.

This module is the ONLY code shared by the CUDA library's tests/benchmark and the CPU oracle.
It draws random numbers and encodes the random expert weights into the block-quantized
storage formats (the offline job a checkpoint loader does); it holds none of the MoE
block's own arithmetic (no routing, no dequantized dot products, no activation quantizer).

Workloads (all seeded, synthetic):
  tiny     4 tokens, H 256, I 128, 8 experts, top-2 softmax renormalised, 1 shared expert
  dec1     1 token,  H 2048, I 768, 128 experts, top-8 softmax renormalised, no shared expert
  dec8     8 tokens, H 7168, I 2048, 256 experts, top-8 sigmoid + correction bias, x2.5,
           1 shared expert (I_s 2048)
  pre4096  4096 tokens with the dec8 shapes and routing, router logits skewed so that the
           per-expert token counts fall off like a Zipf law (s = 1.1); NVFP4 activations
  pre32768 the same with 32768 tokens (compute-bound: ~1000 rows per expert)
  hash64   64 tokens, H 4096, I 2048, 64 experts, top-6 from a tid2eid [32000, 6] table,
           weights 1/6; routed experts MXFP4, shared expert NVFP4

Zero-computation experts (ids E .. E + Z - 1, router width E + Z) appear only in test cases.

Distributions: x ~ N(0,1) in bf16; router ~ N(0, 0.02) in bf16; expert weights
~ N(0, 0.02) fp32 encoded to NVFP4 (per-tensor global amax/(6*448), E4M3 scale per 16 =
E4M3(block amax / 6 / global), nearest E2M1 code) or to MXFP4 (E8M0 scale per 32 =
2^(floor(log2 block amax) - 2), nearest E2M1 code, saturating at 6); correction bias
~ U(-0.1, 0.1) (softmax + bias routing: U(-0.01, 0.01)).
"""
from __future__ import annotations

import dataclasses
import json
import math
import os
from typing import Dict, Optional

import numpy as np
import torch

FMT_NVFP4, FMT_MXFP4 = 0, 1
SCORE_SOFTMAX, SCORE_SIGMOID, SCORE_HASH, SCORE_SQRTSOFTPLUS, SCORE_SOFTMAX_BIAS = 0, 1, 2, 3, 4
SCORE_HASH_SQRTSOFTPLUS = 5  # hash-table ids, weights from the router's sqrt(softplus) scores
ACT_BF16, ACT_NVFP4 = 0, 1


@dataclasses.dataclass(frozen=True)
class MoeConfig:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    scoring: int
    renorm: bool = True
    scaling: float = 1.0
    I_shared: int = 0            # 0 = no shared expert
    fmt: int = FMT_NVFP4         # routed experts
    shared_fmt: int = FMT_NVFP4
    act: int = ACT_BF16
    vocab: int = 0               # hash routing table rows
    zipf_s: float = 0.0          # > 0: skew router logits so expert counts follow Zipf(s)
    zero_experts: int = 0        # zero-computation experts (ids E .. E + Z - 1, output = input)

    @property
    def pairs(self) -> int:
        return self.T * self.k

    def with_T(self, T: int) -> "MoeConfig":
        return dataclasses.replace(self, T=T)


CONFIGS: Dict[str, MoeConfig] = {
    "tiny": MoeConfig("tiny", T=4, H=256, I=128, E=8, k=2, scoring=SCORE_SOFTMAX, I_shared=128),
    "dec1": MoeConfig("dec1", T=1, H=2048, I=768, E=128, k=8, scoring=SCORE_SOFTMAX),
    "dec8": MoeConfig("dec8", T=8, H=7168, I=2048, E=256, k=8, scoring=SCORE_SIGMOID,
                      scaling=2.5, I_shared=2048),
    "pre4096": MoeConfig("pre4096", T=4096, H=7168, I=2048, E=256, k=8, scoring=SCORE_SIGMOID,
                         scaling=2.5, I_shared=2048, act=ACT_NVFP4, zipf_s=1.1),
    # the prefill shapes with 8x the tokens: ~1000 rows per expert, above the FP4 ridge
    # (the compute-bound variant of the 4096-token case)
    "pre32768": MoeConfig("pre32768", T=32768, H=7168, I=2048, E=256, k=8, scoring=SCORE_SIGMOID,
                          scaling=2.5, I_shared=2048, act=ACT_NVFP4, zipf_s=1.1),
    "hash64": MoeConfig("hash64", T=64, H=4096, I=2048, E=64, k=6, scoring=SCORE_HASH,
                        I_shared=2048, fmt=FMT_MXFP4, shared_fmt=FMT_NVFP4, vocab=32000),
    # decode-shaped (8 tokens, dec8 shapes) and prefill-shaped cases small enough (32 experts,
    # ~0.9 GB of weights) for multi-pass profiler captures
    "dec8_e32": MoeConfig("dec8_e32", T=8, H=7168, I=2048, E=32, k=8, scoring=SCORE_SIGMOID,
                          scaling=2.5, I_shared=2048),
    "pre1024_e32": MoeConfig("pre1024_e32", T=1024, H=7168, I=2048, E=32, k=8,
                             scoring=SCORE_SIGMOID, scaling=2.5, I_shared=2048, act=ACT_NVFP4),
}

# Router-logit skew for the Zipf workloads: column H-1 of x is 1 and column H-1 of the router
# holds a per-expert lift, so every token's logit of an expert is raised by that expert's lift.
# The lift of the expert of Zipf rank r starts from ZIPF_TAU * ln(target_r / T), target_r the
# water-filled Zipf(s) pair count of rank r (zipf_targets); ZIPF_TAU is the single lift scale
# whose realized counts come closest to the targets (total variation) for the 4096-token
# workload.  One scale cannot match head and tail together (the token-to-token spread of the
# logits is larger than the lifts), so for the named prefill workloads tests/zipf_fit.py then
# refines each rank's lift by damped fixed-point passes of the oracle's fp64 routing and writes
# the lifts to zipf_lifts.json (read here); other Zipf configurations use the single-scale
# form.  The realized counts are reported by the benchmark.
ZIPF_TAU = 0.9193
_ZIPF_LIFTS_FILE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "zipf_lifts.json")
_zipf_lifts_cache: Optional[dict] = None


def stored_zipf_lifts(name: str) -> Optional[np.ndarray]:
    """Per-rank lifts written by the Zipf fit for workload `name`, or None."""
    global _zipf_lifts_cache
    if _zipf_lifts_cache is None:
        _zipf_lifts_cache = {}
        if os.path.exists(_ZIPF_LIFTS_FILE):
            with open(_ZIPF_LIFTS_FILE) as fh:
                _zipf_lifts_cache = json.load(fh)
    v = _zipf_lifts_cache.get(name)
    return None if v is None else np.asarray(v["lifts"], dtype=np.float64)


def zipf_targets(T: int, k: int, E: int, s: float) -> np.ndarray:
    """Per-rank pair counts (float64, rank 1 first): the T * k pairs shared in proportion to
    rank^-s, no expert above T (an expert takes each token at most once); the excess of a
    capped expert is spread over the others in proportion to their shares, repeatedly."""
    p = np.arange(1, E + 1, dtype=np.float64) ** -s
    total = float(T * k)
    capped = np.zeros(E, dtype=bool)
    while True:
        free = ~capped
        share = (total - T * capped.sum()) * p / p[free].sum()
        newly = free & (share > T)
        if not newly.any():
            return np.where(capped, float(T), share)
        capped |= newly


_E2M1_MIDPOINTS = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


def _gen(seed: int, *salt: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    s = seed & 0xFFFFFFFF
    for v in salt:
        s = (s * 1000003 + (v & 0xFFFFFFFF) + 0x9E3779B9) & 0xFFFFFFFFFFFF
    g.manual_seed(s)
    return g


def _nearest_e2m1_codes(q: torch.Tensor) -> torch.Tensor:
    """Nearest E2M1 code (sign in bit 3) for each value, magnitudes saturating at 6."""
    mag = torch.bucketize(q.abs(), _E2M1_MIDPOINTS.to(q.device))
    return (mag | ((q < 0).to(torch.int64) << 3)).to(torch.uint8)


def _pack_nibbles(codes: torch.Tensor) -> torch.Tensor:
    """[..., K] codes -> [..., K/2] bytes, element 2i in the low nibble."""
    lo = codes[..., 0::2]
    hi = codes[..., 1::2]
    return (lo | (hi << 4)).to(torch.uint8)


def encode_nvfp4(w: torch.Tensor):
    """w [E, N, K] float32 -> dict(packed [E,N,K/2] u8, scales [E,N,K/16] u8, globals [E] f32)."""
    E, N, K = w.shape
    amax = w.abs().amax(dim=(1, 2)).clamp_min(1e-30)
    glob = (amax / (6.0 * 448.0)).float()
    blocks = w.reshape(E, N, K // 16, 16)
    bamax = blocks.abs().amax(-1)
    s = (bamax / 6.0 / glob[:, None, None]).clamp(max=448.0).to(torch.float8_e4m3fn)
    denom = s.float() * glob[:, None, None]
    q = torch.where(denom[..., None] > 0, blocks / denom[..., None].clamp_min(1e-30),
                    torch.zeros_like(blocks))
    codes = _nearest_e2m1_codes(q).reshape(E, N, K)
    return dict(packed=_pack_nibbles(codes), scales=s.view(torch.uint8), globals=glob,
                fmt=FMT_NVFP4)


def encode_mxfp4(w: torch.Tensor):
    """w [E, N, K] float32 -> dict(packed [E,N,K/2] u8, scales [E,N,K/32] u8 (E8M0), globals None)."""
    E, N, K = w.shape
    blocks = w.reshape(E, N, K // 32, 32)
    bamax = blocks.abs().amax(-1)
    expo = torch.floor(torch.log2(bamax.clamp_min(2.0 ** -126))) - 2.0
    expo = expo.clamp(-127, 127)
    sbyte = (expo + 127).to(torch.uint8)
    q = blocks / torch.exp2(expo)[..., None]
    codes = _nearest_e2m1_codes(q).reshape(E, N, K)
    return dict(packed=_pack_nibbles(codes), scales=sbyte, globals=None, fmt=FMT_MXFP4)


def _expert_weights(E, N, K, fmt, seed, salt, device, chunk=8):
    """Draw N(0, 0.02) weights expert-chunk by expert-chunk and encode them."""
    parts = []
    g = _gen(seed, salt, device=device)
    for e0 in range(0, E, chunk):
        e1 = min(E, e0 + chunk)
        w = torch.randn((e1 - e0, N, K), generator=g, device=device, dtype=torch.float32) * 0.02
        parts.append(encode_nvfp4(w) if fmt == FMT_NVFP4 else encode_mxfp4(w))
        del w
    out = {"fmt": fmt}
    for key in ("packed", "scales", "globals"):
        vals = [p[key] for p in parts]
        out[key] = None if vals[0] is None else torch.cat(vals, 0).contiguous()
    return out


def zipf_logit_offsets(cfg: MoeConfig, seed: int, tau: Optional[float] = None,
                       lifts: Optional[np.ndarray] = None) -> torch.Tensor:
    """Per-expert logit lifts.  `lifts` (per rank) if given, else the stored per-rank lifts of
    the workload when the fit wrote some and no `tau` is asked for, else tau * ln(target_r / T)
    (tau defaults to ZIPF_TAU); rank r -> expert id is a seeded permutation."""
    if lifts is None and tau is None:
        lifts = stored_zipf_lifts(cfg.name)
    if lifts is None:
        tau = ZIPF_TAU if tau is None else tau
        lifts = tau * np.log(zipf_targets(cfg.T, cfg.k, cfg.E, cfg.zipf_s) / cfg.T)
    perm = torch.randperm(cfg.E, generator=_gen(seed, 77))
    c = torch.empty(cfg.E, dtype=torch.float64)
    c[perm] = torch.from_numpy(np.asarray(lifts, dtype=np.float64))
    return c


def zipf_rank_of_expert(cfg: MoeConfig, seed: int) -> np.ndarray:
    """rank index (0 = the largest target) of every expert id, as zipf_logit_offsets lays them."""
    perm = torch.randperm(cfg.E, generator=_gen(seed, 77))
    rank = np.empty(cfg.E, dtype=np.int64)
    rank[perm.numpy()] = np.arange(cfg.E)
    return rank


def make_inputs(cfg: MoeConfig, seed: int = 0, device="cpu",
                resample: Optional[Dict[int, int]] = None, with_weights: bool = True,
                zipf_tau: Optional[float] = None, zipf_lifts: Optional[np.ndarray] = None):
    """Build one layer's inputs.

    Activations, router, bias, hash table and token ids are drawn on the CPU (so they are
    identical whatever the device); expert weights are drawn on ``device`` (CPU and CUDA
    random streams differ, so a test builds them once and copies them to both sides).
    ``resample`` maps a token index to a redraw counter: that token's x row is redrawn from
    an independent stream (used to enforce a minimum top-K score gap).
    """
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
    Er = E + cfg.zero_experts  # router outputs: real experts, then zero-computation experts
    inp = {"cfg": cfg}
    x = torch.randn((T, H), generator=_gen(seed, 1), dtype=torch.float32)
    for t, cnt in (resample or {}).items():
        if cnt > 0:
            x[t] = torch.randn((H,), generator=_gen(seed, 2, t, cnt), dtype=torch.float32)
    if cfg.scoring != SCORE_HASH:
        wr = torch.randn((Er, H), generator=_gen(seed, 3), dtype=torch.float32) * 0.02
        if cfg.zipf_s > 0:
            x[:, H - 1] = 1.0
            wr[:, H - 1] = zipf_logit_offsets(cfg, seed, zipf_tau, zipf_lifts).float()
        inp["w_router"] = wr.to(torch.bfloat16)
    inp["x"] = x.to(torch.bfloat16)
    if cfg.scoring in (SCORE_SIGMOID, SCORE_SQRTSOFTPLUS, SCORE_SOFTMAX_BIAS):
        u = torch.rand((Er,), generator=_gen(seed, 4), dtype=torch.float32) * 0.2 - 0.1
        # softmax probabilities are ~1/Er: a bias of +-0.01 is on their scale
        inp["bias"] = u * 0.1 if cfg.scoring == SCORE_SOFTMAX_BIAS else u
    if cfg.scoring in (SCORE_HASH, SCORE_HASH_SQRTSOFTPLUS):
        gt = _gen(seed, 5)
        inp["tid2eid"] = torch.rand((cfg.vocab, Er), generator=gt).argsort(dim=1)[:, :k].contiguous().to(torch.int64)
        inp["token_ids"] = torch.randint(0, cfg.vocab, (T,), generator=_gen(seed, 6), dtype=torch.int32)
    if with_weights:
        inp["gate"] = _expert_weights(E, I, H, cfg.fmt, seed, 10, device)
        inp["up"] = _expert_weights(E, I, H, cfg.fmt, seed, 11, device)
        inp["down"] = _expert_weights(E, H, I, cfg.fmt, seed, 12, device)
        if cfg.I_shared:
            Is = cfg.I_shared
            inp["sh_gate"] = _expert_weights(1, Is, H, cfg.shared_fmt, seed, 20, device)
            inp["sh_up"] = _expert_weights(1, Is, H, cfg.shared_fmt, seed, 21, device)
            inp["sh_down"] = _expert_weights(1, H, Is, cfg.shared_fmt, seed, 22, device)
    return inp


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 array of its bit patterns."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_numpy_proj(p):
    """Weight dict (torch) -> weight dict (numpy, host) for the oracle."""
    if p is None:
        return None
    return dict(packed=p["packed"].cpu().numpy(), scales=p["scales"].cpu().numpy(),
                globals=None if p["globals"] is None else p["globals"].cpu().numpy(),
                fmt=p["fmt"])


def weight_bytes_per_expert(cfg: MoeConfig, I: Optional[int] = None, fmt: Optional[int] = None) -> int:
    """Bytes of one expert's gate+up+down (packed codes + block scales + globals)."""
    I = cfg.I if I is None else I
    fmt = cfg.fmt if fmt is None else fmt
    sv = 16 if fmt == FMT_NVFP4 else 32
    n = 3 * cfg.H * I
    return n // 2 + n // sv + (3 * 4 if fmt == FMT_NVFP4 else 0)


def expected_distinct(E: int, picks_per_token: int, T: int) -> float:
    """Expected number of distinct experts touched by T tokens with uniform routing."""
    return E * (1.0 - (1.0 - picks_per_token / E) ** T)


__all__ = ["MoeConfig", "CONFIGS", "make_inputs", "encode_nvfp4", "encode_mxfp4", "bf16_bits",
           "to_numpy_proj", "weight_bytes_per_expert", "expected_distinct", "zipf_targets",
           "zipf_logit_offsets", "zipf_rank_of_expert", "stored_zipf_lifts", "math"]
