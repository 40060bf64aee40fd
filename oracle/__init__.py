"""CPU oracle for the MoE FFN block -- TEST INFRASTRUCTURE ONLY.

This package is the slow, plain, fp64 reference that the CUDA library is checked against.
Only the test-suite, the package smoke check and the benchmark's CPU-baseline leg may import
it.  It shares no code with the CUDA library and never imports it; the CUDA library never
imports this package.

The arithmetic lives in ``moe_oracle.cpp`` (multithreaded C++, table decoding, fp64
accumulation), compiled to a shared object by :func:`build` and called through ctypes.
Every function cites the passage of the spark_model MoE pages it follows; see the C++ header.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmoe_oracle.so")
_lib = None

SCORE_SOFTMAX, SCORE_SIGMOID, SCORE_HASH, SCORE_SQRTSOFTPLUS, SCORE_SOFTMAX_BIAS = 0, 1, 2, 3, 4
SCORE_HASH_SQRTSOFTPLUS = 5  # ids from the hash table, weights from sqrt(softplus) router scores
FMT_NVFP4, FMT_MXFP4 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (-O2, no fast-math) into oracle/_build/."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-fno-fast-math", "-std=c++17", "-shared", "-fPIC",
                               "-pthread", _SRC, "-o", tmp])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Proj(ctypes.Structure):
    _fields_ = [("packed", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("globals", ctypes.c_void_p), ("fmt", ctypes.c_int)]


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    vp, i32, i64, f32, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double
    lib.orc_tables.argtypes = [vp, vp, vp]
    lib.orc_e2m1_encode.argtypes = [f32]
    lib.orc_e2m1_encode.restype = ctypes.c_uint8
    lib.orc_e4m3_encode.argtypes = [f32]
    lib.orc_e4m3_encode.restype = ctypes.c_uint8
    lib.orc_quant_nvfp4.argtypes = [vp, i64, i64, f32, vp, vp, vp]
    lib.orc_dequant.argtypes = [vp, vp, f64, i32, i64, i64, vp]
    lib.orc_route.argtypes = [i32, i32, i32, i32, i32, i32, f64, vp, vp, vp, vp, vp, i64, vp,
                              vp, vp, vp, vp, vp, i32]
    lib.orc_route.restype = i32
    lib.orc_moe_ffn.argtypes = [i32, i32, i32, i32, i32, i32, _Proj, _Proj, _Proj, i32, _Proj,
                                _Proj, _Proj, i32, f32, f32, vp, vp, vp, vp, i32]
    lib.orc_moe_ffn.restype = i32
    lib.orc_hardware_threads.restype = i32
    _lib = lib
    return lib


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _as(a, dtype):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=dtype)


def hardware_threads() -> int:
    return int(_load().orc_hardware_threads())


def tables():
    """(e2m1[16], e4m3[256], e8m0[256]) decode tables, fp64 (NaN codes included)."""
    lib = _load()
    a, b, c = np.zeros(16), np.zeros(256), np.zeros(256)
    lib.orc_tables(_ptr(a), _ptr(b), _ptr(c))
    return a, b, c


def e2m1_encode(v: float) -> int:
    return int(_load().orc_e2m1_encode(float(np.float32(v))))


def e4m3_encode(v: float) -> int:
    return int(_load().orc_e4m3_encode(float(np.float32(v))))


def quant_nvfp4(v: np.ndarray, g: float = 1.0):
    """Activation quantizer Q (fp32): rows of v [R, K] -> (packed [R,K/2], scales [R,K/16], deq fp64)."""
    v = _as(v, np.float32)
    if v.ndim == 1:
        v = v[None, :]
    R, K = v.shape
    assert K % 16 == 0
    packed = np.zeros((R, K // 2), np.uint8)
    scales = np.zeros((R, K // 16), np.uint8)
    deq = np.zeros((R, K), np.float64)
    _load().orc_quant_nvfp4(_ptr(v), R, K, float(g), _ptr(packed), _ptr(scales), _ptr(deq))
    return packed, scales, deq


def dequant(packed: np.ndarray, scales: np.ndarray, global_scale: float, fmt: int) -> np.ndarray:
    """Dequantize one [N, K] block-quantized matrix to fp64."""
    packed = _as(packed, np.uint8)
    scales = _as(scales, np.uint8)
    N = packed.shape[0]
    K = packed.shape[1] * 2
    out = np.zeros((N, K), np.float64)
    _load().orc_dequant(_ptr(packed), _ptr(scales), float(global_scale), int(fmt), N, K, _ptr(out))
    return out


def route(*, T, E, k, scoring, renorm=True, scaling=1.0, x_bf16=None, w_router_bf16=None,
          logits_in=None, bias=None, tid2eid=None, token_ids=None, vocab=0, nthreads=0):
    """Router GEMM (fp64) + top-K selection + routing weights.

    x_bf16 / w_router_bf16 are uint16 arrays holding bf16 bit patterns.
    Returns dict(ids [T,k] int32, w [T,k] fp64, logits [T,E] fp64 or None,
    score [T,E] fp64 or None, status int).
    """
    lib = _load()
    H = 0 if x_bf16 is None else x_bf16.shape[1]
    x_bf16, w_router_bf16 = _as(x_bf16, np.uint16), _as(w_router_bf16, np.uint16)
    logits_in, bias = _as(logits_in, np.float32), _as(bias, np.float32)
    tid2eid, token_ids = _as(tid2eid, np.int64), _as(token_ids, np.int32)
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    want_scores = scoring != SCORE_HASH
    logits = np.zeros((T, E), np.float64) if want_scores else None
    score = np.zeros((T, E), np.float64) if want_scores else None
    status = np.zeros(1, np.int32)
    rc = lib.orc_route(T, E, H, k, scoring, int(bool(renorm)), float(scaling), _ptr(x_bf16),
                       _ptr(w_router_bf16), _ptr(logits_in), _ptr(bias), _ptr(tid2eid), int(vocab),
                       _ptr(token_ids), _ptr(logits), _ptr(ids), _ptr(w), _ptr(score),
                       _ptr(status), int(nthreads))
    if rc != 0:
        raise ValueError("oracle route: invalid arguments")
    return dict(ids=ids, w=w, logits=logits, score=score, status=int(status[0]))


def _proj(p):
    """p = dict(packed, scales, globals or None, fmt) -> (_Proj, keepalive list)."""
    if p is None:
        return _Proj(None, None, None, 0), []
    packed = _as(p["packed"], np.uint8)
    scales = _as(p["scales"], np.uint8)
    glob = _as(p.get("globals"), np.float32)
    return _Proj(_ptr(packed), _ptr(scales), _ptr(glob), int(p["fmt"])), [packed, scales, glob]


def moe_ffn(*, T, E, H, I, k, gate, up, down, x_bf16, ids, w, sh_I=0, sh_gate=None, sh_up=None,
            sh_down=None, act_mode=0, g1=1.0, g2=1.0, zero_experts=0, nthreads=0):
    """Expert FFN for every (token, slot) pair + weighted sum + shared expert, fp64 [T,H].
    Ids in [E, E + zero_experts) are zero-computation experts (they add w * x)."""
    lib = _load()
    keep = []
    projs = []
    for p in (gate, up, down, sh_gate, sh_up, sh_down):
        cp, kp = _proj(p)
        projs.append(cp)
        keep += kp
    x_bf16 = _as(x_bf16, np.uint16)
    ids = _as(ids, np.int32)
    w = _as(w, np.float64)
    out = np.zeros((T, H), np.float64)
    rc = lib.orc_moe_ffn(T, E, H, I, k, int(zero_experts), projs[0], projs[1], projs[2], int(sh_I), projs[3],
                         projs[4], projs[5], int(act_mode), float(g1), float(g2), _ptr(x_bf16),
                         _ptr(ids), _ptr(w), _ptr(out), int(nthreads))
    if rc != 0:
        raise ValueError("oracle moe_ffn: invalid arguments")
    return out
