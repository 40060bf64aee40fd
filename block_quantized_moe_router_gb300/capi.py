"""ctypes binding of the C ABI in include/moe.h (argument marshalling only).

Every function here has the name of the C entry point it calls and does no arithmetic of its
own: it checks dtypes/shapes of torch tensors, passes their device pointers and the current
CUDA stream, and turns a nonzero moe_status_t into an exception.  If the CUDA library is
missing, loading fails loudly; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_WORKSPACE = range(5)
MOE_DEV_BAD_EXPERT_ID, MOE_DEV_BAD_TOKEN_ID, MOE_DEV_NONFINITE, MOE_DEV_TIMEOUT = 1, 2, 4, 8
MOE_SCORE_SOFTMAX, MOE_SCORE_SIGMOID, MOE_SCORE_HASH, MOE_SCORE_SQRTSOFTPLUS = 0, 1, 2, 3
MOE_SCORE_SOFTMAX_BIAS, MOE_SCORE_HASH_SQRTSOFTPLUS = 4, 5
MOE_FMT_NVFP4, MOE_FMT_MXFP4 = 0, 1
MOE_ACT_BF16, MOE_ACT_NVFP4 = 0, 1

# Every symbol include/moe.h declares.
EXPORTED = ["moe_route", "moe_workspace_size", "moe_prepare_weights", "moe_release_weights",
            "moe_ffn_forward", "moe_forward", "moe_workspace_size_host", "moe_forward_host",
            "moe_ffn_forward_noalloc", "moe_quantize_act_nvfp4",
            "moe_set_wait_limit", "moe_skew_barrier", "moe_profile_enable", "moe_profile_read",
            "moe_status_string"]


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {moe_status_string(status)} (status {status})")
        self.status = status


class moe_qtensor(ctypes.Structure):
    _fields_ = [("packed", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("globals", ctypes.c_void_p), ("fmt", ctypes.c_int32)]


class moe_ffn_desc(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("I_shared", ctypes.c_int32),
                ("gate", moe_qtensor), ("up", moe_qtensor), ("down", moe_qtensor),
                ("sh_gate", moe_qtensor), ("sh_up", moe_qtensor), ("sh_down", moe_qtensor),
                ("zero_experts", ctypes.c_int32)]


class moe_route_desc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("E", ctypes.c_int32), ("H", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("scoring", ctypes.c_int32),
                ("renormalize", ctypes.c_int32), ("routed_scaling", ctypes.c_float),
                ("w_router", ctypes.c_void_p), ("correction_bias", ctypes.c_void_p),
                ("tid2eid", ctypes.c_void_p), ("vocab", ctypes.c_int64),
                ("token_ids", ctypes.c_void_p), ("zero_experts", ctypes.c_int32)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libmoe_gb300.so; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.moe_status_string.argtypes = [ctypes.c_int]
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_route.argtypes = [ctypes.POINTER(moe_route_desc), vp, vp, vp, vp, vp, vp, vp]
    lib.moe_route.restype = ctypes.c_int
    lib.moe_workspace_size.argtypes = [ctypes.POINTER(moe_ffn_desc), i32, i32, ctypes.POINTER(sz)]
    lib.moe_workspace_size.restype = ctypes.c_int
    lib.moe_prepare_weights.argtypes = [ctypes.POINTER(moe_ffn_desc), ctypes.POINTER(vp), vp]
    lib.moe_prepare_weights.restype = ctypes.c_int
    lib.moe_release_weights.argtypes = [vp]
    lib.moe_release_weights.restype = ctypes.c_int
    lib.moe_ffn_forward.argtypes = [vp, i32, i32, f32, f32, vp, vp, vp, vp, vp, sz, vp, vp]
    lib.moe_ffn_forward.restype = ctypes.c_int
    lib.moe_forward.argtypes = [vp, ctypes.POINTER(moe_route_desc), i32, f32, f32, vp, vp, vp, vp,
                                vp, vp, vp, sz, vp, vp]
    lib.moe_forward.restype = ctypes.c_int
    lib.moe_workspace_size_host.argtypes = [ctypes.POINTER(moe_ffn_desc), i32, i32, ctypes.POINTER(sz)]
    lib.moe_workspace_size_host.restype = ctypes.c_int
    lib.moe_forward_host.argtypes = [vp, ctypes.POINTER(moe_route_desc), i32, f32, f32, vp, vp, vp,
                                     vp, vp, vp, sz, vp, vp]
    lib.moe_forward_host.restype = ctypes.c_int
    lib.moe_ffn_forward_noalloc.argtypes = [vp, i32, i32, f32, f32, vp, vp, vp, vp, vp, vp]
    lib.moe_ffn_forward_noalloc.restype = ctypes.c_int
    lib.moe_quantize_act_nvfp4.argtypes = [vp, i64, i64, f32, vp, vp, vp]
    lib.moe_quantize_act_nvfp4.restype = ctypes.c_int
    lib.moe_set_wait_limit.argtypes = [vp, ctypes.c_uint64]
    lib.moe_set_wait_limit.restype = ctypes.c_int
    lib.moe_skew_barrier.argtypes = [vp, vp]
    lib.moe_skew_barrier.restype = ctypes.c_int
    lib.moe_profile_enable.argtypes = [vp, ctypes.c_uint32]
    lib.moe_profile_enable.restype = ctypes.c_int
    lib.moe_profile_read.argtypes = [vp, ctypes.POINTER(ctypes.c_float)]
    lib.moe_profile_read.restype = ctypes.c_int
    _lib = lib
    return lib


def moe_status_string(status: int) -> str:
    return load_library().moe_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where)


def _dptr(t: Optional[torch.Tensor], dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _hptr(t: Optional[torch.Tensor], dtype, name="tensor"):
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def qtensor(p: Optional[dict]) -> moe_qtensor:
    """Weight dict {packed, scales, globals, fmt} of CUDA tensors -> moe_qtensor."""
    if p is None:
        return moe_qtensor(None, None, None, 0)
    return moe_qtensor(_dptr(p["packed"], torch.uint8, "packed"),
                       _dptr(p["scales"], torch.uint8, "scales"),
                       _dptr(p.get("globals"), torch.float32, "globals"), int(p["fmt"]))


def ffn_desc(E, H, I, top_k, I_shared, gate, up, down, sh_gate=None, sh_up=None, sh_down=None,
             zero_experts=0):
    return moe_ffn_desc(E, H, I, top_k, I_shared, qtensor(gate), qtensor(up), qtensor(down),
                        qtensor(sh_gate), qtensor(sh_up), qtensor(sh_down), int(zero_experts))


def route_desc(*, T, E, H, top_k, scoring, renormalize, routed_scaling, w_router=None,
               correction_bias=None, tid2eid=None, vocab=0, token_ids=None,
               zero_experts=0) -> moe_route_desc:
    return moe_route_desc(int(T), int(E), int(H), int(top_k), int(scoring), int(bool(renormalize)),
                          float(routed_scaling), _dptr(w_router, torch.bfloat16, "w_router"),
                          _dptr(correction_bias, torch.float32, "correction_bias"),
                          _dptr(tid2eid, torch.int64, "tid2eid"), int(vocab),
                          _dptr(token_ids, torch.int32, "token_ids"), int(zero_experts))


def moe_route(*, T, E, H, top_k, scoring, renormalize, routed_scaling, x=None, w_router=None,
              logits_in=None, logits_out=None, correction_bias=None, tid2eid=None, vocab=0,
              token_ids=None, topk_ids, topk_w, dev_status=None, stream=None, zero_experts=0):
    lib = load_library()
    d = route_desc(T=T, E=E, H=H, top_k=top_k, scoring=scoring, renormalize=renormalize,
                   routed_scaling=routed_scaling, w_router=w_router,
                   correction_bias=correction_bias, tid2eid=tid2eid, vocab=vocab,
                   token_ids=token_ids, zero_experts=zero_experts)
    st = lib.moe_route(ctypes.byref(d), _dptr(x, torch.bfloat16, "x"),
                       _dptr(logits_in, torch.float32, "logits_in"),
                       _dptr(logits_out, torch.float32, "logits_out"),
                       _dptr(topk_ids, torch.int32, "topk_ids"), _dptr(topk_w, torch.float32, "topk_w"),
                       _dptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(st, "moe_route")


def moe_workspace_size(desc: moe_ffn_desc, T: int, act: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().moe_workspace_size(ctypes.byref(desc), int(T), int(act), ctypes.byref(n)),
           "moe_workspace_size")
    return int(n.value)


def moe_prepare_weights(desc: moe_ffn_desc, stream=None) -> int:
    h = ctypes.c_void_p(None)
    _check(load_library().moe_prepare_weights(ctypes.byref(desc), ctypes.byref(h), _stream(stream)),
           "moe_prepare_weights")
    return h.value


def moe_release_weights(handle: int):
    _check(load_library().moe_release_weights(ctypes.c_void_p(handle)), "moe_release_weights")


def moe_ffn_forward(handle: int, T: int, act: int, g_act1: float, g_act2: float, x, topk_ids,
                    topk_w, out, workspace, dev_status=None, stream=None):
    st = load_library().moe_ffn_forward(
        ctypes.c_void_p(handle), int(T), int(act), float(g_act1), float(g_act2),
        _dptr(x, torch.bfloat16, "x"), _dptr(topk_ids, torch.int32, "topk_ids"),
        _dptr(topk_w, torch.float32, "topk_w"), _dptr(out, torch.bfloat16, "out"),
        _dptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        _dptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(st, "moe_ffn_forward")


def moe_forward(handle: int, route: moe_route_desc, act: int, g_act1: float, g_act2: float, x,
                topk_ids, topk_w, out, workspace, logits_in=None, logits_out=None,
                dev_status=None, stream=None):
    """Route + expert FFN in one call (one persistent launch for a few tokens)."""
    st = load_library().moe_forward(
        ctypes.c_void_p(handle), ctypes.byref(route), int(act), float(g_act1), float(g_act2),
        _dptr(x, torch.bfloat16, "x"), _dptr(logits_in, torch.float32, "logits_in"),
        _dptr(logits_out, torch.float32, "logits_out"), _dptr(topk_ids, torch.int32, "topk_ids"),
        _dptr(topk_w, torch.float32, "topk_w"), _dptr(out, torch.bfloat16, "out"),
        _dptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        _dptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(st, "moe_forward")


def moe_workspace_size_host(desc: moe_ffn_desc, T: int, act: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().moe_workspace_size_host(ctypes.byref(desc), int(T), int(act),
                                                  ctypes.byref(n)), "moe_workspace_size_host")
    return int(n.value)


def moe_forward_host(handle: int, route: moe_route_desc, act: int, g_act1: float, g_act2: float,
                     x_host, out_host, workspace, token_ids_host=None, topk_ids_host=None,
                     topk_w_host=None, dev_status=None, stream=None):
    """moe_forward on host buffers (CPU tensors, pinned for asynchronous copies): the copies in
    and out are enqueued on the stream with the forward; synchronise before reading out_host."""
    st = load_library().moe_forward_host(
        ctypes.c_void_p(handle), ctypes.byref(route), int(act), float(g_act1), float(g_act2),
        _hptr(x_host, torch.bfloat16, "x_host"), _hptr(token_ids_host, torch.int32, "token_ids_host"),
        _hptr(out_host, torch.bfloat16, "out_host"), _hptr(topk_ids_host, torch.int32, "topk_ids_host"),
        _hptr(topk_w_host, torch.float32, "topk_w_host"),
        _dptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        _dptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(st, "moe_forward_host")


def moe_ffn_forward_noalloc(handle: int, T: int, act: int, g_act1: float, g_act2: float, x,
                            topk_ids, topk_w, out, dev_status=None, stream=None):
    """moe_ffn_forward with the library's static device workspace (no caller allocation)."""
    st = load_library().moe_ffn_forward_noalloc(
        ctypes.c_void_p(handle), int(T), int(act), float(g_act1), float(g_act2),
        _dptr(x, torch.bfloat16, "x"), _dptr(topk_ids, torch.int32, "topk_ids"),
        _dptr(topk_w, torch.float32, "topk_w"), _dptr(out, torch.bfloat16, "out"),
        _dptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(st, "moe_ffn_forward_noalloc")


def moe_quantize_act_nvfp4(x, g: float, packed, scales, stream=None):
    rows, K = x.shape
    st = load_library().moe_quantize_act_nvfp4(
        _dptr(x, torch.bfloat16, "x"), int(rows), int(K), float(g),
        _dptr(packed, torch.uint8, "packed"), _dptr(scales, torch.uint8, "scales"), _stream(stream))
    _check(st, "moe_quantize_act_nvfp4")


def moe_set_wait_limit(handle: int, cycles: int):
    _check(load_library().moe_set_wait_limit(ctypes.c_void_p(handle), int(cycles)),
           "moe_set_wait_limit")


def moe_skew_barrier(handle: int, stream=None):
    _check(load_library().moe_skew_barrier(ctypes.c_void_p(handle), _stream(stream)),
           "moe_skew_barrier")


PHASE_DISPATCH, PHASE_GATE_UP, PHASE_DOWN, PHASE_COMBINE = 0, 1, 2, 3


def moe_profile_enable(handle: int, mask: int):
    _check(load_library().moe_profile_enable(ctypes.c_void_p(handle), int(mask)), "moe_profile_enable")


def moe_profile_read(handle: int):
    ms = (ctypes.c_float * 4)()
    _check(load_library().moe_profile_read(ctypes.c_void_p(handle), ms), "moe_profile_read")
    return [float(v) for v in ms]
