"""MoeLayer: owns one layer's device buffers and calls the C ABI (marshalling only).

Weights are dicts of CUDA tensors ({packed, scales, globals, fmt}) laid out as include/moe.h
describes.  The layer prepares them once (moe_prepare_weights), keeps a workspace sized for
the largest token count seen, and runs route + FFN on the current CUDA stream with no host
synchronisation.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import capi


class MoeLayer:
    def __init__(self, *, E, H, I, top_k, scoring, gate, up, down, I_shared=0, sh_gate=None,
                 sh_up=None, sh_down=None, w_router=None, correction_bias=None, tid2eid=None,
                 renormalize=True, routed_scaling=1.0, act=capi.MOE_ACT_BF16, g_act1=1.0,
                 g_act2=1.0, zero_experts=0):
        self.E, self.H, self.I, self.top_k, self.I_shared = E, H, I, top_k, I_shared
        self.zero_experts = zero_experts
        self.scoring, self.renormalize, self.routed_scaling = scoring, renormalize, routed_scaling
        self.act, self.g_act1, self.g_act2 = act, g_act1, g_act2
        self.w_router, self.correction_bias, self.tid2eid = w_router, correction_bias, tid2eid
        self._weights = (gate, up, down, sh_gate, sh_up, sh_down)  # keep alive
        self.desc = capi.ffn_desc(E, H, I, top_k, I_shared, gate, up, down, sh_gate, sh_up, sh_down,
                                  zero_experts)
        self.handle = capi.moe_prepare_weights(self.desc)
        self._ws = None
        self._ws_host = None
        self._host_route = {}
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    @classmethod
    def from_inputs(cls, inp: dict, device="cuda"):
        """Build from a synth.make_inputs() dict (tensors moved to `device`)."""
        cfg = inp["cfg"]

        def dev(p):
            if p is None:
                return None
            return {k: (v.to(device).contiguous() if isinstance(v, torch.Tensor) else v)
                    for k, v in p.items()}

        opt = lambda key: inp[key].to(device).contiguous() if key in inp else None
        return cls(E=cfg.E, H=cfg.H, I=cfg.I, top_k=cfg.k, scoring=cfg.scoring,
                   gate=dev(inp["gate"]), up=dev(inp["up"]), down=dev(inp["down"]),
                   I_shared=cfg.I_shared, sh_gate=dev(inp.get("sh_gate")),
                   sh_up=dev(inp.get("sh_up")), sh_down=dev(inp.get("sh_down")),
                   w_router=opt("w_router"), correction_bias=opt("bias"), tid2eid=opt("tid2eid"),
                   renormalize=cfg.renorm, routed_scaling=cfg.scaling, act=cfg.act,
                   zero_experts=cfg.zero_experts)

    def close(self):
        if self.handle:
            capi.moe_release_weights(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def workspace(self, T: int) -> torch.Tensor:
        need = capi.moe_workspace_size(self.desc, T, self.act)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
        return self._ws

    def route(self, x=None, *, token_ids=None, logits_in=None, topk_ids=None, topk_w=None,
              logits_out=None, stream=None):
        T = (x.shape[0] if x is not None else
             token_ids.shape[0] if token_ids is not None else logits_in.shape[0])
        if topk_ids is None:
            topk_ids = torch.empty((T, self.top_k), dtype=torch.int32, device="cuda")
        if topk_w is None:
            topk_w = torch.empty((T, self.top_k), dtype=torch.float32, device="cuda")
        if (logits_out is None and logits_in is None and self.scoring != capi.MOE_SCORE_HASH):
            logits_out = torch.empty((T, self.E + self.zero_experts), dtype=torch.float32,
                                     device="cuda")
        capi.moe_route(T=T, E=self.E, H=self.H, top_k=self.top_k, scoring=self.scoring,
                       renormalize=self.renormalize, routed_scaling=self.routed_scaling, x=x,
                       w_router=None if logits_in is not None else self.w_router,
                       logits_in=logits_in, logits_out=logits_out,
                       correction_bias=self.correction_bias, tid2eid=self.tid2eid,
                       vocab=0 if self.tid2eid is None else self.tid2eid.shape[0],
                       token_ids=token_ids, topk_ids=topk_ids, topk_w=topk_w,
                       dev_status=self.status, stream=stream, zero_experts=self.zero_experts)
        return topk_ids, topk_w, logits_out

    def ffn(self, x, topk_ids, topk_w, out=None, stream=None):
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.bfloat16, device="cuda")
        capi.moe_ffn_forward(self.handle, T, self.act, self.g_act1, self.g_act2, x, topk_ids,
                             topk_w, out, self.workspace(T), dev_status=self.status, stream=stream)
        return out

    def forward(self, x=None, *, token_ids=None, logits_in=None, out=None, topk_ids=None,
                topk_w=None, logits_out=None, stream=None):
        """Route + FFN through moe_forward (one launch for a few tokens).
        Returns (out, topk_ids, topk_w, logits_out)."""
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.bfloat16, device="cuda")
        if topk_ids is None:
            topk_ids = torch.empty((T, self.top_k), dtype=torch.int32, device="cuda")
        if topk_w is None:
            topk_w = torch.empty((T, self.top_k), dtype=torch.float32, device="cuda")
        if (logits_out is None and logits_in is None and self.scoring != capi.MOE_SCORE_HASH):
            logits_out = torch.empty((T, self.E + self.zero_experts), dtype=torch.float32,
                                     device="cuda")
        d = capi.route_desc(T=T, E=self.E, H=self.H, top_k=self.top_k, scoring=self.scoring,
                            renormalize=self.renormalize, routed_scaling=self.routed_scaling,
                            w_router=None if logits_in is not None else self.w_router,
                            correction_bias=self.correction_bias, tid2eid=self.tid2eid,
                            vocab=0 if self.tid2eid is None else self.tid2eid.shape[0],
                            token_ids=token_ids, zero_experts=self.zero_experts)
        capi.moe_forward(self.handle, d, self.act, self.g_act1, self.g_act2, x, topk_ids, topk_w,
                         out, self.workspace(T), logits_in=logits_in, logits_out=logits_out,
                         dev_status=self.status, stream=stream)
        return out, topk_ids, topk_w, logits_out

    def forward_host(self, x_host, out_host, *, token_ids_host=None, topk_ids_host=None,
                     topk_w_host=None, stream=None):
        """Route + FFN on host buffers through moe_forward_host: x_host (and token_ids_host for
        hash routing) are copied in, out_host (and the ids / weights when given) copied back, all
        enqueued on the stream; the caller synchronises before reading the outputs."""
        T = x_host.shape[0]
        cached = self._host_route.get(T)
        if cached is None:
            d = capi.route_desc(T=T, E=self.E, H=self.H, top_k=self.top_k, scoring=self.scoring,
                                renormalize=self.renormalize, routed_scaling=self.routed_scaling,
                                w_router=self.w_router, correction_bias=self.correction_bias,
                                tid2eid=self.tid2eid,
                                vocab=0 if self.tid2eid is None else self.tid2eid.shape[0],
                                zero_experts=self.zero_experts)
            cached = self._host_route[T] = (d, capi.moe_workspace_size_host(self.desc, T, self.act))
        d, need = cached
        if self._ws_host is None or self._ws_host.numel() < need:
            self._ws_host = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
        capi.moe_forward_host(self.handle, d, self.act, self.g_act1, self.g_act2, x_host, out_host,
                              self._ws_host, token_ids_host=token_ids_host,
                              topk_ids_host=topk_ids_host, topk_w_host=topk_w_host,
                              dev_status=self.status, stream=stream)
        return out_host
