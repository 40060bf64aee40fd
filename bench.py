"""Benchmark of the MoE FFN block (router -> top-K -> NVFP4/MXFP4 experts -> combine).

One step = one MoE layer forward (moe_forward: route + FFN) over one batch of T synthetic
tokens.  Steps cycle through L replicas of the layer's weights (distinct device copies, as the
layers of a model would be) with L * touched-bytes >= 4 * L2, so every step streams its expert
weights from HBM.  One CUDA graph holds one step of each replica in turn (as a serving engine
captures the layers of a decode step in one graph) and is replayed; single-step graphs make
up any remainder, so the timed region is exactly K steps, between a barrier + device
synchronisation on both sides, timed with CUDA events on the launching stream, max over
ranks.

Prints one JSON line: MoE-layer tokens/s (whole job), the roofline of the dominant kernel
(algorithmic bytes / its CUDA-event duration measured inside the timed region), the clocks
seen during the timed region, an end-to-end figure through the public API with host buffers,
and the CPU oracle's throughput on a bounded sample.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--config dec1] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from block_quantized_moe_router_gb300 import synth  # noqa: E402

METRIC = "MoE-layer tokens/s and achieved HBM GB/s or FP4 TFLOP/s vs GB300 peak"
DEFAULT_CONFIG = "dec1"
FALLBACK_HBM_GBS = 6800.0

# ncu DRAM traffic (read + write bytes per launch) of the dominant kernel, keyed by workload,
# with the hash of that kernel's sources when it was captured; reported only while it matches.
KERNEL_SOURCES = {
    "decode": ("decode_kernel.cuh", "decode_t1.cu", "topk.cuh", "frag.cuh", "common.cuh"),
    "tc": ("prefill_tc.cu", "tc_ptx.cuh", "common.cuh"),
    "mma": ("ffn.cu", "frag.cuh", "common.cuh"),
}
TRAFFIC = {"dec1": (21877760 + 1536, "df65e1498ea2565c")}  # profiles/dec_fused_dec1.md


def kernel_source_hash(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "block_quantized_moe_router_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


FALLBACK_BF16_TFLOPS = 1900.0
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense ratio (13.5 vs 2.25 PFLOP/s)


def measured_peaks():
    """(HBM GB/s, dense bf16 TFLOP/s burst, source) from MEASURED_PEAKS.json, else fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    hbm, bf16, src = FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"
    try:
        with open(path) as fh:
            d = json.load(fh)
        for key in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs"):
            if key in d:
                hbm, src = float(d[key]), "measured"
                break
        for key in ("bf16_tflops", "bf16_TFLOPs"):
            if key in d:
                bf16 = float(d[key])
                break
    except Exception:
        pass
    return hbm, bf16, src


# ------------------------------------------------------------------------------------------
# multi-rank helpers (one process per GPU; each rank runs its own replica on its own tokens)
# ------------------------------------------------------------------------------------------
def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise max of per-rank timings (the slowest rank sets the job's time)."""
    if dist is None or not dist.is_initialized():
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def auto_steps(step_s, replicas, target_s=1.0, floor=2000, cap=2_000_000):
    """Timed steps for about target_s of device time, given the seconds one step took in the
    warm-up: at least floor, at most cap, a multiple of the replica count."""
    try:
        n = int(math.ceil(target_s / step_s))
    except (ValueError, OverflowError, ZeroDivisionError):
        n = floor
    n = min(cap, max(floor, n))
    r = max(1, int(replicas))
    return -(-n // r) * r


def job_tokens_per_s(tokens_per_rank, world, seconds):
    """Whole-job throughput under weak scaling: every rank processed its own batch."""
    return tokens_per_rank * world / seconds


# ------------------------------------------------------------------------------------------
# clocks
# ------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, cmd=("nvidia-smi",)):
        self.gpu = gpu_index
        self.cmd = list(cmd)
        self.proc = None
        self.path = None
        self.marks = []

    def start(self):
        self.marks = []
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                self.cmd + ["-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            os.unlink(self.path)

    def mark(self):
        """Notes how many samples have been written so far; two marks bound the timed region."""
        n = 0
        try:
            if self.proc is not None:
                with open(self.path) as fh:
                    n = sum(1 for line in fh if line.endswith("\n"))
        except Exception:
            n = 0
        self.marks.append(n)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        with open(self.path) as fh:
            lines = fh.read().splitlines()
        os.unlink(self.path)
        # the samples written between the two marks, if any landed there (nvidia-smi may
        # buffer its output); otherwise every sample of the run
        inside = len(self.marks) >= 2 and self.marks[1] > self.marks[0]
        window = lines[self.marks[0]:self.marks[1]] if inside else lines
        rows = []
        for line in window:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows),
                "window": "timed region" if inside else "whole run"}


# ------------------------------------------------------------------------------------------
# workload accounting
# ------------------------------------------------------------------------------------------
def proj_bytes(N, K, fmt):
    sv = 16 if fmt == synth.FMT_NVFP4 else 32
    return N * K // 2 + N * K // sv + (4 if fmt == synth.FMT_NVFP4 else 0)


def step_bytes(cfg, n_touched):
    """Algorithmic HBM bytes of one layer step (touched experts only)."""
    H, I, Is = cfg.H, cfg.I, cfg.I_shared
    gate_up = 2 * proj_bytes(I, H, cfg.fmt)
    down = proj_bytes(H, I, cfg.fmt)
    sh_gate_up = 2 * proj_bytes(Is, H, cfg.shared_fmt) if Is else 0
    sh_down = proj_bytes(H, Is, cfg.shared_fmt) if Is else 0
    router = cfg.E * H * 2 if cfg.scoring != synth.SCORE_HASH else cfg.T * cfg.k * 8
    acts = cfg.T * H * 2 * 2
    pairs = cfg.T * cfg.k
    return {"gate_up": n_touched * gate_up + sh_gate_up + cfg.T * H * 2,
            "total": n_touched * (gate_up + down) + sh_gate_up + sh_down + router + acts,
            "gate_up_flops": 2 * 2 * I * H * pairs + (2 * 2 * Is * H * cfg.T if Is else 0),
            "flops": 2 * 3 * I * H * pairs + (2 * 3 * Is * H * cfg.T if Is else 0)
            + (2 * cfg.T * H * cfg.E if cfg.scoring != synth.SCORE_HASH else 0)}


def is_decode(cfg):
    """The few-token case that runs as one persistent launch (route + FFN)."""
    return cfg.T <= 8 and cfg.T * cfg.k <= 64 and cfg.act == synth.ACT_BF16


# ------------------------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline)
# ------------------------------------------------------------------------------------------
def oracle_step(cfg, inp_np, tokens, n_threads=0):
    """One oracle layer pass over `tokens` (route + expert FFN + combine)."""
    import oracle
    x = inp_np["x"][tokens]
    if cfg.scoring == synth.SCORE_HASH:
        r = oracle.route(T=len(tokens), E=cfg.E, k=cfg.k, scoring=2, scaling=cfg.scaling,
                         tid2eid=inp_np["tid2eid"], token_ids=inp_np["token_ids"][tokens],
                         vocab=cfg.vocab, nthreads=n_threads)
    else:
        r = oracle.route(T=len(tokens), E=cfg.E, k=cfg.k, scoring=cfg.scoring, renorm=cfg.renorm,
                         scaling=cfg.scaling, x_bf16=x, w_router_bf16=inp_np["w_router"],
                         bias=inp_np.get("bias"), nthreads=n_threads)
    return oracle.moe_ffn(T=len(tokens), E=cfg.E, H=cfg.H, I=cfg.I, k=cfg.k, gate=inp_np["gate"],
                          up=inp_np["up"], down=inp_np["down"], x_bf16=x, ids=r["ids"], w=r["w"],
                          sh_I=cfg.I_shared, sh_gate=inp_np.get("sh_gate"), sh_up=inp_np.get("sh_up"),
                          sh_down=inp_np.get("sh_down"), act_mode=cfg.act, nthreads=n_threads)


def host_inputs(cfg, seed):
    inp = synth.make_inputs(cfg, seed=seed, device="cuda" if torch.cuda.is_available() else "cpu")
    d = {"x": synth.bf16_bits(inp["x"])}
    if "w_router" in inp:
        d["w_router"] = synth.bf16_bits(inp["w_router"])
    for key in ("bias", "tid2eid", "token_ids"):
        if key in inp:
            d[key] = inp[key].cpu().numpy()
    for key in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down"):
        if key in inp:
            d[key] = synth.to_numpy_proj(inp[key])
    return inp, d


def cpu_baseline(cfg, inp_np, budget_s=10.0):
    """Oracle tokens/s on the host cores over a bounded sample of the workload."""
    import oracle
    oracle.build()
    threads = oracle.hardware_threads()
    # one of the workload's tokens per host thread (the oracle threads over tokens)
    n_tok = max(1, threads)
    tokens = np.arange(n_tok) % cfg.T
    t0 = time.perf_counter()
    done = 0
    while True:
        oracle_step(cfg, inp_np, tokens)
        done += len(tokens)
        if time.perf_counter() - t0 >= budget_s:  # the same tokens again until the budget is spent
            break
    dt = time.perf_counter() - t0
    return {"value": done / dt, "unit": "tokens/s", "cores": min(threads, len(tokens)), "kind": "oracle",
            "sample": f"{done} tokens of workload {cfg.name} in batches of {n_tok}, {dt:.1f} s"}


def run_reference(args, cfg):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    _, inp_np = host_inputs(cfg, seed=0)
    tokens_all = np.arange(cfg.T)
    # size each step's sample so that warmup + steps fit in about two minutes
    t0 = time.perf_counter()
    oracle_step(cfg, inp_np, tokens_all[:1])
    t_tok = time.perf_counter() - t0
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    n_tok = int(max(1, min(cfg.T, per_step_budget // max(t_tok, 1e-6))))
    sample = tokens_all[:n_tok]
    for _ in range(args.warmup):
        oracle_step(cfg, inp_np, sample)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(cfg, inp_np, sample)
    dt = (time.perf_counter() - t0) / args.steps
    value = n_tok / dt
    threads = min(oracle.hardware_threads(), n_tok)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3 * cfg.T / n_tok, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "I": cfg.I, "E": cfg.E,
                       "top_k": cfg.k, "I_shared": cfg.I_shared},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": f"{n_tok} of {cfg.T} tokens per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------
def run_ours(args, cfg):
    from block_quantized_moe_router_gb300 import build, capi
    from block_quantized_moe_router_gb300.layer import MoeLayer

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    build.build()
    capi.load_library()
    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 0) or 128 * 2 ** 20

    inp = synth.make_inputs(cfg, seed=rank, device="cuda")
    base = MoeLayer.from_inputs(inp)
    x = inp["x"].cuda()
    tok = inp["token_ids"].cuda() if "token_ids" in inp else None
    T = cfg.T
    ids0, _, _ = base.route(x, token_ids=tok)
    torch.cuda.synchronize()
    touched = int(torch.unique(ids0[ids0 >= 0]).numel())
    nbytes = step_bytes(cfg, touched)
    replicas = max(1, math.ceil(4 * l2 / nbytes["total"]))
    if args.replicas:
        replicas = args.replicas

    layers = [base]
    for _ in range(replicas - 1):
        clone = {k: ({kk: (vv.clone() if isinstance(vv, torch.Tensor) else vv)
                      for kk, vv in v.items()} if isinstance(v, dict) else v)
                 for k, v in inp.items()}
        layers.append(MoeLayer.from_inputs(clone))
    bufs = []
    for layer in layers:
        layer.workspace(T)
        bufs.append(dict(ids=torch.empty((T, cfg.k), dtype=torch.int32, device="cuda"),
                         w=torch.empty((T, cfg.k), dtype=torch.float32, device="cuda"),
                         logits=torch.empty((T, cfg.E), dtype=torch.float32, device="cuda"),
                         out=torch.empty((T, cfg.H), dtype=torch.bfloat16, device="cuda")))
    # time the dominant kernel live in one replica only: its event nodes break the programmatic
    # launch chain of that replica's steps, the other replicas run undisturbed
    capi.moe_profile_enable(layers[0].handle, 1 << capi.PHASE_GATE_UP)

    stream = torch.cuda.Stream()
    graphs = []
    def step(layer, b):  # one layer step through the public API: route + FFN in one call
        layer.forward(x, token_ids=tok, out=b["out"], topk_ids=b["ids"], topk_w=b["w"],
                      logits_out=None if tok is not None else b["logits"])

    # One graph holds one step of every weight replica in turn (as a serving engine captures
    # all layers of a decode step in one graph); single-replica graphs make up the remainder
    # so that exactly `steps` layer steps run in the timed region.
    with torch.cuda.stream(stream):
        for layer, b in zip(layers, bufs):   # one eager pass per replica before capture
            step(layer, b)
        stream.synchronize()
        for layer, b in zip(layers, bufs):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(layer, b)
            graphs.append(g)
        cycle = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cycle, stream=stream):
            for layer, b in zip(layers, bufs):
                step(layer, b)
    torch.cuda.synchronize()

    def run_steps(first, n):
        """Layer steps first .. first + n - 1 (replica i % replicas), as graph replays."""
        i = first
        while i < first + n:
            if i % replicas == 0 and first + n - i >= replicas:
                cycle.replay()
                i += replicas
            else:
                graphs[i % replicas].replay()
                i += 1

    def barrier():
        if dist is not None:
            dist.barrier()

    clocks = ClockSampler(local)
    clocks.start()
    with torch.cuda.stream(stream):
        w0 = torch.cuda.Event(enable_timing=True)
        w1 = torch.cuda.Event(enable_timing=True)
        w0.record(stream)
        run_steps(0, args.warmup)
        w1.record(stream)
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        if args.steps is None:  # about one second of timed work, the same on every rank
            try:
                steps = auto_steps(w0.elapsed_time(w1) * 1e-3 / args.warmup, replicas)
            except Exception:  # no usable warm-up timing: the fixed default
                steps = 2000
            args.steps = int(max_over_ranks([steps], dist, device="cuda")[0])
        barrier()
        torch.cuda.synchronize()
        clocks.mark()
        ev0.record(stream)
        run_steps(args.warmup, args.steps)
        ev1.record(stream)
    torch.cuda.synchronize()
    clocks.mark()
    barrier()
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1) / args.steps
    # dominant kernel: the last execution of replica 0's gate+up GEMM (inside the timed region
    # when steps >= replicas)
    dom_ms = float(capi.moe_profile_read(layers[0].handle)[capi.PHASE_GATE_UP])
    ms, dom_ms = max_over_ranks([ms, dom_ms], dist, device="cuda")
    ok = all(torch.equal(bufs[0]["out"], b["out"]) for b in bufs[1:])

    # end to end through the public API with host buffers: H2D of x, route + FFN, D2H of out
    e2e_s = float("nan")
    x_host = inp["x"].pin_memory()
    out_host = torch.empty((T, cfg.H), dtype=torch.bfloat16).pin_memory()
    tok_host = inp["token_ids"].pin_memory() if tok is not None else None
    x_dev = torch.empty_like(x)
    tok_dev = torch.empty_like(tok) if tok is not None else None
    e2e_steps = max(3, min(args.steps, 200)) if args.e2e else 0
    e2e_mode = None

    def e2e_step(layer, b):  # H2D of the step's inputs, route + FFN, D2H of its output
        x_dev.copy_(x_host, non_blocking=True)
        if tok_dev is not None:
            tok_dev.copy_(tok_host, non_blocking=True)
        layer.forward(x_dev, token_ids=tok_dev, out=b["out"], topk_ids=b["ids"], topk_w=b["w"],
                      logits_out=None if tok is not None else b["logits"])
        out_host.copy_(b["out"], non_blocking=True)

    if args.e2e:
        # as a serving loop runs it: each step (copies included) captured once as a CUDA graph
        # from the public-API calls and replayed, the host waiting for every step's result
        e2e_graphs = []
        try:
            with torch.cuda.stream(stream):
                for layer, b in zip(layers, bufs):
                    e2e_step(layer, b)
                stream.synchronize()
                for layer, b in zip(layers, bufs):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        e2e_step(layer, b)
                    e2e_graphs.append(g)
            e2e_mode = "graph"
        except RuntimeError:
            e2e_graphs = []
            e2e_mode = "eager"
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for i in range(e2e_steps + args.warmup):
                if i == args.warmup:
                    barrier()
                    torch.cuda.synchronize()
                    t0 = time.perf_counter()
                if e2e_graphs:
                    e2e_graphs[i % replicas].replay()
                else:
                    e2e_step(layers[i % replicas], bufs[i % replicas])
                stream.synchronize()
        e2e_s = (time.perf_counter() - t0) / e2e_steps
    e2e_s = max_over_ranks([e2e_s], dist, device="cuda")[0]
    h2d = T * cfg.H * 2 + (T * 4 if tok is not None else 0)
    d2h = T * cfg.H * 2

    if rank == 0:
        peak, bf16_peak, peak_kind = measured_peaks()
        dec = is_decode(cfg)
        # dominant kernel: the whole-layer persistent kernel for a few tokens, else gate+up
        dom_bytes = nbytes["total"] if dec else nbytes["gate_up"]
        dom_flops = nbytes["flops"] if dec else nbytes["gate_up_flops"]
        dom_name = ("dec_fused_kernel (route + FFN)" if dec else "gate+up GEMM (" +
                    ("tc_gemm_kernel" if cfg.act == synth.ACT_NVFP4 else "expert_mma_kernel") + ")")
        achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
        fp4_peak = bf16_peak * FP4_OVER_BF16
        tflops = dom_flops / (dom_ms * 1e-3) / 1e12
        layer_gbs = nbytes["total"] / (ms * 1e-3) / 1e9
        src = kernel_source_hash(KERNEL_SOURCES["decode" if dec else
                                                "tc" if cfg.act == synth.ACT_NVFP4 else "mma"])
        tr = TRAFFIC.get(cfg.name)
        traffic = tr[0] if tr and tr[1] == src else None
        line = {
            "metric": METRIC, "value": job_tokens_per_s(T, world, ms * 1e-3), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "nvfp4 weights, f16 mma / f32 accumulate" if cfg.act == synth.ACT_BF16
            else "nvfp4 weights and activations, f32 accumulate",
            "data": "synthetic",
            "config": {"workload": cfg.name, "T": T, "H": cfg.H, "I": cfg.I, "E": cfg.E,
                       "top_k": cfg.k, "I_shared": cfg.I_shared, "replicas": replicas,
                       "l2_policy": f"inputs larger than L2: {replicas} weight replicas cycled, "
                                    f"{replicas * nbytes['total'] / 1e6:.0f} MB touched per cycle",
                       "launch": f"CUDA graph of {replicas} layer steps (one per replica), replayed",
                       "touched_experts": touched},
            "gpu_launches": args.steps * launches_per_step(cfg),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic, "kernel": dom_name,
                         "bytes_per_launch": dom_bytes, "launch_ms": dom_ms,
                         "peak_source": peak_kind},
            "tensor_view": {"achieved_tflops": tflops,
                            "peak_tflops": fp4_peak if cfg.act == synth.ACT_NVFP4 else bf16_peak,
                            "frac": tflops / (fp4_peak if cfg.act == synth.ACT_NVFP4 else bf16_peak),
                            "dtype": "nvfp4 x nvfp4" if cfg.act == synth.ACT_NVFP4 else "f16 mma",
                            "flops_per_launch": dom_flops,
                            "peak_source": peak_kind + " bf16 x nominal fp4/bf16 ratio"
                            if cfg.act == synth.ACT_NVFP4 else peak_kind},
            "layer_roofline": {"achieved": layer_gbs, "peak": peak, "unit": "GB/s",
                               "frac": layer_gbs / peak, "bytes_per_step": nbytes["total"]},
            "clocks": clk,
            "e2e": {"value": job_tokens_per_s(T, world, e2e_s), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "mode": e2e_mode, "ms_per_step": e2e_s * 1e3},
            "replica_outputs_equal": ok,
            "kernel_source": src,
        }
        if args.cpu_baseline:
            _, inp_np = host_inputs_from(inp)
            line["cpu_baseline"] = cpu_baseline(cfg, inp_np, budget_s=args.cpu_budget)
        print(json.dumps(line), flush=True)
    for layer in layers:
        layer.close()
    if dist is not None:
        dist.destroy_process_group()


def host_inputs_from(inp):
    d = {"x": synth.bf16_bits(inp["x"])}
    if "w_router" in inp:
        d["w_router"] = synth.bf16_bits(inp["w_router"])
    for key in ("bias", "tid2eid", "token_ids"):
        if key in inp:
            d[key] = inp[key].cpu().numpy()
    for key in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down"):
        if key in inp:
            d[key] = synth.to_numpy_proj(inp[key])
    return inp, d


def launches_per_step(cfg):
    """Kernels one step launches.  A few tokens: one persistent kernel.  Otherwise router
    GEMM + top-K (or the hash lookup), then the FFN: tcgen05 path -- histogram, scan, scatter,
    token quantizer, row gather, gate+up GEMM, down GEMM, combine; mma path -- prep, gate+up,
    down, combine."""
    if is_decode(cfg):
        return 1
    route = 1 if cfg.scoring == synth.SCORE_HASH else 2
    return route + (8 if cfg.act == synth.ACT_NVFP4 else 4)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: about one second of device time, at least 2000)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=list(synth.CONFIGS))
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--replicas", type=int, default=0,
                    help="weight replicas to cycle (default: enough to exceed 4x L2)")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    cfg = synth.CONFIGS[args.config]
    if args.impl == "reference":
        if args.steps is None:
            args.steps = 20
        run_reference(args, cfg)
    else:
        run_ours(args, cfg)


if __name__ == "__main__":
    main()
