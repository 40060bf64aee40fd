"""Benchmark of the MoE FFN block (router -> top-K -> NVFP4/MXFP4 experts -> combine).

One step = one MoE layer forward (moe_forward: route + FFN) over one batch of T synthetic
tokens.  Steps cycle through L replicas of the layer's weights (distinct device copies, as the
layers of a model would be) with L * touched-bytes >= 4 * L2, so every step streams its expert
weights from HBM.  One CUDA graph holds one step of each replica in turn (as a serving engine
captures the layers of a step in one graph), repeated to at least 4 steps, and is replayed;
single-step graphs make up any remainder, so a timed region is exactly K steps, between a
barrier + device synchronisation on
both sides, timed with CUDA events on the launching stream, max over ranks.  When K steps take
less than about a second the region is repeated (each repetition again exactly K steps) and the
median region is reported, so that the clock sampler sees the load.

The headline workload is the 4096-token prefill (the largest configuration); the same run adds
one line per other workload (dec1, dec8, hash64, pre32768) under "per_workload".  Each line
carries MoE-layer tokens/s (whole job), the roofline of the dominant kernel (algorithmic bytes
or FLOPs / its CUDA-event duration inside the timed regions), the clocks seen during the timed
regions, an end-to-end figure through the public API with host buffers, and (headline only) the
CPU oracle's throughput on a bounded sample.  The per-workload lines time regions of whole cycles
over their weight replicas and of at least --min-region-ms of work (a given step count is rounded
up accordingly); the headline times exactly the given K.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--config pre4096] [--impl reference]
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
DEFAULT_CONFIG = "pre4096"
PER_WORKLOAD = ("dec1", "dec8", "hash64", "pre32768")
FALLBACK_HBM_GBS = 6800.0

# ncu DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum per launch) of each workload's
# dominant kernel, with the hash of that kernel's sources when it was captured; reported only
# while the hash still matches (null once the kernel has changed).
KERNEL_SOURCES = {
    "decode": ("decode_kernel.cuh", "decode_t1.cu", "decode.cu", "topk.cuh", "frag.cuh",
               "common.cuh"),
    "tc": ("prefill_tc.cu", "tc_ptx.cuh", "quant.cuh", "common.cuh"),
    "mma": ("ffn.cu", "frag.cuh", "quant.cuh", "common.cuh"),
}
TRAFFIC = {  # one-pass captures at full size (the commands are in the profile summaries)
    "pre4096": (4597807616, "376201d900e9e811"),
    "pre32768": (5849034496, "376201d900e9e811"),
    "dec1": (21881344, "047b93c02bb9da69"),
    "dec8": (1270784256, "047b93c02bb9da69"),
    "hash64": (585473024, "072a5ab91b57aa02"),
}


def captured_traffic(workload: str, src_hash: str):
    """DRAM bytes per launch of the workload's dominant kernel from its ncu capture, or None when
    there is none or the kernel's sources have changed since (their hash differs)."""
    tr = TRAFFIC.get(workload)
    return tr[0] if tr and tr[1] == src_hash else None


def kernel_source_hash(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "block_quantized_moe_router_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


FALLBACK_BF16_TFLOPS = 1900.0
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense ratio (13.5 vs 2.25 PFLOP/s)


FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0


def measured_peaks():
    """HBM GB/s, dense bf16 TFLOP/s (burst and sustained) and their source, from
    MEASURED_PEAKS.json, else the fallback figures."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    out = {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
           "bf16_tflops_sustained": FALLBACK_BF16_TFLOPS_SUSTAINED, "source": "fallback"}
    try:
        with open(path) as fh:
            d = json.load(fh)
        if "hbm_gbs" in d:
            out["hbm_gbs"], out["source"] = float(d["hbm_gbs"]), "measured"
        for key in ("bf16_tflops", "bf16_tflops_sustained"):
            if key in d:
                out[key] = float(d[key])
    except Exception:
        pass
    return out


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
    hash_kw = {}
    if cfg.scoring in (synth.SCORE_HASH, synth.SCORE_HASH_SQRTSOFTPLUS):
        hash_kw = dict(tid2eid=inp_np["tid2eid"], token_ids=inp_np["token_ids"][tokens],
                       vocab=cfg.vocab)
    if cfg.scoring == synth.SCORE_HASH:
        r = oracle.route(T=len(tokens), E=cfg.E, k=cfg.k, scoring=2, scaling=cfg.scaling,
                         nthreads=n_threads, **hash_kw)
    else:
        r = oracle.route(T=len(tokens), E=cfg.E, k=cfg.k, scoring=cfg.scoring, renorm=cfg.renorm,
                         scaling=cfg.scaling, x_bf16=x, w_router_bf16=inp_np["w_router"],
                         bias=inp_np.get("bias"), nthreads=n_threads, **hash_kw)
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
    # size each step's sample so that warmup + steps fit in about two minutes: the oracle
    # threads over tokens, so a step of n * threads tokens takes about n one-token times
    t0 = time.perf_counter()
    oracle_step(cfg, inp_np, tokens_all[:1])
    t_tok = time.perf_counter() - t0
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    per_thread = int(per_step_budget // max(t_tok, 1e-6))
    n_tok = int(max(1, min(cfg.T, max(1, per_thread) * (oracle.hardware_threads() if per_thread else 1))))
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
def launches_per_step(cfg):
    """Kernels one step launches.  A few tokens: one persistent kernel.  Otherwise router
    GEMM + top-K (or the hash lookup), then the FFN: tcgen05 path -- histogram, scan, scatter,
    token quantizer, row gather, gate+up GEMM, down GEMM, combine; mma path -- prep, gate+up,
    down, combine."""
    if is_decode(cfg):
        return 1
    route = 1 if cfg.scoring == synth.SCORE_HASH else 2
    return route + (8 if cfg.act == synth.ACT_NVFP4 else 4)


def zipf_record(cfg, ids):
    """The realized per-expert pair counts of a Zipf workload against its water-filled
    targets (by Zipf rank)."""
    counts = np.bincount(ids[ids >= 0].ravel(), minlength=cfg.E)
    by_rank = np.empty(cfg.E, dtype=np.int64)
    by_rank[synth.zipf_rank_of_expert(cfg, 0)] = counts
    tgt = synth.zipf_targets(cfg.T, cfg.k, cfg.E, cfg.zipf_s)
    srt = np.sort(counts)[::-1]
    return {"targets_top5": [round(float(v), 1) for v in tgt[:5]],
            "realized_top5_by_rank": by_rank[:5].tolist(),
            "sorted_counts_top10": srt[:10].tolist(), "median": float(np.median(counts)),
            "min": int(srt[-1]), "experts_touched": int((counts > 0).sum()),
            "total_variation_vs_targets": round(float(np.abs(by_rank - tgt).sum() / (2.0 * cfg.T * cfg.k)), 4)}


def measure(cfg, args, steps, dist, world, rank, local, want_e2e=True, whole_cycles=False):
    """One workload: build its replicas, capture the step graphs, warm up, run the timed
    regions, then the end-to-end leg.  Returns the line's fields (rank 0) or None.
    whole_cycles: for the extra per-workload lines -- regions of whole cycles over the weight
    replicas (fewer steps would replay one-step graphs, each its own graph launch) and of at
    least min_region_ms of work (a region also times the launch of its first graph)."""
    from block_quantized_moe_router_gb300 import capi
    from block_quantized_moe_router_gb300.layer import MoeLayer

    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 0) or 128 * 2 ** 20
    inp = synth.make_inputs(cfg, seed=rank, device="cuda")
    base = MoeLayer.from_inputs(inp)
    x = inp["x"].cuda()
    tok = inp["token_ids"].cuda() if "token_ids" in inp else None
    T = cfg.T
    ids0, _, _ = base.route(x, token_ids=tok)
    torch.cuda.synchronize()
    ids0_h = ids0.cpu().numpy()
    real = ids0_h[(ids0_h >= 0) & (ids0_h < cfg.E)]
    touched = int(np.unique(real).size)
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
    dec = is_decode(cfg)
    if not dec:
        # the gate+up GEMM timed by events around it in every replica's step; read back after
        # each timed region (the last execution of every replica, all inside that region)
        for layer in layers:
            capi.moe_profile_enable(layer.handle, 1 << capi.PHASE_GATE_UP)

    stream = torch.cuda.Stream()
    graphs = []

    def step(layer, b):  # one layer step through the public API: route + FFN in one call
        layer.forward(x, token_ids=tok, out=b["out"], topk_ids=b["ids"], topk_w=b["w"],
                      logits_out=None if cfg.scoring == synth.SCORE_HASH else b["logits"])

    with torch.cuda.stream(stream):
        for layer, b in zip(layers, bufs):   # one eager pass per replica before capture
            step(layer, b)
        stream.synchronize()
        for layer, b in zip(layers, bufs):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(layer, b)
            graphs.append(g)
        # one graph of whole passes over the replicas, at least 4 steps (fewer graph launches
        # between steps; the steps and their order are the same)
        cyc_len = replicas * max(1, -(-4 // replicas))
        cycle = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cycle, stream=stream):
            for _ in range(cyc_len // replicas):
                for layer, b in zip(layers, bufs):
                    step(layer, b)
    torch.cuda.synchronize()

    def run_steps(first, n):
        """Layer steps first .. first + n - 1 (replica i % replicas), as graph replays."""
        i = first
        while i < first + n:
            if i % replicas == 0 and first + n - i >= cyc_len:
                cycle.replay()
                i += cyc_len
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
        torch.cuda.synchronize()
        step_s = w0.elapsed_time(w1) * 1e-3 / args.warmup
        if whole_cycles and steps is not None:
            per_cycle = max(step_s * replicas, 1e-9)
            cycles = max(-(-steps // replicas), int(math.ceil(args.min_region_ms * 1e-3 / per_cycle)))
            steps = int(max_over_ranks([cycles * replicas], dist, device="cuda")[0])
        if steps is None:  # about one second of timed work, the same on every rank
            try:
                steps = auto_steps(step_s, replicas)
            except Exception:  # no usable warm-up timing: the fixed default
                steps = 2000
            steps = int(max_over_ranks([steps], dist, device="cuda")[0])
        # regions of exactly `steps` steps, repeated until about args.min_timed_s of timed work
        est = max(step_s * steps, 1e-6)
        regions = int(min(args.max_regions, max(1, math.ceil(args.min_timed_s / est))))
        regions = int(max_over_ranks([regions], dist, device="cuda")[0])
        region_ms, dom_ms = [], []
        first = args.warmup
        barrier()
        torch.cuda.synchronize()
        clocks.mark()
        for _ in range(regions):
            ev0 = torch.cuda.Event(enable_timing=True)
            ev1 = torch.cuda.Event(enable_timing=True)
            barrier()
            torch.cuda.synchronize()
            ev0.record(stream)
            run_steps(first, steps)
            ev1.record(stream)
            torch.cuda.synchronize()
            barrier()
            first += steps
            region_ms.append(ev0.elapsed_time(ev1) / steps)
            if not dec:
                per = [float(capi.moe_profile_read(layer.handle)[capi.PHASE_GATE_UP]) for layer in layers]
                dom_ms.append(sum(per) / len(per))
    torch.cuda.synchronize()
    clocks.mark()
    clk = clocks.stop()
    ms = statistics.median(region_ms)
    # a few tokens: the step is one launch, so the kernel's time per launch is the step time
    # (inter-launch gaps included); otherwise the gate+up GEMM's event time
    launch_ms = ms if dec else statistics.median(dom_ms)
    ms, launch_ms = max_over_ranks([ms, launch_ms], dist, device="cuda")
    assert launch_ms <= ms * 1.0001 or not dec
    ok = all(torch.equal(bufs[0]["out"], b["out"]) for b in bufs[1:])
    if not dec:
        for layer in layers:
            capi.moe_profile_enable(layer.handle, 0)

    # end to end through the public API with host buffers: every step copies its x (and token
    # ids) in from pinned host memory, runs route + FFN, and copies its output back to pinned
    # host memory, and the host sees every step's output.  Three loops are timed and the
    # fastest one reported (every figure is in the line):
    #   serial  -- one stream, each step one CUDA graph (copies + route + FFN), the host waiting
    #              for every step's output before the next;
    #   overlap -- the layer steps run one after another on one compute stream (each a CUDA
    #              graph of route + FFN), the copies on their own in / out streams with two
    #              buffer slots, so step i's copies overlap the compute of steps i - 1 and
    #              i + 1; before issuing step i the host waits for step i - 2's output;
    #   host    -- the library's host-buffer entry point (moe_forward_host: copy in, route +
    #              FFN, copy out, enqueued by the library on one stream) called once per step
    #              with two pinned buffer slots in turn; the host waits for step i - 2's
    #              output before reusing its slot.
    nsl = 2
    x_host = [inp["x"].pin_memory() for _ in range(nsl)]
    out_host = [torch.empty((T, cfg.H), dtype=torch.bfloat16).pin_memory() for _ in range(nsl)]
    tok_host = [inp["token_ids"].pin_memory() for _ in range(nsl)] if tok is not None else None
    x_dev = [torch.empty_like(x) for _ in range(nsl)]
    tok_dev = [torch.empty_like(tok) for _ in range(nsl)] if tok is not None else None
    sout = [torch.empty((T, cfg.H), dtype=torch.bfloat16, device="cuda") for _ in range(nsl)]
    e2e_runs = {}

    def fwd(layer, b, s, out):
        layer.forward(x_dev[s], token_ids=None if tok_dev is None else tok_dev[s], out=out,
                      topk_ids=b["ids"], topk_w=b["w"],
                      logits_out=None if cfg.scoring == synth.SCORE_HASH else b["logits"])

    def copy_in(s):
        x_dev[s].copy_(x_host[s], non_blocking=True)
        if tok_dev is not None:
            tok_dev[s].copy_(tok_host[s], non_blocking=True)

    if want_e2e:
        e2e_steps = max(4, min(steps, 200, int(math.ceil(0.5 / max(step_s, 1e-6)))))
        # serial: slot 0 only
        g_serial = []
        with torch.cuda.stream(stream):
            for layer, b in zip(layers, bufs):
                copy_in(0)
                fwd(layer, b, 0, sout[0])
                out_host[0].copy_(sout[0], non_blocking=True)
            stream.synchronize()
            for layer, b in zip(layers, bufs):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    copy_in(0)
                    fwd(layer, b, 0, sout[0])
                    out_host[0].copy_(sout[0], non_blocking=True)
                g_serial.append(g)
        torch.cuda.synchronize()
        for i in range(e2e_steps + args.warmup):
            if i == args.warmup:
                barrier()
                torch.cuda.synchronize()
                t0 = time.perf_counter()
            with torch.cuda.stream(stream):
                g_serial[i % replicas].replay()
            stream.synchronize()
        e2e_runs["serial"] = (time.perf_counter() - t0) / e2e_steps
        # overlap: compute graphs (route + FFN) per replica and slot on `stream`
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        g_comp = {}
        with torch.cuda.stream(stream):
            for s in range(nsl):
                copy_in(s)
            for s in range(nsl):
                for r, (layer, b) in enumerate(zip(layers, bufs)):
                    fwd(layer, b, s, sout[s])
            stream.synchronize()
            for s in range(nsl):
                for r, (layer, b) in enumerate(zip(layers, bufs)):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        fwd(layer, b, s, sout[s])
                    g_comp[(r, s)] = g
        torch.cuda.synchronize()
        ev_in = [torch.cuda.Event() for _ in range(nsl)]
        ev_comp = [torch.cuda.Event() for _ in range(nsl)]
        ev_out = [torch.cuda.Event() for _ in range(nsl)]
        for i in range(e2e_steps + args.warmup):
            s, r = i % nsl, i % replicas
            if i == args.warmup:
                barrier()
                torch.cuda.synchronize()
                t0 = time.perf_counter()
            if i >= nsl:
                ev_out[s].synchronize()       # step i - 2's output is in out_host[s]
            with torch.cuda.stream(s_in):     # slot s's inputs are free once step i - 2 ran
                if i >= nsl:
                    s_in.wait_event(ev_comp[s])
                copy_in(s)
                ev_in[s].record(s_in)
            with torch.cuda.stream(stream):
                stream.wait_event(ev_in[s])
                g_comp[(r, s)].replay()
                ev_comp[s].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[s])
                out_host[s].copy_(sout[s], non_blocking=True)
                ev_out[s].record(s_out)
        for ev in ev_out:
            ev.synchronize()
        e2e_runs["overlap"] = (time.perf_counter() - t0) / e2e_steps
        # host: moe_forward_host per step, on `stream`
        ev_h = [torch.cuda.Event() for _ in range(nsl)]
        for i in range(e2e_steps + args.warmup):
            s, r = i % nsl, i % replicas
            if i == args.warmup:
                barrier()
                torch.cuda.synchronize()
                t0 = time.perf_counter()
            if i >= nsl:
                ev_h[s].synchronize()         # step i - 2's output is in out_host[s]
            layers[r].forward_host(x_host[s], out_host[s],
                                   token_ids_host=None if tok_host is None else tok_host[s],
                                   stream=stream)
            ev_h[s].record(stream)
        for ev in ev_h:
            ev.synchronize()
        e2e_runs["host"] = (time.perf_counter() - t0) / e2e_steps
        last = e2e_steps + args.warmup - 1
        host_ok = bool(torch.equal(out_host[last % nsl], bufs[0]["out"].cpu()))
        e2e_mode = min(e2e_runs, key=e2e_runs.get)
        e2e_s = e2e_runs[e2e_mode]
    else:
        e2e_s, e2e_mode, host_ok = float("nan"), None, None
    e2e_s = max_over_ranks([e2e_s], dist, device="cuda")[0]
    e2e_runs = {k: max_over_ranks([v], dist, device="cuda")[0] for k, v in e2e_runs.items()}
    h2d = T * cfg.H * 2 + (T * 4 if tok is not None else 0)
    d2h = T * cfg.H * 2

    result = None
    if rank == 0:
        pk = measured_peaks()
        hbm = pk["hbm_gbs"]
        fp4_peak = pk["bf16_tflops_sustained"] * FP4_OVER_BF16
        dom_bytes = nbytes["total"] if dec else nbytes["gate_up"]
        dom_flops = nbytes["flops"] if dec else nbytes["gate_up_flops"]
        a4 = cfg.act == synth.ACT_NVFP4
        dom_name = ("dec_fused_kernel (route + FFN, one launch per step)" if dec else
                    "gate+up GEMM (" + ("tc_gemm_kernel" if a4 else "expert_mma_kernel") + ")")
        gbs = dom_bytes / (launch_ms * 1e-3) / 1e9
        tflops = dom_flops / (launch_ms * 1e-3) / 1e12
        mma_peak = fp4_peak if a4 else pk["bf16_tflops_sustained"]
        # the bound: whichever roof is lower for this launch's bytes and FLOPs
        tensor_bound = a4 and dom_flops / (mma_peak * 1e12) > dom_bytes / (hbm * 1e9)
        src = kernel_source_hash(KERNEL_SOURCES["decode" if dec else "tc" if a4 else "mma"])
        traffic = captured_traffic(cfg.name, src)
        if tensor_bound:
            roof = {"bound": "tensor", "achieved": tflops, "peak": mma_peak, "unit": "TFLOP/s",
                    "frac": tflops / mma_peak, "traffic": traffic,
                    "peak_source": f"{pk['source']} sustained bf16 x nominal fp4/bf16 ratio"}
        else:
            roof = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                    "frac": gbs / hbm, "traffic": traffic, "peak_source": pk["source"] + " copy"}
        roof.update({"kernel": dom_name, "bytes_per_launch": dom_bytes,
                     "flops_per_launch": dom_flops, "launch_ms": launch_ms,
                     "launch_timing": "step time (one launch per step)" if dec else
                     "CUDA events around the launch in every replica, median of regions"})
        layer_gbs = nbytes["total"] / (ms * 1e-3) / 1e9
        result = {
            "value": job_tokens_per_s(T, world, ms * 1e-3), "ms_per_step": ms,
            "steps": steps, "regions": regions,
            "config": {"workload": cfg.name, "T": T, "H": cfg.H, "I": cfg.I, "E": cfg.E,
                       "top_k": cfg.k, "I_shared": cfg.I_shared, "replicas": replicas,
                       "l2_policy": f"inputs larger than L2: {replicas} weight replicas cycled, "
                                    f"{replicas * nbytes['total'] / 1e6:.0f} MB touched per cycle",
                       "launch": f"CUDA graph of {replicas} layer steps (one per replica), replayed",
                       "timed_regions": f"{regions} regions of {steps} steps, median reported",
                       "touched_experts": touched},
            "gpu_launches": steps * launches_per_step(cfg),
            "roofline": roof,
            "tensor_view": {"achieved_tflops": tflops, "peak_tflops": mma_peak,
                            "frac": tflops / mma_peak,
                            "dtype": "nvfp4 x nvfp4" if a4 else "f16 mma",
                            "peak_source": f"{pk['source']} sustained bf16" +
                                           (" x nominal fp4/bf16 ratio" if a4 else "")},
            "layer_roofline": {"achieved": layer_gbs, "peak": hbm, "unit": "GB/s",
                               "frac": layer_gbs / hbm, "bytes_per_step": nbytes["total"],
                               "flops_per_step": nbytes["flops"]},
            "clocks": clk,
            "e2e": {"value": job_tokens_per_s(T, world, e2e_s), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "mode": e2e_mode,
                    "ms_per_step": e2e_s * 1e3,
                    "loops_ms_per_step": {k: v * 1e3 for k, v in e2e_runs.items()},
                    "host_entry_output_equal": host_ok,
                    "loops": "serial: one graph per step (copies + route + FFN), host waits "
                             "for each step; overlap: steps one after another on one compute "
                             "stream, copies on in/out streams with two buffer slots, host "
                             "waits for step i - 2; host: moe_forward_host (the library's "
                             "host-buffer entry: copies and launches issued in C) per step, "
                             "two pinned slots, host waits for step i - 2"},
            "replica_outputs_equal": ok,
            "kernel_source": src,
        }
        if cfg.zipf_s > 0:
            result["config"]["zipf_counts"] = zipf_record(cfg, ids0_h)
    for layer in layers:
        layer.close()
    del layers, bufs, graphs, cycle, inp, base, x
    torch.cuda.empty_cache()
    return result


def run_ours(args, cfg):
    from block_quantized_moe_router_gb300 import build, capi

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

    head = measure(cfg, args, args.steps, dist, world, rank, local, want_e2e=args.e2e)
    others = {}
    if args.per_workload:
        for name in PER_WORKLOAD:
            if name == cfg.name:
                continue
            res = measure(synth.CONFIGS[name], args, args.steps, dist, world, rank, local,
                          want_e2e=args.e2e, whole_cycles=True)
            if res is not None:
                others[name] = res
    if rank == 0:
        line = {"metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
                "steps": head["steps"], "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "nvfp4 weights and activations, f32 accumulate"
                if cfg.act == synth.ACT_NVFP4 else "nvfp4 weights, f16 mma / f32 accumulate",
                "data": "synthetic (seeded; shapes and distributions of the named workload)"}
        for key in ("config", "gpu_launches", "roofline", "tensor_view", "layer_roofline", "clocks",
                    "e2e", "replica_outputs_equal", "kernel_source", "regions"):
            line[key] = head[key]
        line["gpu_launches_scope"] = "one timed region of `steps` steps"
        if others:
            line["per_workload"] = others
        if args.cpu_baseline:
            _, inp_np = host_inputs(cfg, seed=rank)
            line["cpu_baseline"] = cpu_baseline(cfg, inp_np, budget_s=args.cpu_budget)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="steps per timed region (default: about one second of device time)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=list(synth.CONFIGS))
    ap.add_argument("--per-workload", dest="per_workload", action="store_true", default=None,
                    help="also measure dec1, dec8, hash64 and pre32768 (default: with the "
                         "default workload only)")
    ap.add_argument("--no-per-workload", dest="per_workload", action="store_false")
    ap.add_argument("--min-timed-s", type=float, default=1.0,
                    help="repeat the timed region until about this much timed work")
    ap.add_argument("--max-regions", type=int, default=5000)
    ap.add_argument("--min-region-ms", type=float, default=5.0,
                    help="per-workload lines: at least this much work per timed region")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--replicas", type=int, default=0,
                    help="weight replicas to cycle (default: enough to exceed 4x L2)")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.per_workload is None:
        args.per_workload = args.config == DEFAULT_CONFIG
    cfg = synth.CONFIGS[args.config]
    if args.impl == "reference":
        if args.steps is None:
            args.steps = 20
        run_reference(args, cfg)
    else:
        run_ours(args, cfg)


if __name__ == "__main__":
    main()
