"""Benchmark of the Beam MoE layer on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config decode]
    python bench.py --impl reference ...      # the CPU oracle as the reference arm

A step is one call of the whole layer (router, selection, permute, gather of
the token rows (inside the gate/up GEMM for decode-sized batches), gate/up
GEMM, down GEMM, combine) on one batch of the workload, with every
input resident in device memory.  Metric: layer tokens/s.  The headline is
--config (the decode batch by default); the default run also measures the
prefill chunk, the skewed routing, the NVFP4 batch (quantised and 16-bit
activations), the dynamic FP8 decode and prefill batches and the MXFP8
decode batch in the same process with the same steps, each as a record under "workloads" (a summary
of each also under "roofline").  The expert weights
a step touches (about 12 GB for the decode batch) are far larger than L2, so
no flush is needed between steps.  Timing: CUDA events on the launching
stream around the K timed steps, bracketed by a barrier and a device
synchronisation, max over ranks.  Per-kernel durations come from events the
library records at its step boundaries during the same timed steps.

Multi-GPU: the layer's token batches are independent; under torchrun each
rank runs its own replica on its own GPU (replicas only, no collective on the
data path; the process group only aggregates timings).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import re
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import group_limited_routed_gb300 as pkg  # noqa: E402
from group_limited_routed_gb300 import inputs  # noqa: E402

METRIC = "Beam MoE-layer tokens/s"
UNIT = "tokens/s"
STAGES = ["router", "select", "permute", "gather", "gate_up", "down", "combine"]
# the dominant kernel of each expert format (its gate/up GEMM) and the source
# files that define it; a stored traffic counter holds while they are unchanged
DOMINANT = {"bf16": "gate_up", "nvfp4": "fp4_gate_up", "a16": "w4a16_gate_up",
            "fp8": "fp8_gate_up", "mxfp8": "mx_gate_up"}
DOMINANT_SRC = {k: [os.path.join(ROOT, "group_limited_routed_gb300", "csrc", f) for f in v]
                for k, v in {
                    "gate_up": ("expert_gemm_kernel.cuh", "expert_gemm_pair_kernel.cuh",
                                "expert_gemm.cuh", "gemm_common.cuh", "common.cuh", "ptx.cuh"),
                    "fp4_gate_up": ("nvfp4.cu", "gemm_common.cuh", "common.cuh", "ptx.cuh"),
                    "w4a16_gate_up": ("w4a16.cu", "gemm_common.cuh", "common.cuh", "ptx.cuh"),
                    "fp8_gate_up": ("expert_gemm_kernel.cuh", "expert_gemm_pair_kernel.cuh",
                                    "expert_gemm.cuh", "gemm_common.cuh", "common.cuh", "ptx.cuh"),
                    "mx_gate_up": ("nvfp4.cu", "gemm_common.cuh", "common.cuh", "ptx.cuh"),
                }.items()}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


# ------------------------------------------------------------------ helpers
def reduce_max(values, use_dist: bool, device="cpu"):
    """Element-wise max over ranks (the job's time is its slowest rank's)."""
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if use_dist:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(world: int, tokens_per_rank: int, steps: int, ms: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank * steps / (ms / 1e3)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), ws


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": float(j["hbm_gbs"]), "bf16_tflops": float(j["bf16_tflops"]),
                "bf16_tflops_sustained": float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 9:
                    rows.append(p)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def touched_experts(ws, cfg) -> int:
    idx = ws.view("topk_idx", torch.int32, (cfg.T, cfg.topk))
    return int(torch.unique(idx).numel())


def file_sha(paths) -> str:
    """Hash of the sources' code: comments and whitespace do not count, so
    a comment edit keeps a capture valid; any code change invalidates it."""
    h = hashlib.sha256()
    for p in paths:
        with open(p, encoding="utf-8") as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update("".join(src.split()).encode())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu capture, when the kernel's
    source is unchanged since it was taken."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        j = json.load(f)
    ent = j.get(kernel, {}).get(workload)
    if not ent or ent.get("source_sha") != file_sha(DOMINANT_SRC[kernel]):
        return None
    return ent.get("bytes_per_launch")


# ------------------------------------------------------------------ CPU oracle
def oracle_sample(cfg, t, n_tokens: int, seed: int = 0, a16: bool = False):
    """Runs the CPU oracle (router + selection for the whole batch, experts
    and combine for n_tokens sampled tokens); returns (seconds, sampled)."""
    import oracle
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(cfg.T, size=min(n_tokens, cfg.T), replace=False))
    x = inputs.bf16_bits(t["hidden"])
    wr = t["router_w"].cpu().numpy()
    b = t["corr_bias"].cpu().numpy()
    # weights the sample needs, fetched before the clock starts
    lg = oracle.router_logits(x, wr)
    r = oracle.route(lg, b, cfg.n_groups, cfg.topk_groups, cfg.topk, cfg.routed_scale)
    need = sorted({int(e) for e in r["idx"][rows].reshape(-1)})
    if cfg.weight_fmt == "nvfp4":
        proj = [{"q": {e: p["q"][e].cpu().numpy() for e in need},
                 "sf": {e: p["sf"][e].cpu().numpy() for e in need},
                 "gs": p["gs"].cpu().numpy()} for p in (t["w_gate"], t["w_up"], t["w_down"])]
    elif cfg.weight_fmt in ("fp8", "mxfp8"):
        proj = [{"q": {e: p["q"][e].cpu().numpy() for e in need},
                 "s": {e: p["s"][e].cpu().numpy() for e in need}}
                for p in (t["w_gate"], t["w_up"], t["w_down"])]
    else:
        proj = [{e: inputs.bf16_bits(t[n][e]) for e in need} for n in ("w_gate", "w_up", "w_down")]
    t0 = time.perf_counter()
    lg = oracle.router_logits(x[rows], wr)
    r = oracle.route(lg, b, cfg.n_groups, cfg.topk_groups, cfg.topk, cfg.routed_scale)
    if cfg.weight_fmt == "nvfp4":
        oracle.experts_nvfp4(x[rows], r["idx"], r["w"], *proj, cfg.n_experts,
                             act_quant=oracle.ACT_F16 if a16 else oracle.ACT_NVFP4)
    elif cfg.weight_fmt == "fp8":
        oracle.experts_fp8(x[rows], r["idx"], r["w"], *proj, cfg.n_experts, act_quant=True)
    elif cfg.weight_fmt == "mxfp8":
        oracle.experts_mxfp8(x[rows], r["idx"], r["w"], *proj, cfg.n_experts, act_quant=True)
    else:
        oracle.experts_bf16(x[rows], r["idx"], r["w"], *proj, cfg.n_experts)
    return time.perf_counter() - t0, len(rows)


def cpu_baseline(cfg, t, budget_s: float = 12.0, a16: bool = False) -> dict:
    """The oracle on about budget_s seconds of the same workload: sampled
    tokens of the batch, or the whole batch repeated when it is quicker."""
    import oracle
    sec1, n1 = oracle_sample(cfg, t, 1, seed=1, a16=a16)
    per_tok = sec1 / n1
    n = int(max(1, min(cfg.T, budget_s / max(per_tok, 1e-6))))
    reps = 1
    if n == cfg.T:
        full, _ = oracle_sample(cfg, t, cfg.T, seed=2, a16=a16)
        reps = int(max(1, min(100, budget_s / max(full, 1e-6))))
    sec = 0.0
    toks = 0
    for r in range(reps):
        s, m = oracle_sample(cfg, t, n, seed=2 + r, a16=a16)
        sec += s
        toks += m
    what = (f"the whole {cfg.T}-token {cfg.name} batch, {reps} times" if n == cfg.T
            else f"{n} of the {cfg.T} tokens of one {cfg.name} batch")
    return {"value": toks / sec, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": (f"{what}: FP32 router and group-limited selection, the tokens' 8 SwiGLU "
                       f"experts and the combine, FP64 accumulation; {sec:.1f} s of CPU work")}


# ------------------------------------------------------------------ arms
def run_reference(args, cfg):
    rank, local, world = dist_env()
    if rank != 0:
        return 0
    import oracle
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    gen_cfg = cfg if dev.type == "cuda" else cfg.replace(cpu_generator=True)
    t = inputs.generate(gen_cfg, dev)
    a16 = cfg.weight_fmt == "nvfp4" and args.a16
    # size each step so the whole run stays within about two minutes; the
    # oracle spreads tokens over its threads, so a step samples at least one
    # token per thread when that fits (one token alone would use one core)
    cores = oracle.num_threads()
    # the experts the whole batch touches, from the oracle's own routing
    r = oracle.route(oracle.router_logits(inputs.bf16_bits(t["hidden"]),
                                          t["router_w"].cpu().numpy()),
                     t["corr_bias"].cpu().numpy(), cfg.n_groups, cfg.topk_groups, cfg.topk,
                     cfg.routed_scale)
    touched = int(np.unique(r["idx"]).size)
    sec1, _ = oracle_sample(cfg, t, 1, seed=1, a16=a16)
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    n = int(max(1, min(cfg.T, cores * per_step_budget / max(sec1, 1e-6))))
    for i in range(args.warmup):
        oracle_sample(cfg, t, n, seed=100 + i, a16=a16)
    secs = 0.0
    toks = 0
    for i in range(args.steps):
        s, m = oracle_sample(cfg, t, n, seed=1000 + i, a16=a16)
        secs += s
        toks += m
    value = toks / secs
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_record(cfg, touched, a16=a16),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores,
                             "kind": "oracle",
                             "sample": f"{n} sampled tokens of the {cfg.T}-token batch per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_record(cfg, touched, routed=False, a16=False, graph=False):
    rec = {"workload": cfg.description, "T": cfg.T, "d": cfg.d, "n_experts": cfg.n_experts,
           "n_groups": cfg.n_groups, "topk_groups": cfg.topk_groups, "topk": cfg.topk,
           "d_ff": cfg.d_ff, "routed_scale": cfg.routed_scale, "weights": cfg.weight_fmt,
           "seed": cfg.seed, "parallelism": "replicas (one independent layer per GPU)",
           "l2": "no flush: each step streams the touched experts' weights, far larger than "
                 "the 129 MB L2"}
    if touched is not None:
        rec["touched_experts"] = touched
    if routed:
        rec["routing"] = "replayed (recorded once; steps run experts + combine)"
    if a16:
        rec["activations"] = "f16 (not quantised): W4A16"
    if graph:
        rec["launch"] = "one layer call captured in a CUDA graph, replayed each step"
    return rec


# Nominal dense tensor rate of each expert format relative to BF16 on GB300
# (2.25 PFLOP/s BF16, 4.5 FP8, 13.5 FP4); W4A16 multiplies in F16.
TC_RATIO = {"bf16": 1.0, "fp8": 2.0, "nvfp4": 6.0, "a16": 1.0, "mxfp8": 2.0}
NOMINAL_HBM_GBS = 7900.0


def kernel_roofline(kernel, bytes_alg, flops, us, fmt, pk, traffic=None, intermediates=None):
    """One kernel's place against its bounds.  bytes_alg: the algorithmic
    bytes it must move (the touched experts' weights of its projections, and
    the layer's hidden input for gate/up); intermediates: the bytes of the
    implementation's own buffers it reads and writes, reported apart.  Bound
    "tensor" when its flops per algorithmic byte exceed the ridge of the
    sustained tensor peak of its dtype over the copy bandwidth.  The copy
    bandwidth moves as many bytes written as read, so a read-dominated kernel
    can pass it: the fraction of the nominal HBM rate is reported beside."""
    sec = us / 1e6
    gbs = bytes_alg / sec / 1e9
    tflops = flops / sec / 1e12
    sus = pk["bf16_tflops_sustained"] * TC_RATIO[fmt]
    burst = pk["bf16_tflops"] * TC_RATIO[fmt]
    ridge = sus * 1e12 / (pk["hbm_gbs"] * 1e9)
    tensor = flops / bytes_alg > ridge
    rec = {"kernel": kernel, "us": round(us, 2), "algorithmic_bytes_per_launch": int(bytes_alg),
           "algorithmic_flops_per_launch": int(flops),
           "hbm": {"achieved": gbs, "peak": pk["hbm_gbs"], "frac": gbs / pk["hbm_gbs"],
                   "frac_nominal": gbs / NOMINAL_HBM_GBS},
           "tensor": {"achieved": tflops, "peak_sustained": sus, "frac_sustained": tflops / sus,
                      "peak_burst": burst, "frac_burst": tflops / burst},
           "roofline_frac": max(bytes_alg / (pk["hbm_gbs"] * 1e9), flops / (sus * 1e12)) / sec}
    if tensor:
        rec.update({"bound": "tensor", "achieved": tflops, "peak": sus, "unit": "TFLOP/s",
                    "frac": tflops / sus})
    else:
        rec.update({"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": gbs / pk["hbm_gbs"]})
    rec["traffic"] = traffic
    if intermediates:
        rec["intermediate_bytes"] = {k: int(v) for k, v in intermediates.items()}
    return rec


def measure(cfg, args, dev, rank, world, use_dist, *, a16=False, routed=False, graph=False,
            cpu=False):
    """One workload: W warm-up steps, then the K timed steps of the layer as
    a caller runs it, the same K steps again with the library's stage events
    (per-kernel times), and K end-to-end steps from pinned host memory.
    Returns its record (tokens/s over the slowest rank)."""
    t = inputs.generate(cfg.replace(seed=cfg.seed + 1000 * rank) if rank else cfg, dev)
    fp4 = cfg.weight_fmt == "nvfp4"
    fp8 = cfg.weight_fmt == "fp8"
    mx = cfg.weight_fmt == "mxfp8"
    a16 = fp4 and a16
    fmt_name = ("a16" if a16 else "nvfp4") if fp4 else "fp8" if fp8 else "mxfp8" if mx else "bf16"
    fmt = ((pkg.NVFP4_A16 if a16 else pkg.NVFP4) if fp4 else pkg.FP8 if fp8
           else pkg.MXFP8 if mx else 0)
    ws = pkg.Workspace(cfg, cfg.T, dev, weight_fmt=fmt)
    stream = torch.cuda.current_stream()
    out = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16, device=dev)
    ridx = None
    if fp4:
        wts = [pkg.Fp4Weight.of(t[n]) for n in ("w_gate", "w_up", "w_down")]
        fwd = pkg.forward_nvfp4_a16 if a16 else pkg.forward_nvfp4

        def layer(x, o):
            return fwd(cfg, x, t["router_w"], t["corr_bias"], *wts, out=o, ws=ws,
                       stream=torch.cuda.current_stream())
    elif fp8:
        wts = [pkg.Fp8Weight.of(t[n]) for n in ("w_gate", "w_up", "w_down")]

        def layer(x, o):
            return pkg.forward_fp8(cfg, x, t["router_w"], t["corr_bias"], *wts, out=o, ws=ws,
                                   stream=torch.cuda.current_stream())
    elif mx:
        wts = [pkg.Mxfp8Weight.of(t[n]) for n in ("w_gate", "w_up", "w_down")]

        def layer(x, o):
            return pkg.forward_mxfp8(cfg, x, t["router_w"], t["corr_bias"], *wts, out=o, ws=ws,
                                     stream=torch.cuda.current_stream())
    elif routed:
        # routing replay: the routes are recorded once, the timed steps run
        # the experts and the combine on them
        ridx, rw = pkg.route(cfg, t["hidden"], t["router_w"], t["corr_bias"], stream=stream)

        def layer(x, o):
            return pkg.forward_routed(cfg, x, ridx, rw, t["w_gate"], t["w_up"], t["w_down"],
                                      out=o, ws=ws, stream=torch.cuda.current_stream())
    else:
        def layer(x, o):
            return pkg.forward(cfg, x, t["router_w"], t["corr_bias"], t["w_gate"], t["w_up"],
                               t["w_down"], out=o, ws=ws, stream=torch.cuda.current_stream())

    def step(o=out):
        return layer(t["hidden"], o)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if pkg.check_status(ws) != 0:
        raise RuntimeError(f"{cfg.name}: device status after warm-up")
    touched = int(torch.unique(ridx).numel()) if routed else touched_experts(ws, cfg)

    # per-step stage events (created and recorded once so the handles exist)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(args.steps)]
    for row in evs:
        for e in row:
            e.record(stream)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    for _ in range(max(3, args.warmup)):
        step()
    if use_dist:
        dist_barrier()
    torch.cuda.synchronize()
    graphs = None
    if graph:
        # one layer call captured twice: plain, and with its stage events
        # (event-record nodes; each replay records them again, so they hold
        # the last replay's times)
        gevs = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
        for e in gevs:
            e.record(stream)  # creates the handles
        graphs = [torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()]
        with torch.cuda.graph(graphs[0]):
            step()
        pkg.set_stage_events(gevs)
        with torch.cuda.graph(graphs[1]):
            step()
        pkg.set_stage_events(None)
        for g in graphs:
            for _ in range(3):
                g.replay()
        torch.cuda.synchronize()

    def timed_loop(with_events: bool) -> float:
        """K steps between a barrier and a synchronize on both sides; with
        stage events the library records each step's stage boundaries (they
        cost GPU time of their own, so the headline loop runs without)."""
        if use_dist:
            dist_barrier()
        torch.cuda.synchronize()
        t_start.record(stream)
        for i in range(args.steps):
            if graphs is not None:
                graphs[1 if with_events else 0].replay()
            else:
                pkg.set_stage_events(evs[i] if with_events else None)
                step()
        t_end.record(stream)
        torch.cuda.synchronize()
        if use_dist:
            dist_barrier()
        pkg.set_stage_events(None)
        return t_start.elapsed_time(t_end)

    ms = timed_loop(False)          # the layer as a caller runs it
    ms_events = timed_loop(True)    # the same steps with stage events: per-kernel times
    clocks = sampler.stop()
    if graphs is not None:
        stage_ms = np.array([gevs[j].elapsed_time(gevs[j + 1]) for j in range(7)])
    else:
        stage_ms = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(7)]
                             for i in range(args.steps)]).mean(axis=0)
    if pkg.check_status(ws) != 0:
        raise RuntimeError(f"{cfg.name}: device status after the timed region")

    # end to end through the public API: pinned host in, pinned host out
    x_host = t["hidden"].cpu().pin_memory()
    o_host = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(t["hidden"])

    def e2e_step():
        x_dev.copy_(x_host, non_blocking=True)
        layer(x_dev, out)
        o_host.copy_(out, non_blocking=True)

    e2e_steps = max(3, min(args.steps, 200))
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)

    ms, e2e_ms = reduce_max([ms, e2e_ms], use_dist, dev)
    value = job_throughput(world, cfg.T, args.steps, ms)
    e2e_value = job_throughput(world, cfg.T, e2e_steps, e2e_ms)

    pk = peaks()
    T, d, F, E, k = cfg.T, cfg.d, cfg.d_ff, cfg.n_experts, cfg.topk
    TK = T * k
    # weight bytes of one projection of one expert: BF16, E2M1 + E4M3 per 16,
    # E4M3 + one FP32 scale per output row, or E4M3 + E8M0 per 32
    E_b = (d * F // 2 + d * F // 16 if fp4 else d * F if fp8 else d * F + d * F // 32 if mx
           else d * F * 2)
    gu_w = touched * 2 * (E_b + (4 * F if fp8 else 0))
    dn_w = touched * (E_b + (4 * d if fp8 else 0))
    hidden_b = T * d * 2
    # the implementation's own buffers (not algorithmic bytes): token rows in
    # expert order, h, the FP32 expert rows y
    # (MXFP8: a byte per element and a 16-byte scale slot per 128)
    x_row = d * (0.5625 if fp4 and not a16 else 1 if fp8 else 1.125 if mx else 2)
    h_row = F * (0.5625 if fp4 and not a16 else 1.125 if mx else 2)
    small = TK <= 4 * E
    gu_inter = {"token_rows_read": TK * x_row, "h_written": TK * h_row}
    if fp8:
        gu_inter["h_bf16_written"] = TK * F * 2
        gu_inter.pop("h_written")
    dn_inter = {"h_read": TK * (F if fp8 else h_row), "y_written": TK * d * 4}
    gu_flops = 4 * TK * d * F
    dn_flops = 2 * TK * d * F
    dom = DOMINANT[fmt_name]
    kernels = {
        "gate_up": kernel_roofline(dom, gu_w + hidden_b, gu_flops, stage_ms[4] * 1e3, fmt_name,
                                   pk, traffic_for(dom, cfg.name), gu_inter),
        "down": kernel_roofline(dom.replace("gate_up", "down"), dn_w, dn_flops,
                                stage_ms[5] * 1e3, fmt_name, pk, None, dn_inter),
    }
    layer_bytes = touched * (3 * E_b + (4 * (2 * F + d) if fp8 else 0)) + E * d * 4 + E * 4 \
        + 2 * T * d * 2
    layer_ms = ms / args.steps
    layer_flops = 2 * T * d * E + 6 * TK * d * F
    sus = pk["bf16_tflops_sustained"] * TC_RATIO[fmt_name]
    burst = pk["bf16_tflops"] * TC_RATIO[fmt_name]
    lsec = layer_ms / 1e3
    layer_roof = {
        "algorithmic_bytes": int(layer_bytes), "algorithmic_flops": int(layer_flops),
        "hbm": {"achieved": layer_bytes / lsec / 1e9, "peak": pk["hbm_gbs"],
                "frac": layer_bytes / lsec / 1e9 / pk["hbm_gbs"],
                "frac_nominal": layer_bytes / lsec / 1e9 / NOMINAL_HBM_GBS},
        "tensor": {"achieved": layer_flops / lsec / 1e12, "peak_sustained": sus,
                   "frac_sustained": layer_flops / lsec / 1e12 / sus, "peak_burst": burst,
                   "frac_burst": layer_flops / lsec / 1e12 / burst},
        # max(bytes / BW, flops / TC) / time, the sustained tensor peak
        "roofline_frac": max(layer_bytes / (pk["hbm_gbs"] * 1e9),
                             layer_flops / (sus * 1e12)) / lsec,
        "intermediate_bytes": {
            "scatter": 0 if small or fp4 or mx else int(T * x_row + TK * x_row),
            "gate_up": int(sum(gu_inter.values())), "down": int(sum(dn_inter.values())),
            "combine": int(TK * d * 4 + T * d * 2)}}
    gu = kernels["gate_up"]
    roofline = {k: gu[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")}
    roofline.update({"kernel": dom, "peak_source": pk["source"] + (
        " (sustained bf16" + (f" x {TC_RATIO[fmt_name]:g}, the nominal ratio)" if
                              TC_RATIO[fmt_name] != 1 else ")") if gu["bound"] == "tensor"
        else " (copy bandwidth)"),
        "algorithmic_bytes_per_launch": gu["algorithmic_bytes_per_launch"],
        "algorithmic_flops_per_launch": gu["algorithmic_flops_per_launch"],
        "frac_nominal_hbm": gu["hbm"]["frac_nominal"], "nominal_hbm_gbs": NOMINAL_HBM_GBS})
    rec = {
        "value": value, "unit": UNIT, "ms_per_step": layer_ms,
        "dtype": ("nvfp4 weights x f16 activations" if a16 else "nvfp4 (e2m1 x e4m3 per 16)")
        if fp4 else "fp8 (e4m3, fp32 scale per row)" if fp8
        else "mxfp8 (e4m3 x e8m0 per 32)" if mx else "bf16",
        "config": config_record(cfg, touched, routed, a16, graph),
        "roofline": roofline, "kernels": kernels, "layer_roofline": layer_roof,
        "stage_us": {n: round(float(v) * 1e3, 1) for n, v in zip(STAGES, stage_ms)},
        # the per-stage times (and the kernels' times) come from a second
        # timed loop of the same steps with stage events recorded
        "stage_events_ms_per_step": ms_events / args.steps,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": T * d * 2,
                "d2h_bytes_per_step": T * d * 2},
        "gpu_launches": args.steps * pkg.kernels_per_forward(cfg, T, fmt, routed),
        "clocks": clocks,
    }
    if cpu:
        rec["cpu_baseline"] = cpu_baseline(cfg, t, a16=a16)
    del t, ws, out
    torch.cuda.empty_cache()
    return rec


def dist_barrier():
    import torch.distributed as dist
    dist.barrier()


# The workloads measured beside the headline in the default run: the
# prefill chunk and skewed routing (BF16), the NVFP4 batch with quantised
# and with 16-bit activations, the dynamic FP8 decode and prefill, and the
# MXFP8 decode batch.
SUB_WORKLOADS = [("prefill", False), ("skewed", False), ("nvfp4", False), ("nvfp4", True),
                 ("fp8", False), ("fp8_prefill", False), ("mxfp8", False)]


def summary(name, rec):
    """The figures of one sub-workload that the headline line repeats."""
    gu, dn, lr = rec["kernels"]["gate_up"], rec["kernels"]["down"], rec["layer_roofline"]
    return {"ms_per_step": rec["ms_per_step"], "tokens_per_s": rec["value"],
            "layer_hbm_frac": lr["hbm"]["frac"], "layer_tflops": lr["tensor"]["achieved"],
            "layer_tensor_frac_sustained": lr["tensor"]["frac_sustained"],
            "layer_tensor_frac_burst": lr["tensor"]["frac_burst"],
            "layer_roofline_frac": lr["roofline_frac"],
            "gate_up": {"bound": gu["bound"], "frac": gu["frac"], "us": gu["us"]},
            "down": {"bound": dn["bound"], "frac": dn["frac"], "us": dn["us"]},
            "sm_mhz": rec["clocks"].get("sm_mhz"), "reasons": rec["clocks"].get("reasons")}


def run_gpu(args, cfg):
    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    use_dist = world > 1
    if use_dist:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    head = measure(cfg, args, dev, rank, world, use_dist, a16=args.a16, routed=args.routed,
                   graph=args.graph,
                   cpu=rank == 0 and world == 1 and not args.no_cpu_baseline and not args.routed)
    line = {"metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": head["dtype"], "data": "synthetic"}
    line.update({k: v for k, v in head.items() if k not in ("value", "unit", "ms_per_step",
                                                             "dtype")})
    subs = [] if args.headline_only else [
        (n, a) for n, a in SUB_WORKLOADS if not (n == args.config and a == args.a16)]
    if subs:
        line["workloads"] = {}
        for name, sub_a16 in subs:
            key = name + ("_a16" if sub_a16 else "")
            rec = measure(inputs.CONFIGS[name], args, dev, rank, world, use_dist, a16=sub_a16)
            line["workloads"][key] = rec
        # the sub-workloads' headline figures, also inside the roofline record
        line["roofline"]["workloads"] = {k: summary(k, v) for k, v in line["workloads"].items()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if use_dist:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="decode", choices=sorted(inputs.CONFIGS))
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--a16", action="store_true",
                    help="NVFP4 configs: 16-bit activations (beam_moe_forward_nvfp4_a16)")
    ap.add_argument("--graph", action="store_true",
                    help="replay the layer call from a CUDA graph (stage times of the last replay)")
    ap.add_argument("--routed", action="store_true",
                    help="time beam_moe_forward_routed on recorded routes (routing replay)")
    ap.add_argument("--headline-only", action="store_true",
                    help="measure only --config, without the other workloads")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)
    cfg = inputs.CONFIGS[args.config]
    if args.impl == "reference":
        return run_reference(args, cfg)
    return run_gpu(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
