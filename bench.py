"""Benchmark of the gated delta rule prefill on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference] [--workload NAME]

One step = one gdr_chunk_fwd over one row of the workload (default: L = 4096 tokens, 16 key heads
-> 32 value heads, D = 128, bf16 q/k/v, float32 gates and states, initial state in, final state
out): the whole hot path (normalisation, chunk decay, WY factors, state recurrence, outputs).
Under torchrun each rank runs its own row on its own GPU (independent problems: weak scaling, no
collective on the data path); rank 0 prints one JSON line with the max time over ranks.

Timing: W untimed warm-up steps, then exactly K steps between CUDA events on the launch stream
(barrier + synchronize on both sides), with nothing recorded between the launches. Inputs rotate
over several resident copies whose total exceeds the 129 MB L2, so every step reads its inputs
from HBM. Per-kernel times come from a second pass of the same K steps with the library's stage
timer (CUDA events recorded around each of its launches on the same stream); those events keep the
state kernel from starting before the prep kernel ends, so that pass is not the headline value.
The e2e figure is the same step through the same call with host buffers: pinned host -> device
copies of the inputs, the call, and device -> host copies of o and S_T, all inside its timed
region, double-buffered (step i's uploads on a copy stream while step i - 1 computes, its
downloads on another while step i + 1 computes); the serial form is reported beside it. The "rows" object adds the fork pass and the decode step of the fork workload (256 forks
of one trunk state), the GDN prologue (conv + SiLU, gates and carry at the prefill row's shapes)
and the gated RMSNorm epilogue on the prefill row's output, each with its own HBM roofline.

--impl reference times the float64 CPU oracle (the checker the tests use) on a bounded sample of
the same workload on the host cores, as the reference arm.
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "gated-delta-rule prefill tokens/s (Hv=32,D=128,L=4096), % of roofline"
UNIT = "tokens/s"
L2_BYTES = 129 * 1024 * 1024
D = 128

WORKLOADS = {
    # name: (L, Hk, Hv, with S0, input regime)
    "prefill4096": (4096, 16, 32, True, "R1"),
    "prefill8192": (8192, 16, 16, False, "R2"),
}


def algorithmic(L: int, Hk: int, Hv: int, s0: bool) -> tuple[int, float]:
    """(bytes, flops) the path must move / compute for one row.

    Bytes: q, k read once at the key heads, v, g, beta, o (bf16 o), S0 in (if any), S_T out.
    FLOPs: per (value head, 64-token chunk) 5 * 2 C^2 D (A, W, U, Q K^T, P Vnew)
           + 3 * 2 C D^2 (W S, Q S, K^T Vnew) + C^3 / 3 (triangular inverse), C = 64.
    """
    b = 2 * L * Hk * D * 2 + L * Hv * D * 2 + 2 * L * Hv * 4 + L * Hv * D * 2
    b += Hv * D * D * 4 * (2 if s0 else 1)
    C = 64
    nc = -(-L // C)
    f = Hv * nc * (5 * 2 * C * C * D + 3 * 2 * C * D * D + C ** 3 / 3)
    return b, f


def kernel_bytes(L: int, Hk: int, Hv: int, s0: bool) -> dict:
    """Algorithmic bytes per launch of each kernel of the step: the prep kernel must read q, k (at
    the key heads), v, g and beta; the state kernel must read S0 and write o (bf16) and S_T."""
    prep = 2 * L * Hk * D * 2 + L * Hv * D * 2 + 2 * L * Hv * 4
    state = L * Hv * D * 2 + Hv * D * D * 4 * (2 if s0 else 1)
    return {"gdr_chunk_prep": prep, "gdr_chunk_state": state}


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def source_digest() -> str:
    """Digest of the sources of the prefill kernels (the tensor-core chunk path and its helpers)."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_deltanet_rule_gb300", "csrc")
    for name in ("gdr_chunk.cu", "gdr_internal.h", "gdr_inverse.cuh", "ptx.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per step from the committed ncu summary, if it was taken on the current sources."""
    path = os.path.join(ROOT, "profiles", f"dram_traffic_{workload}.md")
    if not os.path.exists(path):
        return None, None
    text = open(path).read()
    m = re.search(r"sources:\s*([0-9a-f]{16})", text)
    t = re.search(r"dram bytes per step:\s*([0-9]+)", text)
    if not m or not t or m.group(1) != source_digest():
        return None, None
    per_kernel = {k: int(v) for k, v in re.findall(r"^\|\s*(gdr_[a-z_0-9]+)\s*\|\s*([0-9]+)\s*\|", text, re.M)}
    return int(t.group(1)), per_kernel


# ------------------------------------------------------------------------------------------------
# distributed plumbing (also exercised by the CPU tests with gloo)
# ------------------------------------------------------------------------------------------------

def dist_env() -> tuple[int, int, int]:
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))


def reduce_max(x: float) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: float, seconds_this_rank: float) -> tuple[float, float]:
    """(whole-job units/s, max seconds over ranks): every rank processed units_per_rank."""
    import torch.distributed as dist
    n = dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1
    tmax = reduce_max(seconds_this_rank)
    return n * units_per_rank / tmax, tmax


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


# ------------------------------------------------------------------------------------------------
# clocks
# ------------------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
                except ValueError:
                    pass
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [r for r in rows if r[2] > 0.3 * max(x[2] for x in rows)] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(loaded), "power_w_max": max(r[2] for r in rows), "reasons": reasons}


# ------------------------------------------------------------------------------------------------
# GB300 arm
# ------------------------------------------------------------------------------------------------

def make_row(workload: str, seed: int):
    from gated_deltanet_rule_gb300 import inputs
    if workload == "prefill4096":
        return inputs.config3(seed=seed)
    if workload == "prefill8192":
        return inputs.config4(seed=seed)
    import torch
    L, Hk, Hv, s0, regime = WORKLOADS[workload]
    x = inputs.regime(regime, L, seed, Hk, Hv, D, init_state=s0, dtype=torch.bfloat16)
    x.meta["workload"] = f"{workload} bf16 L={L} Hk={Hk} Hv={Hv} D={D}"
    return x


def run_gb300(args) -> dict | None:
    import torch
    import torch.distributed as dist
    from gated_deltanet_rule_gb300 import gdr

    rank, local_rank, world = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    L, Hk, Hv, s0, _ = WORKLOADS[args.workload]

    x = make_row(args.workload, seed=3 + rank)
    host = [x.q, x.k, x.v, x.g, x.beta] + ([x.S0] if s0 else [])
    set_bytes = sum(t.numel() * t.element_size() for t in host)
    n_sets = max(2, -(-2 * L2_BYTES // set_bytes))       # resident copies, > 2x L2 in total
    sets = []
    for _ in range(n_sets):
        sets.append([t.to(dev, non_blocking=False).contiguous() for t in host])
    o = torch.empty_like(sets[0][2])
    S_T = torch.empty(1, Hv, D, D, device=dev, dtype=torch.float32)
    ws = torch.empty(max(1, gdr.workspace_bytes(1, L, Hk, Hv)), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(i):
        s = sets[i % n_sets]
        gdr.gdr_chunk_fwd(s[0], s[1], s[2], s[3], s[4], s[5] if s0 else None, o=o, S_T=S_T, ws=ws, stream=stream)

    for i in range(args.warmup):
        step(i)
    gdr.gdr_sync_status()

    # clocks: sample through a short untimed soak of the same step and through the timed steps
    sampler = ClockSampler(local_rank)
    sampler.start()
    t_end = time.time() + args.soak
    i = 0
    while time.time() < t_end:
        step(i)
        i += 1
        if i % 64 == 0:
            torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    gdr.gdr_sync_status()
    assert torch.isfinite(o.float()).all() and torch.isfinite(S_T).all()
    # per-kernel times: the same steps again with the library's stage timer, whose events between
    # the two launches keep the state kernel from starting early (so this pass is not the value)
    gdr.stage_timer_enable(True, 4 * args.steps + 16)
    for i in range(args.steps):
        step(i)
    torch.cuda.synchronize()
    stages = gdr.stage_timer_collect()
    gdr.stage_timer_enable(False, 0)
    gdr.gdr_sync_status()

    ms = e0.elapsed_time(e1) / args.steps
    value, tmax = aggregate(L * args.steps, ms * args.steps / 1e3)
    ms_max = tmax * 1e3 / args.steps
    launches = sum(c for _, c in stages.values())

    # e2e: host buffers through the same call, every step's copies inside the timed region. Two
    # device input sets and two output sets: step i's inputs go up on a copy stream while step i - 1
    # computes, and its o and S_T come back on another while step i + 1 computes (each copy waits
    # only for what it overwrites or reads). The serial form (copies and call on one stream) is
    # reported beside it.
    pinned = [t.pin_memory() for t in host]
    o_h = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    S_h = torch.empty(S_T.shape, dtype=S_T.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in pinned)
    d2h = o_h.numel() * o_h.element_size() + S_h.numel() * S_h.element_size()
    dbufs = [sets[0], sets[1]]
    outs = [(o, S_T), (torch.empty_like(o), torch.empty_like(S_T))]
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    ups, comps, downs = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def e2e_run(n, pipelined):
        if not pipelined:
            for _ in range(n):
                for d_, h_ in zip(dbufs[0], pinned):
                    d_.copy_(h_, non_blocking=True)
                gdr.gdr_chunk_fwd(*dbufs[0][:5], dbufs[0][5] if s0 else None, o=o, S_T=S_T, ws=ws, stream=stream)
                o_h.copy_(o, non_blocking=True)
                S_h.copy_(S_T, non_blocking=True)
            return
        start = ev()
        start.record(stream)
        up.wait_event(start)
        down.wait_event(start)
        for i in range(n):
            j = i % 2
            buf, (o_d, S_d) = dbufs[j], outs[j]
            if i >= 2:
                up.wait_event(comps[j])        # step i - 2 has read this input set
            with torch.cuda.stream(up):
                for d_, h_ in zip(buf, pinned):
                    d_.copy_(h_, non_blocking=True)
                ups[j].record(up)
            stream.wait_event(ups[j])
            if i >= 2:
                stream.wait_event(downs[j])    # step i - 2's outputs have been read back
            gdr.gdr_chunk_fwd(*buf[:5], buf[5] if s0 else None, o=o_d, S_T=S_d, ws=ws, stream=stream)
            comps[j].record(stream)
            down.wait_event(comps[j])
            with torch.cuda.stream(down):
                o_h.copy_(o_d, non_blocking=True)
                S_h.copy_(S_d, non_blocking=True)
                downs[j].record(down)
        stream.wait_event(downs[(n - 1) % 2])
        if n >= 2:
            stream.wait_event(downs[(n - 2) % 2])

    e2e = {}
    for name, pipelined in (("serial", False), ("pipelined", True)):
        e2e_run(max(3, args.warmup), pipelined)
        torch.cuda.synchronize()
        barrier()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        e2e_run(args.steps, pipelined)
        f1.record(stream)
        torch.cuda.synchronize()
        e2e[name], _ = aggregate(L * args.steps, f0.elapsed_time(f1) / 1e3)
        barrier()
    gdr.gdr_sync_status()
    e2e_value = e2e["pipelined"]

    peaks = measured_peaks()
    alg_bytes, alg_flops = algorithmic(L, Hk, Hv, s0)
    t_s = ms_max / 1e3
    hbm_time = alg_bytes / (peaks["hbm_gbs"] * 1e9)
    tc_time = alg_flops / (peaks["bf16_tflops"] * 1e12)
    bound = "hbm" if hbm_time >= tc_time else "tensor"
    achieved = alg_bytes / t_s / 1e9 if bound == "hbm" else alg_flops / t_s / 1e12
    peak = peaks["hbm_gbs"] if bound == "hbm" else peaks["bf16_tflops"]
    traffic, traffic_k = profiled_traffic(args.workload)
    kern = {}
    total_stage = sum(v[0] for v in stages.values()) or 1.0
    for name, (tot, cnt) in stages.items():
        if cnt:
            kern[name] = {"launches": cnt, "avg_us": round(tot / cnt * 1e3, 2), "share": round(tot / total_stage, 4)}
    # the dominant kernel's own roofline: the algorithmic bytes it must move per launch
    share = kernel_bytes(L, Hk, Hv, s0)
    dom = max(kern, key=lambda k: kern[k]["share"])
    dom_bytes = share[dom]
    dom_gbs = dom_bytes / (kern[dom]["avg_us"] * 1e-6) / 1e9

    if rank != 0:
        return None
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": x.meta.get("workload"), "L": L, "Hk": Hk, "Hv": Hv, "D": D, "rows_per_gpu": 1,
                   "S0": s0, "parallelism": f"replicas x{world}" if world > 1 else "single gpu",
                   "l2": f"{n_sets} resident input sets of {set_bytes / 2**20:.0f} MiB rotated (> L2)"},
        "roofline": {"bound": "hbm", "achieved": round(dom_gbs, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(dom_gbs / peaks["hbm_gbs"], 4),
                     "traffic": (traffic_k or {}).get(dom) if traffic is not None else None,
                     "kernel": dom, "algorithmic_bytes": dom_bytes,
                     "peak_source": f"MEASURED_PEAKS.json ({peaks['source']}, burst copy)",
                     "path": {"bound": bound, "achieved": round(achieved, 2), "peak": peak,
                              "unit": "GB/s" if bound == "hbm" else "TFLOP/s", "frac": round(achieved / peak, 4),
                              "traffic": traffic, "scope": "whole step (all kernels of the path)",
                              "algorithmic_bytes": alg_bytes, "algorithmic_flops": alg_flops}},
        "kernels": kern,
        "clocks": clocks,
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": "double-buffered: a step's uploads overlap the previous step's call, its downloads "
                          "the next step's",
                "serial_value": round(e2e["serial"], 1)},
        "gpu_launches": launches,
    }
    if traffic_k:
        line["roofline"]["traffic_per_kernel"] = traffic_k
    if world == 1 and not args.no_rows:
        line["rows"] = run_fork_decode(reps=max(3, min(args.steps, 20)), warmup=args.warmup)
        line["rows"]["next_f1_prologue"] = run_prologue(reps=max(3, min(args.steps, 50)), warmup=args.warmup)
        line["rows"]["next_f1_prologue"]["fused_into_prefill"] = run_fused_prologue(
            reps=max(3, min(args.steps, 20)), warmup=args.warmup)
        line["rows"]["next_f2_gated_rmsnorm"] = run_epilogue(reps=max(3, min(args.steps, 50)), warmup=args.warmup)
        line["rows"]["next_f2_gated_rmsnorm"]["fused_into_prefill"] = run_gated_prefill(
            reps=max(3, min(args.steps, 20)), warmup=args.warmup)
        line["rows"]["next_f4_backward"] = run_backward(reps=max(3, min(args.steps, 10)), warmup=args.warmup)
        line["rows"]["configs"] = run_configs(reps=max(3, min(args.steps, 50)), warmup=args.warmup)
        line["rows"]["next_f3_varlen"] = run_varlen(reps=max(3, min(args.steps, 20)), warmup=args.warmup)
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, budget_s=args.cpu_budget)
    return line


# ------------------------------------------------------------------------------------------------
# the other rows of the path: the fork pass and the decode step (one trunk state, 256 forks)
# ------------------------------------------------------------------------------------------------

def fork_decode_bytes(F: int, L_pad: int, Hk: int, Hv: int, N: int) -> tuple[int, int]:
    """Algorithmic bytes of one fork pass and of one decode step (bf16 q/k/v/o, fp32 gates/states).

    Fork pass: q, k at the key heads, v, o, g, beta for every padded position, the trunk states read
    once, every fork's final state written. Decode step: one token of q, k, v, o, g, beta per fork and
    the fork states read and written in place.
    """
    st = Hv * D * D * 4
    fork = F * L_pad * (2 * Hk * D * 2 + 2 * Hv * D * 2 + 2 * Hv * 4) + N * st + F * st
    dec = F * (2 * Hk * D * 2 + 2 * Hv * D * 2 + 2 * Hv * 4) + 2 * F * st
    return fork, dec


def run_fork_decode(reps: int, warmup: int) -> dict:
    """Times rows a6 (fork pass) and a7 (decode step) of the hot path on the fork workload."""
    import torch
    from gated_deltanet_rule_gb300 import gdr, inputs
    x = inputs.config5()
    f = x.fork
    d = lambda t: t.cuda().contiguous()
    q, k, v, g, beta = (d(t) for t in (f.q, f.k, f.v, f.g, f.beta))
    trunk, idx = d(x.trunk), d(x.trunk_idx)
    F, L_pad, Hk, _ = q.shape
    Hv = v.shape[2]
    o = torch.empty_like(v)
    states = torch.empty(F, Hv, D, D, device="cuda", dtype=torch.float32)
    dec = [[d(t) for t in (s.q, s.k, s.v, s.g, s.beta)] for s in x.decode]
    od = torch.empty_like(dec[0][2])
    stream = torch.cuda.current_stream()
    peaks = measured_peaks()
    fb, db = fork_decode_bytes(F, L_pad, Hk, Hv, trunk.shape[0])

    ws = torch.empty(max(1, gdr.fork_workspace_bytes(F, L_pad, Hk, Hv)), dtype=torch.uint8, device="cuda")

    def fork_pass():
        gdr.gdr_fork_fwd(q, k, v, g, beta, trunk, idx, o=o, states_out=states, stream=stream, ws=ws)

    def decode_round():
        for s in dec:
            gdr.gdr_decode_step(s[0], s[1], s[2], s[3], s[4], states, o=od, stream=stream)

    out = {}
    for name, fn, per, nbytes, tok in (("a6_fork_pass", fork_pass, 1, fb, int(x.lengths.sum())),
                                       ("a7_decode_step", decode_round, len(dec), db, F)):
        for _ in range(warmup):
            fn()
        gdr.gdr_sync_status()
        gdr.stage_timer_enable(True, 4 * reps * per + 16)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        stages = gdr.stage_timer_collect()
        gdr.stage_timer_enable(False, 0)
        gdr.gdr_sync_status()
        us = e0.elapsed_time(e1) * 1e3 / (reps * per)
        gbs = nbytes / (us * 1e-6) / 1e9
        out[name] = {
            "us_per_call": round(us, 2), "tokens_per_s": round(tok / (us * 1e-6), 1),
            "tokens": "real tokens of the fork batch" if per == 1 else "one token per fork",
            "roofline": {"bound": "hbm", "achieved": round(gbs, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "algorithmic_bytes": nbytes},
            "kernels": {kname: {"launches": c, "avg_us": round(t / c * 1e3, 2)} for kname, (t, c) in stages.items() if c},
        }
    assert torch.isfinite(states).all() and torch.isfinite(o.float()).all()
    out["workload"] = x.meta["workload"] + f" (F={F}, Hk={Hk}, Hv={Hv}, D={D}, bf16 q/k/v)"
    return out


def _graph_us(call, reps: int, per_graph: int = 24) -> float:
    """GPU microseconds per call of call(stream), from CUDA-graph replays of per_graph calls (no
    Python or launch overhead between the kernels: a 15-35 us kernel launched from a Python loop is
    bound by the loop)."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(per_graph):
            call(s)
    cur = torch.cuda.current_stream()
    g.replay()
    cur.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(1, reps // per_graph + 1)
    e0.record(cur)
    for _ in range(n):
        g.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (n * per_graph)


def run_prologue(reps: int, warmup: int) -> dict:
    """Times the GDN prologue (the first adjacent row: conv + SiLU, gates, carry) on the prefill
    row's shapes, L = 4096, 16 -> 32 heads, K = 4, with its HBM roofline."""
    import torch
    from gated_deltanet_rule_gb300 import gdr, inputs
    K, L, Hk, Hv = 4, 4096, 16, 32
    x = inputs.prologue_inputs(1, L, 3, Hk=Hk, Hv=Hv, K=K)
    d = lambda t: t.cuda().contiguous()
    mixed, w, a, b, A_log, dt_bias, tail = (d(t) for t in (x.mixed, x.conv_w, x.a, x.b, x.A_log, x.dt_bias, x.tail))
    C = mixed.shape[2]
    # two input and output sets (272 MB, over twice the L2), used in turn
    sets = [(mixed, a, b, tail), tuple(t.clone() for t in (mixed, a, b, tail))]
    outs = [gdr.gdr_prologue(m_, w, a_, b_, A_log, dt_bias, Hk, Hv, tail=t_) for m_, a_, b_, t_ in sets]
    stream = torch.cuda.current_stream()
    turn = [0]

    def call(st=stream):
        j = turn[0] = turn[0] ^ 1
        (m_, a_, b_, t_), o_ = sets[j], outs[j]
        gdr.gdr_prologue(m_, w, a_, b_, A_log, dt_bias, Hk, Hv, tail=t_, q=o_[0], k=o_[1], v=o_[2], g=o_[3],
                         beta=o_[4], new_tail=o_[5], stream=st)

    # algorithmic bytes: mixed and tail read, q, k, v and the carry written (bf16); a, b read and
    # g, beta written (float32); the weights
    nbytes = (L + K - 1) * C * 2 + L * C * 2 + (K - 1) * C * 2 + 4 * L * Hv * 4 + C * K * 4 + 2 * Hv * 4
    for _ in range(warmup):
        call()
    gdr.gdr_sync_status()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    us_eager = e0.elapsed_time(e1) * 1e3 / reps
    us = _graph_us(call, reps)
    # the kernel's own time from a second pass with the stage timer (its events add a little)
    gdr.stage_timer_enable(True, 4 * reps + 16)
    for _ in range(reps):
        call()
    torch.cuda.synchronize()
    stages = gdr.stage_timer_collect()
    gdr.stage_timer_enable(False, 0)
    gdr.gdr_sync_status()
    gbs = nbytes / (us * 1e-6) / 1e9
    peaks = measured_peaks()
    assert all(torch.isfinite(o_[3]).all() and torch.isfinite(o_[0].float()).all() for o_ in outs)
    return {"us_per_call": round(us, 2), "tokens_per_s": round(L / (us * 1e-6), 1),
            "timing": "CUDA-graph replays of 24 calls over input sets larger than L2 in turn; us_per_call_eager: "
                      "the same calls from a Python loop",
            "us_per_call_eager": round(us_eager, 2),
            "workload": f"GDN prologue L={L} Hk={Hk} Hv={Hv} D={D} K={K} (conv + SiLU, gates, carry), bf16",
            "roofline": {"bound": "hbm", "achieved": round(gbs, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "algorithmic_bytes": nbytes},
            "kernels": {kname: {"launches": c, "avg_us": round(t / c * 1e3, 2)} for kname, (t, c) in stages.items() if c}}


def run_epilogue(reps: int, warmup: int) -> dict:
    """Times the gated RMSNorm epilogue (the second adjacent row) on the prefill row's output,
    o [1, 4096, 32, 128] bf16 with its gate z, with its HBM roofline."""
    import torch
    from gated_deltanet_rule_gb300 import gdr
    L, Hv = 4096, 32
    gen = torch.Generator().manual_seed(3)
    x = torch.randn(1, L, Hv, D, generator=gen).bfloat16().cuda()
    z = torch.randn(1, L, Hv, D, generator=gen).bfloat16().cuda()
    w = (0.5 + torch.rand(D, generator=gen)).cuda()
    # three (x, z, out) sets (302 MB, over twice the L2), used in turn
    sets = [(x, z, torch.empty_like(x))] + [(x.clone(), z.clone(), torch.empty_like(x)) for _ in range(2)]
    out = sets[0][2]
    stream = torch.cuda.current_stream()
    nbytes = 3 * x.numel() * 2 + D * 4   # x and z read, out written (bf16), the weight
    turn = [0]

    def call(st=stream):
        turn[0] = (turn[0] + 1) % 3
        x_, z_, o_ = sets[turn[0]]
        gdr.gdr_gated_rmsnorm(x_, z_, w, 1e-6, out=o_, stream=st)

    for _ in range(warmup):
        call()
    gdr.gdr_sync_status()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    us_eager = e0.elapsed_time(e1) * 1e3 / reps
    us = _graph_us(call, reps)
    gdr.stage_timer_enable(True, 4 * reps + 16)
    for _ in range(reps):
        call()
    torch.cuda.synchronize()
    stages = gdr.stage_timer_collect()
    gdr.stage_timer_enable(False, 0)
    gdr.gdr_sync_status()
    gbs = nbytes / (us * 1e-6) / 1e9
    peaks = measured_peaks()
    assert torch.isfinite(out.float()).all()
    return {"us_per_call": round(us, 2), "tokens_per_s": round(L / (us * 1e-6), 1),
            "timing": "CUDA-graph replays of 24 calls over input sets larger than L2 in turn; us_per_call_eager: "
                      "the same calls from a Python loop",
            "us_per_call_eager": round(us_eager, 2),
            "workload": f"gated RMSNorm over o [1, {L}, {Hv}, {D}] bf16 with gate z",
            "roofline": {"bound": "hbm", "achieved": round(gbs, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "algorithmic_bytes": nbytes},
            "kernels": {kname: {"launches": c, "avg_us": round(t / c * 1e3, 2)} for kname, (t, c) in stages.items() if c}}


def run_backward(reps: int, warmup: int) -> dict:
    """Times the backward on the prefill workload, L = 4096, Hk = 16, Hv = 32, bf16 q, k, v, dO,
    with dS_T: gdr_backward_chunked (the chunked tensor-core form: forward factors, chunk-entry
    states, Nb = Q'^T dO, the adjoint chain, the chunk-local gradients, the key-head reduction) as
    the row, and gdr_backward (the checkpointed float32 token loop) beside it. The HBM roofline
    counts the algorithmic bytes: q, k, v, dO, g, beta, dS_T read once, every gradient written once."""
    import torch
    from gated_deltanet_rule_gb300 import gdr, inputs
    L, Hk, Hv = 4096, 16, 32
    x = inputs.regime("R1", L, 3, Hk=Hk, Hv=Hv, B=1, dtype=torch.bfloat16)
    dO, dS_T = inputs.upstream_grads(1, L, Hv, 4, dtype=torch.bfloat16)
    q, k, v, g, beta, dO, dS_T = (t.cuda() for t in (x.q, x.k, x.v, x.g, x.beta, dO, dS_T))
    stream = torch.cuda.current_stream()
    nbytes = (2 * L * Hk * D * 2 + 2 * L * Hv * D * 2 + 2 * L * Hv * 4 + Hv * D * D * 4       # inputs
              + 2 * L * Hk * D * 4 + L * Hv * D * 4 + 2 * L * Hv * 4 + Hv * D * D * 4)       # gradients
    peaks = measured_peaks()
    workload = f"backward of the prefill row [1, {L}], Hk={Hk}, Hv={Hv}, D={D}, bf16 q/k/v/dO, float32 gradients"

    def timed(fn, ws_bytes):
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        out = []

        def call(_i):
            out[:] = fn(q, k, v, g, beta, None, dO, dS_T, ws=ws, stream=stream)
        us, stages = _time_calls(call, reps, warmup, stream)
        gdr.gdr_sync_status()
        assert all(torch.isfinite(t).all() for t in out if t is not None)
        del ws
        gbs = nbytes / (us * 1e-6) / 1e9
        return {"us_per_call": round(us, 2), "tokens_per_s": round(L / (us * 1e-6), 1),
                "roofline": {"bound": "hbm", "achieved": round(gbs, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": round(gbs / peaks["hbm_gbs"], 4), "algorithmic_bytes": nbytes},
                "kernels": stages}

    row = timed(gdr.gdr_backward_chunked, gdr.backward_chunked_workspace_bytes(1, L, Hk, Hv))
    row["workload"] = workload
    row["roofline"]["note"] = ("latency of the sequential passes (the forward's chunk chain again and the adjoint "
                               "chain, 64 steps each) and of the chunk-local products; far from this roofline")
    loop = timed(gdr.gdr_backward, gdr.backward_workspace_bytes(1, L, Hk, Hv))
    loop["roofline"]["note"] = "a sequential token loop on CUDA cores: latency-bound, far from this roofline"
    row["token_loop_float32"] = loop
    # a training step's forward + backward: checkpointed (gdr_chunk_fwd, then the backward recomputes
    # the forward's passes) against kept intermediates (gdr_chunk_fwd_save, gdr_backward_chunked_saved)
    wsb = gdr.backward_chunked_workspace_bytes(1, L, Hk, Hv)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    fws = torch.empty(max(1, gdr.workspace_bytes(1, L, Hk, Hv)), dtype=torch.uint8, device="cuda")
    o = torch.empty_like(v)
    S_T = torch.empty(1, Hv, D, D, dtype=torch.float32, device="cuda")

    def recompute(_i):
        gdr.gdr_chunk_fwd(q, k, v, g, beta, None, o=o, S_T=S_T, ws=fws, stream=stream)
        gdr.gdr_backward_chunked(q, k, v, g, beta, None, dO, dS_T, ws=ws, stream=stream)

    def keep(_i):
        gdr.gdr_chunk_fwd_save(q, k, v, g, beta, None, saved=ws, o=o, S_T=S_T, stream=stream)
        gdr.gdr_backward_chunked(q, k, v, g, beta, None, dO, dS_T, saved=ws, stream=stream)

    step = {"workload": f"forward + backward of the prefill row [1, {L}], Hk={Hk}, Hv={Hv}, D={D}, bf16",
            "saved_bytes": wsb}
    for name, fn in (("checkpointed", recompute), ("kept_intermediates", keep)):
        us, stages = _time_calls(fn, reps, warmup, stream)
        step[name] = {"us_per_step": round(us, 2), "tokens_per_s": round(L / (us * 1e-6), 1), "kernels": stages}
    gdr.gdr_sync_status()
    row["training_step"] = step
    return row


def _time_calls(fn, reps: int, warmup: int, stream) -> tuple[float, dict]:
    """Average microseconds per call of fn (CUDA events on `stream` around `reps` calls), then the
    library's per-kernel stage times from a second pass."""
    import torch
    from gated_deltanet_rule_gb300 import gdr
    for _ in range(warmup):
        fn(0)
    gdr.gdr_sync_status()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(reps):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / reps
    gdr.stage_timer_enable(True, 8 * reps + 16)
    for i in range(reps):
        fn(i)
    torch.cuda.synchronize()
    stages = gdr.stage_timer_collect()
    gdr.stage_timer_enable(False, 0)
    gdr.gdr_sync_status()
    return us, {kname: {"launches": c, "avg_us": round(t / c * 1e3, 2)} for kname, (t, c) in stages.items() if c}


def run_gated_prefill(reps: int, warmup: int) -> dict:
    """Times the gated RMSNorm fused into the prefill's output (gdr_chunk_fwd_gated) on the prefill
    row (L = 4096, 16 -> 32 heads, bf16, S0) against the same prefill followed by the separate
    gdr_gated_rmsnorm pass over its o."""
    import torch
    from gated_deltanet_rule_gb300 import gdr, inputs
    x = inputs.config3()
    q, k, v, g, beta, S0 = (t.cuda().contiguous() for t in (x.q, x.k, x.v, x.g, x.beta, x.S0))
    gen = torch.Generator().manual_seed(9)
    z = torch.randn(v.shape, generator=gen).bfloat16().cuda()
    w = (0.5 + torch.rand(D, generator=gen)).cuda()
    L, Hk, Hv = q.shape[1], q.shape[2], v.shape[2]
    o = torch.empty_like(v)
    out = torch.empty_like(v)
    S_T = torch.empty_like(S0)
    ws = torch.empty(gdr.workspace_bytes(1, L, Hk, Hv), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def fused(i):
        gdr.gdr_chunk_fwd_gated(q, k, v, g, beta, S0, z, w, 1e-6, out=out, S_T=S_T, ws=ws, stream=stream)

    def separate(i):
        gdr.gdr_chunk_fwd(q, k, v, g, beta, S0, o=o, S_T=S_T, ws=ws, stream=stream)
        gdr.gdr_gated_rmsnorm(o, z, w, 1e-6, out=out, stream=stream)

    res = {"workload": f"prefill L={L} Hk={Hk} Hv={Hv} D={D} bf16 with S0, then the gated RMSNorm of its output"}
    for name, fn in (("fused", fused), ("separate_pass", separate)):
        us, kern = _time_calls(fn, reps, warmup, stream)
        res[name] = {"us_per_call": round(us, 2), "tokens_per_s": round(L / (us * 1e-6), 1), "kernels": kern}
    return res


def run_fused_prologue(reps: int, warmup: int) -> dict:
    """Times the GDN prologue fused into the prefill (gdr_chunk_fwd_prologue: q, k, v, g, beta formed
    inside the chunk kernel) on the prefill row (L = 4096, 16 -> 32 heads, K = 4, with a carry and
    S0) against gdr_prologue followed by gdr_chunk_fwd on its outputs."""
    import torch
    from gated_deltanet_rule_gb300 import gdr, inputs
    K, L, Hk, Hv = 4, 4096, 16, 32
    x = inputs.prologue_inputs(1, L, 3, Hk=Hk, Hv=Hv, K=K)
    d = lambda t: t.cuda().contiguous()
    mixed, w, a, b, A_log, dt_bias, tail = (d(t) for t in (x.mixed, x.conv_w, x.a, x.b, x.A_log, x.dt_bias, x.tail))
    gen = torch.Generator().manual_seed(8)
    S0 = (0.1 * torch.randn(1, Hv, D, D, generator=gen)).cuda()
    pro = gdr.gdr_prologue(mixed, w, a, b, A_log, dt_bias, Hk, Hv, tail=tail)
    o = torch.empty(1, L, Hv, D, dtype=torch.bfloat16, device="cuda")
    S_T = torch.empty_like(S0)
    new_tail = torch.empty_like(tail)
    ws = torch.empty(max(gdr.workspace_bytes(1, L, Hk, Hv), gdr.prologue_workspace_bytes(1, L, Hk, Hv, K)),
                     dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def fused(i):
        gdr.gdr_chunk_fwd_prologue(mixed, w, a, b, A_log, dt_bias, Hk, Hv, S0=S0, tail=tail, o=o, S_T=S_T,
                                   new_tail=new_tail, ws=ws, stream=stream)

    def separate(i):
        gdr.gdr_prologue(mixed, w, a, b, A_log, dt_bias, Hk, Hv, tail=tail, q=pro[0], k=pro[1], v=pro[2], g=pro[3],
                         beta=pro[4], new_tail=new_tail, stream=stream)
        gdr.gdr_chunk_fwd(pro[0], pro[1], pro[2], pro[3], pro[4], S0, o=o, S_T=S_T, ws=ws, stream=stream)

    res = {"workload": f"GDN prologue (conv + SiLU, gates, carry) L={L} Hk={Hk} Hv={Hv} D={D} K={K}, then the "
                       f"prefill with S0, bf16"}
    for name, fn in (("fused", fused), ("separate_pass", separate)):
        us, kern = _time_calls(fn, reps, warmup, stream)
        res[name] = {"us_per_call": round(us, 2), "tokens_per_s": round(L / (us * 1e-6), 1), "kernels": kern}
    return res


def run_varlen(reps: int, warmup: int) -> dict:
    """Times the variable-length prefill (next row f3): 4 right-padded rows of 4096 positions with
    4096, 1000, 1 and 2048 valid tokens at the prefill shapes (16 -> 32 heads, bf16, S0), once with
    their lengths (gdr_chunk_fwd_varlen: chunks past a row's length are skipped) and once as plain
    rows whose pads carry beta = g = 0 (every chunk run). tokens_per_s counts valid tokens."""
    import torch
    from gated_deltanet_rule_gb300 import gdr, inputs
    lens = [4096, 1000, 1, 2048]
    B, L, Hk, Hv = len(lens), 4096, 16, 32
    x = inputs.regime("R1", L, 5, Hk=Hk, Hv=Hv, B=B, init_state=True, dtype=torch.bfloat16)
    for r, n in enumerate(lens):
        x.g[r, n:] = 0.0
        x.beta[r, n:] = 0.0
    q, k, v, g, beta, S0 = (t.cuda().contiguous() for t in (x.q, x.k, x.v, x.g, x.beta, x.S0))
    lengths = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o = torch.empty_like(v)
    S_T = torch.empty_like(S0)
    ws = torch.empty(gdr.workspace_bytes(B, L, Hk, Hv), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    out = {"workload": f"{B} rows of {L} positions, lengths {lens}, Hk={Hk} Hv={Hv} D={D}, bf16, S0"}
    for name, ln in (("with_lengths", lengths), ("all_positions", None)):
        def call(i, ln=ln):
            gdr.gdr_chunk_fwd(q, k, v, g, beta, S0, o=o, S_T=S_T, ws=ws, stream=stream, lengths=ln)
        us, kern = _time_calls(call, reps, warmup, stream)
        out[name] = {"us_per_call": round(us, 2), "tokens_per_s": round(sum(lens) / (us * 1e-6), 1), "kernels": kern}
    return out


def run_configs(reps: int, warmup: int) -> dict:
    """Times the other workloads of the path: the long prefill (L = 8192, 16 = 16 heads, bf16, weak
    decay, no initial state; its own HBM roofline) and the two float32 parity workloads (L = 64 and
    the padded L = 130 row with an initial state; time only, no roofline: the float32 path is the
    token loop on CUDA cores, whose FFMA peak is not measured)."""
    import torch
    from gated_deltanet_rule_gb300 import gdr, inputs
    stream = torch.cuda.current_stream()
    peaks = measured_peaks()
    out = {}
    # long prefill: input sets rotated so that their total exceeds L2
    x = inputs.config4()
    L, Hk, Hv = x.q.shape[1], x.q.shape[2], x.v.shape[2]
    host = [x.q, x.k, x.v, x.g, x.beta]
    set_bytes = sum(t.numel() * t.element_size() for t in host)
    n_sets = max(2, -(-2 * L2_BYTES // set_bytes))
    sets = [[t.cuda().contiguous() for t in host] for _ in range(n_sets)]
    o = torch.empty_like(sets[0][2])
    S_T = torch.empty(1, Hv, D, D, device="cuda", dtype=torch.float32)
    ws = torch.empty(max(1, gdr.workspace_bytes(1, L, Hk, Hv)), dtype=torch.uint8, device="cuda")

    def long_row(i):
        s = sets[i % n_sets]
        gdr.gdr_chunk_fwd(s[0], s[1], s[2], s[3], s[4], None, o=o, S_T=S_T, ws=ws, stream=stream)

    us, kern = _time_calls(long_row, reps, warmup, stream)
    nbytes, nflops = algorithmic(L, Hk, Hv, False)
    gbs = nbytes / (us * 1e-6) / 1e9
    assert torch.isfinite(o.float()).all() and torch.isfinite(S_T).all()
    out["config4_prefill8192"] = {
        "us_per_call": round(us, 2), "tokens_per_s": round(L / (us * 1e-6), 1),
        "workload": f"{x.meta['workload']} ({n_sets} resident input sets rotated, > L2)",
        "roofline": {"bound": "hbm", "achieved": round(gbs, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(gbs / peaks["hbm_gbs"], 4), "algorithmic_bytes": nbytes,
                     "algorithmic_flops": nflops},
        "kernels": kern}
    del sets, o, ws
    # float32 parity workloads (tiny; they stay in L2)
    for name, x in (("config1_fp32_L64", inputs.config1()), ("config2_fp32_L130_padded", inputs.config2("a"))):
        q, k, v, g, beta = (t.cuda().contiguous() for t in (x.q, x.k, x.v, x.g, x.beta))
        S0 = None if x.S0 is None else x.S0.cuda().contiguous()
        o = torch.empty_like(v)
        S_T = torch.empty(q.shape[0], v.shape[2], D, D, device="cuda", dtype=torch.float32)

        def call(i):
            gdr.gdr_chunk_fwd(q, k, v, g, beta, S0, o=o, S_T=S_T, stream=stream)

        us, kern = _time_calls(call, reps, warmup, stream)
        L = q.shape[1]
        out[name] = {"us_per_call": round(us, 2), "tokens_per_s": round(q.shape[0] * L / (us * 1e-6), 1),
                     "workload": f"{x.meta.get('workload', name)}: float32 q/k/v, L={L}, {q.shape[2]}->{v.shape[2]} heads "
                                 "(time only; inputs L2-resident)",
                     "kernels": kern}
    return out


# ------------------------------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ------------------------------------------------------------------------------------------------

def oracle_sample(workload: str, tokens: int):
    """The workload's row (seed 3) restricted to its first `tokens` positions (all heads)."""
    x = make_row(workload, seed=3)
    L = x.q.shape[1]
    t = min(L, tokens)
    args = tuple(None if a is None else a[:, :t].contiguous() for a in (x.q, x.k, x.v, x.g, x.beta))
    return args + (x.S0,), t, x.meta.get("workload")


def cpu_baseline(workload: str, budget_s: float = 20.0) -> dict:
    import oracle
    L, Hk, Hv, s0, _ = WORKLOADS[workload]
    args, tokens, _ = oracle_sample(workload, L)
    t0 = time.perf_counter()
    oracle.forward(*args)
    dt = time.perf_counter() - t0
    reps = [dt]
    while sum(reps) < budget_s / 2 and len(reps) < 3:
        t0 = time.perf_counter()
        oracle.forward(*args)
        reps.append(time.perf_counter() - t0)
    t = statistics.median(reps)
    return {"value": round(tokens / t, 1), "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"the full row (L={L}, {Hk}->{Hv} heads) once per run, float64 oracle, median of {len(reps)} runs"}


def run_reference(args) -> dict | None:
    rank, _, world = dist_env()
    if rank != 0:
        return None
    import oracle
    L, Hk, Hv, s0, _ = WORKLOADS[args.workload]
    sample, tokens, wname = oracle_sample(args.workload, max(64, L // 4))   # bounded sample per step
    for _ in range(args.warmup):
        oracle.forward(*sample)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.forward(*sample)
    dt = time.perf_counter() - t0
    value = tokens * args.steps / dt
    desc = f"the first {tokens} of the row's {L} tokens, all {Hk}->{Hv} heads, per step (float64 oracle)"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wname, "L": L, "Hk": Hk, "Hv": Hv, "D": D},
        "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="prefill4096")
    ap.add_argument("--soak", type=float, default=1.5, help="seconds of untimed steps while clocks are sampled")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-rows", action="store_true", help="skip the fork-pass and decode-step rows")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    line = run_reference(args) if args.impl == "reference" else run_gb300(args)
    if line is not None:
        print(json.dumps(line), flush=True)
    try:
        import torch.distributed as dist
        if dist.is_available() and dist.is_initialized():
            dist.destroy_process_group()
    except Exception:
        pass


if __name__ == "__main__":
    main()
