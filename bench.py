#!/usr/bin/env python
"""Benchmark of the masked HLA-2 forward on the long-context workload.

Workload: B=1, H=16, n=65536, d=dv=64, bf16 inputs, fp32 state, unnormalised, per-head
decay linspace(0.99, 0.9999), chunk width 128 (1,048,576 tokens per step; 536.9 MB of
algorithmic traffic, larger than the 129 MB L2, so no flush is needed between steps).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

After the timed headline it measures more rows of the path on their own workloads
(reported under "secondary"): the decode step (256 sequences x 32 heads, d = dv = 128) on
the packed and on the compact state, a training step (forward + backward, B=4 H=16
n=8192 d = dv = 128), and the asymmetric variant (AHLA) on the long-context shapes.

Prints one JSON line (rank 0).  Under torchrun (N > 1) every rank runs its own replica
of the workload (weak scaling, no collective in the data path); the timed region is
bracketed by barriers and the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "HLA-2 masked fwd tokens/s (B·H·n/s) at n=64K,d=64; % tensor/HBM roofline"
WORKLOAD = "long"
CONFIG_NAME = ("long-context masked HLA-2 forward: B=1 H=16 n=65536 d=dv=64 bf16 in/out, "
               "fp32 state, decay linspace(0.99,0.9999), unnormalised, chunk 128")
PHASES = ("carry_init", "segment_summaries", "segment_scan", "output_pass", "final_state")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the decode and training rows measured after the headline")
    ap.add_argument("--only", choices=("decode", "decode_compact", "decode_unmasked", "decode_mq", "train", "ahla",
                                       "unmasked", "hla3", "prefill", "train_d64", "ahla_backward", "normed",
                                       "prefill_d128", "normed_backward"),
                    default=None,
                    help="measure only this row (for profiler captures; --steps/--warmup apply)")
    ap.add_argument("--decode-seqs", type=int, default=256,
                    help="sequences of the decode row (smaller case for ncu --set full captures)")
    ap.add_argument("--chunk", type=int, default=None,
                    help="chunk width of the unmasked row (--only unmasked)")
    ap.add_argument("--n", type=int, default=None,
                    help="override the sequence length (smaller case for ncu --set full captures; "
                         "the reported metric is only valid at the default)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


# ---------------------------------------------------------------------------------
# distributed plumbing (control plane only)
# ---------------------------------------------------------------------------------

class Dist:
    def __init__(self, backend):
        import torch
        import torch.distributed as dist
        self.dist = dist
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.on = self.world > 1
        if self.on:
            dist.init_process_group(backend=backend)
        self.torch = torch

    def barrier(self):
        if self.on:
            self.dist.barrier()

    def max(self, x: float) -> float:
        if not self.on:
            return x
        t = self.torch.tensor([x], dtype=self.torch.float64,
                              device="cuda" if self.dist.get_backend() == "nccl" else "cpu")
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.on:
            self.dist.destroy_process_group()


def replica_seed(base: int, rank: int) -> int:
    """Seed of rank ``rank``'s replica: every rank draws its own copy of the workload."""
    return base + 1000 * rank


def weak_scaling_value(world: int, tokens_per_rank: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: all ranks' tokens over the slowest rank's time per step."""
    return world * tokens_per_rank / (ms_per_step * 1e-3)


# ---------------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.fh = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        self.t0 = time.time()

    def mark(self):
        return time.time()

    def stop(self, t_begin, t_end):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.flush()
        self.fh.seek(0)
        rows = [r.strip().split(",") for r in self.fh.read().splitlines() if r.strip()]
        os.unlink(self.fh.name)
        if not rows:
            return None
        # nvidia-smi prints at a fixed period; map rows to wall time linearly
        n = len(rows)
        span = max(t_end, time.time()) - self.t0
        times = [self.t0 + span * (i + 0.5) / n for i in range(n)]
        inside = [r for r, t in zip(rows, times) if t_begin <= t <= t_end] or rows[-3:]
        sm = [float(r[1]) for r in inside if r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in inside if r[2].strip().replace(".", "").isdigit()]
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in inside:
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(inside)}


# ---------------------------------------------------------------------------------
# CPU oracle timing (baseline / reference arm)
# ---------------------------------------------------------------------------------

def oracle_sample(target_s: float):
    """Time the float64 C oracle on the workload for about ``target_s`` seconds: the first
    n_s tokens of every head (n_s <= n), repeated when one pass is shorter than the
    target.  Returns (tokens/s, cores, description)."""
    import torch

    from chunked_scan_mixer_gb300 import inputs
    from oracle import cref

    w = inputs.WORKLOADS[WORKLOAD]
    cref.build()
    g = inputs.gammas(w).double().numpy()
    f = lambda t: t.to(torch.float32).numpy()  # noqa: E731
    probe = 256
    x = inputs.make(w, n=probe)
    t = time.perf_counter()
    cref.forward(f(x["q"]), f(x["k"]), f(x["v"]), g)
    rate = w.B * w.H * probe / (time.perf_counter() - t)
    n_s = int(min(w.n, max(64, rate * target_s / (w.B * w.H))))
    reps = max(1, int(round(target_s / (w.B * w.H * n_s / rate))))
    x = inputs.make(w, n=n_s)
    q, k, v = f(x["q"]), f(x["k"]), f(x["v"])
    t = time.perf_counter()
    for _ in range(reps):
        cref.forward(q, k, v, g)
    dt = time.perf_counter() - t
    tokens = w.B * w.H * n_s * reps
    desc = (f"float64 C serial recurrence (OpenMP over heads) on the first {n_s} tokens of all "
            f"{w.B * w.H} heads, {reps} pass(es): {tokens} tokens in {dt:.1f} s")
    return tokens / dt, cref.threads(), desc


def run_reference(args, dist: Dist):
    if dist.rank != 0:
        return
    from oracle import cref

    cref.build()
    per_step = []
    budget = min(2.0, 150.0 / max(1, args.warmup + args.steps))  # whole run within a few minutes
    for i in range(args.warmup + args.steps):
        value, cores, desc = oracle_sample(target_s=budget)
        if i >= args.warmup:
            per_step.append(value)
    value = statistics.median(per_step)
    full_tokens = 1 * 16 * 65536  # one step of the workload; each timed step is a sample of it
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * full_tokens / value,
        "ms_per_step_basis": "the sampled rate applied to one whole step (1,048,576 tokens)",
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": CONFIG_NAME, "B": 1, "H": 16, "n": 65536, "d": 64, "dv": 64, "chunk": 128},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------
# our CUDA path
# ---------------------------------------------------------------------------------

def kernel_source_sha():
    """Hash of the forward tcgen05 kernel sources with // comments and blank lines left out, so
    that an edit of comments alone keeps a recorded traffic capture valid."""
    h = hashlib.sha256()
    for rel in ("chunked_scan_mixer_gb300/csrc/fwd_chunk_tc.cu", "chunked_scan_mixer_gb300/csrc/tc_common.cuh",
                "chunked_scan_mixer_gb300/csrc/common.cuh"):
        with open(os.path.join(ROOT, rel)) as f:
            for line in f:
                code = line.split("//", 1)[0].strip()
                if code:
                    h.update(code.encode())
                    h.update(b"\n")
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu capture, if it matches today's source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(kernel)
    if not ent or ent.get("source_sha") != kernel_source_sha():
        return None
    return ent.get("bytes_per_launch")


def _device_ms(fn, steps, warmup, stream_sync):
    """Mean device time of fn() over `steps` calls after `warmup` calls (CUDA events on the
    current stream, synchronised on both sides)."""
    import torch

    for _ in range(warmup):
        fn()
    stream_sync()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        fn()
    t1.record()
    stream_sync()
    return t0.elapsed_time(t1) / steps


def measure_decode(dev, dist: Dist, hbm_gbs: float, steps: int = 50, warmup: int = 5, seqs: int = 256,
                   compact: bool = False, masked: bool = True):
    """Decode row: 256 sequences x 32 heads, d = dv = 128, one single-token step per
    iteration on a resident fp32 state (the state's values do not change the work: it
    starts from N(0, 1e-4) draws instead of a 4096-token prefill).  Inputs of every step
    are drawn before timing (seed 4000 + step); the 1.6 GB state exceeds the L2.
    masked=False: the unmasked output, which reads and writes S, C and m only."""
    import torch

    import chunked_scan_mixer_gb300 as hla
    from chunked_scan_mixer_gb300 import inputs

    w = inputs.WORKLOADS["decode_prefill"]
    N, H, d, dv = seqs, w.H, w.d, w.dv
    sf = hla.state_floats(d, dv, compact=compact)
    gen = torch.Generator(device=dev)
    gen.manual_seed(replica_seed(w.seed, dist.rank))
    state = torch.randn((N, H, sf), generator=gen, device=dev, dtype=torch.float32) * 1e-2
    gamma = inputs.gammas(w).to(dev)
    xs = [inputs.decode_step_inputs(i, N, H, d, dv, w.dtype, device=dev) for i in range(steps)]
    out = torch.empty((N, H, dv), dtype=w.dtype, device=dev)
    it = [0]

    def one():
        q, k, v = xs[it[0] % steps]
        it[0] += 1
        hla.decode_step(state, q, k, v, gamma=gamma, out=out, compact=compact, masked=masked)

    ms = dist.max(_device_ms(one, steps, warmup, torch.cuda.synchronize))
    heads = N * H
    touched = sf if masked else sf - d * dv - d  # the unmasked step leaves G and h alone
    nbytes = 2 * heads * touched * 4 + heads * (2 * d + dv) * 2 + heads * dv * 2
    achieved = nbytes / (ms * 1e-3) / 1e9
    layout = "compact state (S upper block triangle)" if compact else "packed state"
    return {"workload": f"decode step: {N} sequences x H={H}, d=dv={d}, fp32 {layout}, bf16 q/k/v/out, "
                        f"decay {w.gamma[0]}, {'masked' if masked else 'unmasked'}, unnormalised",
            "metric": "decode tokens/s (sequences x heads per second)", "unit": "tokens/s",
            "value": dist.world * heads / (ms * 1e-3), "us_per_step": ms * 1e3, "steps": steps,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                         "frac": achieved / hbm_gbs, "algorithmic_bytes_per_launch": nbytes}}


def measure_decode_mq(dev, dist: Dist, hbm_gbs: float, steps: int = 50, warmup: int = 5, seqs: int = 256,
                      group: int = 4):
    """Multi-query decode row: the decode row's 256 sequences x 32 query heads, d = dv = 128,
    with the keys and values shared by groups of 4 heads (8 key groups): one S per group
    and per-head C, G, m, h, updated in place on a resident state that exceeds the L2."""
    import torch

    import chunked_scan_mixer_gb300 as hla
    from chunked_scan_mixer_gb300 import inputs

    w = inputs.WORKLOADS["decode_prefill"]
    N, H, d, dv = seqs, w.H, w.d, w.dv
    Hk = H // group
    hsf = hla.mq_head_state_floats(d, dv)
    gen = torch.Generator(device=dev)
    gen.manual_seed(replica_seed(w.seed, dist.rank))
    key_state = torch.randn((N, Hk, d * d), generator=gen, device=dev, dtype=torch.float32) * 1e-2
    head_state = torch.randn((N, H, hsf), generator=gen, device=dev, dtype=torch.float32) * 1e-2
    gamma = torch.full((Hk,), w.gamma[0], dtype=torch.float32, device=dev)
    xs = []
    for i in range(steps):
        q, _, _ = inputs.decode_step_inputs(i, N, H, d, dv, w.dtype, device=dev)
        _, k, v = inputs.decode_step_inputs(10000 + i, N, Hk, d, dv, w.dtype, device=dev)
        xs.append((q, k, v))
    out = torch.empty((N, H, dv), dtype=w.dtype, device=dev)
    it = [0]

    def one():
        q, k, v = xs[it[0] % steps]
        it[0] += 1
        hla.decode_step_mq(key_state, head_state, q, k, v, gamma=gamma, out=out)

    ms = dist.max(_device_ms(one, steps, warmup, torch.cuda.synchronize))
    heads = N * H
    nbytes = 2 * (N * Hk * d * d + heads * hsf) * 4 + heads * d * 2 + N * Hk * (d + dv) * 2 + heads * dv * 2
    achieved = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"multi-query decode step: {N} sequences x H={H} query heads in {Hk} key groups, d=dv={d}, "
                        f"fp32 state (S per group), bf16 q/k/v/out, decay {w.gamma[0]}, masked, unnormalised",
            "metric": "decode tokens/s (sequences x query heads per second)", "unit": "tokens/s",
            "value": dist.world * heads / (ms * 1e-3), "us_per_step": ms * 1e3, "steps": steps,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                         "frac": achieved / hbm_gbs, "algorithmic_bytes_per_launch": nbytes}}


def measure_train(dev, dist: Dist, bf16_tflops: float, hbm_gbs: float, steps: int = 10, warmup: int = 3,
                  d: int | None = None):
    """Training row: B=4 H=16 n=8192 d=dv=128 bf16, decay 0.995, unnormalised, chunk 128 (the
    tcgen05 first-order scan passes); one step = forward (keeping p and the carries for the
    backward) + backward (dq, dk, dv) through the public calls, inputs resident.  d overrides
    the head width (the train_d64 row: d = dv = 64, same batch and length)."""
    import dataclasses

    import torch

    import chunked_scan_mixer_gb300 as hla
    from chunked_scan_mixer_gb300 import inputs

    w = inputs.WORKLOADS["train"]
    if d is not None:
        w = dataclasses.replace(w, d=d, dv=d)
    x = inputs.make(w, device=dev, seed=replica_seed(w.seed, dist.rank))
    q, k, v, do = x["q"], x["k"], x["v"], x["dout"]
    gamma = x["gamma"].to(dev)
    out = torch.empty_like(v)
    gq, gk, gv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def one():
        _, saved = hla.forward(q, k, v, gamma=gamma, chunk=w.chunk, out=out, save_for_backward=True)
        hla.backward(q, k, v, do, gamma=gamma, chunk=w.chunk, dq=gq, dk=gk, dv=gv, saved=saved)

    ms = dist.max(_device_ms(one, steps, warmup, torch.cuda.synchronize))
    tokens = w.B * w.H * w.n
    flops = 3 * tokens * (368640 if w.d == 128 else 98304)  # forward F(64) + backward 2 F(64)
    nbytes = tokens * ((2 * w.d + w.dv) * 2 + w.dv * 2)  # forward
    nbytes += tokens * ((2 * w.d + 2 * w.dv) * 2 + (2 * w.d + w.dv) * 2)  # backward reads, writes
    achieved = flops / (ms * 1e-3) / 1e12
    return {"workload": f"training step (forward + backward): B={w.B} H={w.H} n={w.n} d=dv={w.d} bf16, "
                        f"decay {w.gamma[0]}, unnormalised, chunk {w.chunk}",
            "metric": "training tokens/s (forward + backward)", "unit": "tokens/s",
            "value": dist.world * tokens / (ms * 1e-3), "ms_per_step": ms, "steps": steps,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": bf16_tflops, "unit": "TFLOP/s",
                         "frac": achieved / bf16_tflops, "flops_per_step": flops,
                         "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / hbm_gbs}}


def measure_ahla(dev, dist: Dist, hbm_gbs: float, bf16_tflops: float, steps: int = 50, warmup: int = 5,
                 n: int | None = None):
    """AHLA row: the asymmetric operator on the long-context shapes (B=1 H=16 n=65536
    d=dv=64 bf16, decay linspace(0.99, 0.9999), unnormalised, chunk 128); 1,048,576
    tokens per step; inputs + output exceed the L2."""
    import dataclasses

    import torch

    import chunked_scan_mixer_gb300 as hla
    from chunked_scan_mixer_gb300 import inputs

    w = inputs.WORKLOADS["long"]  # chunk 128: the tcgen05 kernel
    if n is not None:
        w = dataclasses.replace(w, n=n)
    x = inputs.make(w, device=dev, seed=replica_seed(w.seed, dist.rank))
    q, k, v = x["q"], x["k"], x["v"]
    gamma = x["gamma"].to(dev)
    out = torch.empty_like(v)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]

    def one():
        hla.ahla_forward(q, k, v, gamma=gamma, chunk=w.chunk, out=out)

    ms = dist.max(_device_ms(one, steps, warmup, torch.cuda.synchronize))
    hla.ahla_forward(q, k, v, gamma=gamma, chunk=w.chunk, out=out, phase_events=ev)
    torch.cuda.synchronize()
    out_ms = ev[3].elapsed_time(ev[4])
    tokens = w.B * w.H * w.n
    nbytes = tokens * (2 * w.d + 2 * w.dv) * 2
    # chunk products at width W, full (unmasked) counts per token:
    # Q K^T 2 W d, A~ V and A~ Inner 4 W dv, Q P0, Q E0, K~^T V, K~^T Inner 8 d dv
    flops = tokens * (2 * w.chunk * w.d + 4 * w.chunk * w.dv + 8 * w.d * w.dv)
    achieved = nbytes / (out_ms * 1e-3) / 1e9
    return {"workload": f"AHLA forward: B={w.B} H={w.H} n={w.n} d=dv={w.d} bf16, decay linspace(0.99,0.9999), "
                        f"unnormalised, chunk {w.chunk}",
            "metric": "AHLA fwd tokens/s", "unit": "tokens/s", "value": dist.world * tokens / (ms * 1e-3),
            "ms_per_step": ms, "steps": steps, "output_pass_ms": out_ms,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                         "frac": achieved / hbm_gbs, "kernel": "output_pass", "algorithmic_bytes_per_launch": nbytes,
                         "step_tensor_frac": flops / (ms * 1e-3) / 1e12 / bf16_tflops}}


def measure_prefill_d128(dev, dist: Dist, hbm_gbs: float, steps: int = 3, warmup: int = 1, n: int | None = None):
    """Decode-workload prefill row: the 4096-token prefill that starts the streaming decode
    (B=256 sequences x H=32, d=dv=128 bf16, decay 0.999, masked, unnormalised) with the state
    after the last token, at chunk 128 on the first-order scans (33.5M tokens a call); the same
    call on the mma.sync chunk kernels beside it (HLA2_KERNEL=mma).  HBM roofline of the whole
    call over q, k, v read, out and the state written."""
    import dataclasses
    import os

    import torch

    import chunked_scan_mixer_gb300 as hla
    from chunked_scan_mixer_gb300 import inputs

    w = inputs.WORKLOADS["decode_prefill"]
    if n is not None:
        w = dataclasses.replace(w, n=n)
    x = inputs.make(w, device=dev, seed=replica_seed(w.seed, dist.rank))
    q, k, v = x["q"], x["k"], x["v"]
    gamma = x["gamma"].to(dev)
    out = torch.empty_like(v)

    def one():
        hla.forward(q, k, v, gamma=gamma, chunk=128, out=out, return_final_state=True)

    ms = dist.max(_device_ms(one, steps, warmup, torch.cuda.synchronize))
    old = os.environ.get("HLA2_KERNEL")
    os.environ["HLA2_KERNEL"] = "mma"
    try:
        legacy_ms = dist.max(_device_ms(one, max(1, steps - 1), 1, torch.cuda.synchronize))
    finally:
        if old is None:
            os.environ.pop("HLA2_KERNEL", None)
        else:
            os.environ["HLA2_KERNEL"] = old
    tokens = w.B * w.H * w.n
    nbytes = tokens * (2 * w.d + 2 * w.dv) * 2 + w.B * w.H * hla.state_floats(w.d, w.dv) * 4
    achieved = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"decode-workload prefill with the final state: B={w.B} H={w.H} n={w.n} d=dv={w.d} bf16, "
                        f"decay {w.gamma[0]}, unnormalised, chunk 128",
            "metric": "prefill tokens/s", "unit": "tokens/s", "value": dist.world * tokens / (ms * 1e-3),
            "ms_per_step": ms, "steps": steps, "legacy_mma_ms": legacy_ms,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                         "frac": achieved / hbm_gbs, "kernel": "whole call", "algorithmic_bytes_per_step": nbytes}}


def measure_normed(dev, dist: Dist, hbm_gbs: float, steps: int = 200, warmup: int = 10, n: int | None = None):
    """Ratio-normalised rows: the normalised workload (B=2 H=8 n=2048 d=dv=64 bf16, softplus
    q and k, unit-variance v, decay linspace(0.95, 0.999), eps 1e-6) at chunk 128, where the
    tcgen05 stored-p kernels run (the output pass forms the denominator in its epilogue), and
    at its stated chunk 64 on the mma.sync kernels; then the same recipe at the long-context
    length (B=1 H=16 n=65536) at chunk 128.  HBM roofline of the whole call over q, k, v read
    and out written."""
    import dataclasses

    import torch

    import chunked_scan_mixer_gb300 as hla
    from chunked_scan_mixer_gb300 import inputs

    w = inputs.WORKLOADS["normed"]
    rows = {}
    for name, ww, chunk in (("normed_chunk128", w, 128), ("normed_chunk64", w, 64),
                            ("normed_long", dataclasses.replace(w, B=1, H=16, n=n or 65536), 128)):
        x = inputs.make(ww, device=dev, seed=replica_seed(ww.seed, dist.rank))
        q, k, v = x["q"], x["k"], x["v"]
        gamma = x["gamma"].to(dev)
        out = torch.empty_like(v)

        def one():
            hla.forward(q, k, v, gamma=gamma, chunk=chunk, normalize=True, eps=ww.eps, out=out)

        long = name == "normed_long"
        ms = dist.max(_device_ms(one, max(1, steps // 4) if long else steps, warmup, torch.cuda.synchronize))
        tokens = ww.B * ww.H * ww.n
        nbytes = tokens * (2 * ww.d + 2 * ww.dv) * 2
        achieved = nbytes / (ms * 1e-3) / 1e9
        rows[name] = {"workload": f"normalised forward: B={ww.B} H={ww.H} n={ww.n} d=dv={ww.d} bf16, softplus q/k, "
                                  f"decay linspace{tuple(ww.gamma)}, eps {ww.eps}, chunk {chunk}",
                      "metric": "normalised fwd tokens/s", "unit": "tokens/s",
                      "value": dist.world * tokens / (ms * 1e-3), "ms_per_step": ms,
                      "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                                   "frac": achieved / hbm_gbs, "kernel": "whole call",
                                   "algorithmic_bytes_per_step": nbytes}}
    return rows


def measure_normed_backward(dev, dist: Dist, hbm_gbs: float, steps: int = 50, warmup: int = 5,
                            n: int | None = None):
    """Ratio-normalised reverse-mode rows: dq, dk, dv of o / (den + eps) on the normalised
    workload (B=2 H=8 n=2048 d=dv=64 bf16, softplus q and k, decay linspace(0.95, 0.999),
    eps 1e-6, chunk 64), upstream dO ~ N(0, 1), and on the same recipe at B=1 H=16 n=16384.
    The call widens the inputs to float32 and composes float32 passes (two forwards, the
    quotient rule, two backwards).  HBM roofline of the whole call over q, k, v, dO read and
    dq, dk, dv written (bf16)."""
    import dataclasses

    import torch

    import chunked_scan_mixer_gb300 as hla
    from chunked_scan_mixer_gb300 import inputs

    w = dataclasses.replace(inputs.WORKLOADS["normed"], with_dout=True)
    rows = {}
    for name, ww in (("normed_backward", w),
                     ("normed_backward_long", dataclasses.replace(w, B=1, H=16, n=n or 16384))):
        x = inputs.make(ww, device=dev, seed=replica_seed(ww.seed, dist.rank))
        q, k, v, do = x["q"], x["k"], x["v"], x["dout"]
        gamma = x["gamma"].to(dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

        def one():
            hla.backward(q, k, v, do, gamma=gamma, chunk=ww.chunk, normalize=True, eps=ww.eps, dq=dq, dk=dk, dv=dv)

        long = name == "normed_backward_long"
        ms = dist.max(_device_ms(one, max(1, steps // 5) if long else steps, warmup, torch.cuda.synchronize))
        tokens = ww.B * ww.H * ww.n
        nbytes = tokens * (4 * ww.d + 3 * ww.dv) * 2
        achieved = nbytes / (ms * 1e-3) / 1e9
        rows[name] = {"workload": f"normalised backward: B={ww.B} H={ww.H} n={ww.n} d=dv={ww.d} bf16, softplus q/k, "
                                  f"decay linspace{tuple(ww.gamma)}, eps {ww.eps}, chunk {ww.chunk}, float32 passes",
                      "metric": "normalised bwd tokens/s", "unit": "tokens/s",
                      "value": dist.world * tokens / (ms * 1e-3), "ms_per_step": ms,
                      "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                                   "frac": achieved / hbm_gbs, "kernel": "whole call",
                                   "algorithmic_bytes_per_step": nbytes}}
    return rows


def measure_ahla_backward(dev, dist: Dist, hbm_gbs: float, steps: int = 20, warmup: int = 3, n: int | None = None):
    """AHLA reverse-mode row: dq, dk, dv of the unnormalised AHLA output on the long-context
    shapes (B=1 H=16 n=65536 d=dv=64 bf16, decay linspace(0.99, 0.9999), chunk 128: the tcgen05
    first-order scans), upstream dO ~ N(0, 1); HBM roofline of the whole call over its
    algorithmic bytes (q, k, v, dO read, dq, dk, dv written)."""
    import dataclasses

    import torch

    import chunked_scan_mixer_gb300 as hla
    from chunked_scan_mixer_gb300 import inputs

    w = dataclasses.replace(inputs.WORKLOADS["long"], with_dout=True)
    if n is not None:
        w = dataclasses.replace(w, n=n)
    x = inputs.make(w, device=dev, seed=replica_seed(w.seed, dist.rank))
    q, k, v, do = x["q"], x["k"], x["v"], x["dout"]
    gamma = x["gamma"].to(dev)

    def one():
        hla.ahla_backward(q, k, v, do, gamma=gamma, chunk=w.chunk)

    ms = dist.max(_device_ms(one, steps, warmup, torch.cuda.synchronize))
    tokens = w.B * w.H * w.n
    nbytes = tokens * (4 * w.d + 3 * w.dv) * 2
    achieved = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"AHLA backward: B={w.B} H={w.H} n={w.n} d=dv={w.d} bf16, decay linspace(0.99,0.9999), "
                        f"unnormalised, chunk {w.chunk}",
            "metric": "AHLA bwd tokens/s", "unit": "tokens/s", "value": dist.world * tokens / (ms * 1e-3),
            "ms_per_step": ms, "steps": steps,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                         "frac": achieved / hbm_gbs, "kernel": "whole call", "algorithmic_bytes_per_step": nbytes}}


def measure_unmasked(dev, dist: Dist, hbm_gbs: float, steps: int = 50, warmup: int = 5, n: int | None = None,
                     chunk: int = 128):
    """Unmasked-output row: q^T S C on the long-context shapes (B=1 H=16 n=65536 d=dv=64
    bf16, decay linspace(0.99, 0.9999), unnormalised; chunk 128: the tcgen05 kernels);
    1,048,576 tokens per step; inputs + output exceed the L2."""
    import dataclasses

    import torch

    import chunked_scan_mixer_gb300 as hla
    from chunked_scan_mixer_gb300 import inputs

    w = dataclasses.replace(inputs.WORKLOADS["long"], chunk=chunk)
    if n is not None:
        w = dataclasses.replace(w, n=n)
    x = inputs.make(w, device=dev, seed=replica_seed(w.seed, dist.rank))
    q, k, v = x["q"], x["k"], x["v"]
    gamma = x["gamma"].to(dev)
    out = torch.empty_like(v)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]

    def one():
        hla.forward(q, k, v, gamma=gamma, chunk=w.chunk, out=out, masked=False)

    ms = dist.max(_device_ms(one, steps, warmup, torch.cuda.synchronize))
    hla.forward(q, k, v, gamma=gamma, chunk=w.chunk, out=out, masked=False, phase_events=ev)
    torch.cuda.synchronize()
    sum_ms, out_ms = ev[1].elapsed_time(ev[2]), ev[3].elapsed_time(ev[4])
    tokens = w.B * w.H * w.n
    nbytes = tokens * (2 * w.d + 2 * w.dv) * 2
    nseg = hla.forward_plan(w.B, w.H, w.n, w.d, w.dv, w.chunk)[0]
    # stored-p path (d = dv = 64, chunk 128, more than one segment): the summary pass covers
    # every token and writes p, 512 B per token like the output pass; the larger pass is reported
    stored_p = w.d == 64 and w.dv == 64 and w.chunk == 128 and nseg > 1
    if stored_p and sum_ms > out_ms:
        kname, kms = "segment_summaries", sum_ms
    else:
        kname, kms = "output_pass", out_ms
    achieved = nbytes / (kms * 1e-3) / 1e9
    return {"workload": f"unmasked HLA-2 forward (q^T S C): B={w.B} H={w.H} n={w.n} d=dv={w.d} bf16, "
                        f"decay linspace(0.99,0.9999), unnormalised, chunk {w.chunk}",
            "metric": "unmasked fwd tokens/s", "unit": "tokens/s", "value": dist.world * tokens / (ms * 1e-3),
            "ms_per_step": ms, "steps": steps, "output_pass_ms": out_ms, "summary_pass_ms": sum_ms,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                         "frac": achieved / hbm_gbs, "kernel": kname, "algorithmic_bytes_per_launch": nbytes}}


def measure_prefill(dev, dist: Dist, hbm_gbs: float, steps: int = 50, warmup: int = 5, n: int | None = None):
    """Prefill row: the long-context forward (B=1 H=16 n=65536 d=dv=64 bf16, decay
    linspace(0.99, 0.9999), chunk 128) that also returns the state after the last token (the
    decode step's starting state); 1,048,576 tokens per step."""
    import dataclasses

    import torch

    import chunked_scan_mixer_gb300 as hla
    from chunked_scan_mixer_gb300 import inputs

    w = inputs.WORKLOADS["long"]
    if n is not None:
        w = dataclasses.replace(w, n=n)
    x = inputs.make(w, device=dev, seed=replica_seed(w.seed, dist.rank))
    q, k, v = x["q"], x["k"], x["v"]
    gamma = x["gamma"].to(dev)
    out = torch.empty_like(v)

    def one():
        hla.forward(q, k, v, gamma=gamma, chunk=w.chunk, out=out, return_final_state=True)

    ms = dist.max(_device_ms(one, steps, warmup, torch.cuda.synchronize))
    tokens = w.B * w.H * w.n
    # q, k, v read, out written, plus the state written (about 0.3 % of the bytes)
    nbytes = tokens * (2 * w.d + 2 * w.dv) * 2 + w.B * w.H * hla.state_floats(w.d, w.dv) * 4
    achieved = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"prefill: long-context masked forward with the final state, B={w.B} H={w.H} n={w.n} "
                        f"d=dv={w.d} bf16, decay linspace(0.99,0.9999), unnormalised, chunk {w.chunk}",
            "metric": "prefill tokens/s", "unit": "tokens/s", "value": dist.world * tokens / (ms * 1e-3),
            "ms_per_step": ms, "steps": steps,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                         "frac": achieved / hbm_gbs, "kernel": "whole step", "algorithmic_bytes_per_step": nbytes}}


def measure_hla3(dev, dist: Dist, hbm_gbs: float, steps: int = 30, warmup: int = 5, n: int | None = None):
    """Third-order row: the masked third-order output at gamma = 1 on the long-context shapes
    (B=1 H=16 n=65536 d=dv=64 bf16, unnormalised, chunk 128): the first-order pass on the AHLA
    tcgen05 kernel in its first-order mode, then the second-order tcgen05 forward."""
    import dataclasses

    import torch

    import chunked_scan_mixer_gb300 as hla
    from chunked_scan_mixer_gb300 import inputs

    w = inputs.WORKLOADS["long"]
    if n is not None:
        w = dataclasses.replace(w, n=n)
    x = inputs.make(w, device=dev, seed=replica_seed(w.seed, dist.rank))
    q, k, v = x["q"], x["k"], x["v"]
    out = torch.empty_like(v)

    def one():
        hla.hla3_forward(q, k, v, chunk=w.chunk, out=out)

    ms = dist.max(_device_ms(one, steps, warmup, torch.cuda.synchronize))
    tokens = w.B * w.H * w.n
    # two passes over q, k and a value tensor, each reading 3 x 128 B and writing 128 B a token
    nbytes = 2 * tokens * (2 * w.d + 2 * w.dv) * 2
    achieved = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"masked third-order HLA forward (gamma = 1): B={w.B} H={w.H} n={w.n} d=dv={w.d} bf16, "
                        f"unnormalised, chunk {w.chunk}",
            "metric": "third-order fwd tokens/s", "unit": "tokens/s", "value": dist.world * tokens / (ms * 1e-3),
            "ms_per_step": ms, "steps": steps,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                         "frac": achieved / hbm_gbs, "algorithmic_bytes_per_step": nbytes}}


def run_only(args, dist: Dist, dev):
    hbm_gbs, bf16_tflops, _ = peaks()
    if args.only in ("decode", "decode_compact", "decode_unmasked"):
        row = measure_decode(dev, dist, hbm_gbs, steps=args.steps, warmup=args.warmup, seqs=args.decode_seqs,
                             compact=args.only == "decode_compact", masked=args.only != "decode_unmasked")
    elif args.only == "hla3":
        row = measure_hla3(dev, dist, hbm_gbs, steps=args.steps, warmup=args.warmup, n=args.n)
    elif args.only == "decode_mq":
        row = measure_decode_mq(dev, dist, hbm_gbs, steps=args.steps, warmup=args.warmup, seqs=args.decode_seqs)
    elif args.only == "prefill":
        row = measure_prefill(dev, dist, hbm_gbs, steps=args.steps, warmup=args.warmup, n=args.n)
    elif args.only == "unmasked":
        row = measure_unmasked(dev, dist, hbm_gbs, steps=args.steps, warmup=args.warmup, n=args.n,
                               chunk=args.chunk or 128)
    elif args.only == "ahla":
        row = measure_ahla(dev, dist, hbm_gbs, bf16_tflops, steps=args.steps, warmup=args.warmup, n=args.n)
    elif args.only == "ahla_backward":
        row = measure_ahla_backward(dev, dist, hbm_gbs, steps=args.steps, warmup=args.warmup, n=args.n)
    elif args.only == "normed":
        row = measure_normed(dev, dist, hbm_gbs, steps=args.steps, warmup=args.warmup, n=args.n)
    elif args.only == "normed_backward":
        row = measure_normed_backward(dev, dist, hbm_gbs, steps=args.steps, warmup=args.warmup, n=args.n)
    elif args.only == "prefill_d128":
        row = measure_prefill_d128(dev, dist, hbm_gbs, steps=args.steps, warmup=args.warmup, n=args.n)
    elif args.only == "train_d64":
        row = measure_train(dev, dist, bf16_tflops, hbm_gbs, steps=args.steps, warmup=args.warmup, d=64)
    else:
        row = measure_train(dev, dist, bf16_tflops, hbm_gbs, steps=args.steps, warmup=args.warmup)
    if dist.rank == 0:
        print(json.dumps({"only": args.only, "n_gpus": dist.world, "secondary": {args.only: row}}), flush=True)


def run_ours(args, dist: Dist):
    import torch

    import chunked_scan_mixer_gb300 as hla
    from chunked_scan_mixer_gb300 import inputs

    torch.cuda.set_device(dist.local)
    dev = torch.device("cuda", dist.local)
    if args.only:
        return run_only(args, dist, dev)
    w = inputs.WORKLOADS[WORKLOAD]
    if args.n is not None:
        import dataclasses
        w = dataclasses.replace(w, n=args.n)
    tokens = w.B * w.H * w.n
    x = inputs.make(w, device=dev, seed=replica_seed(w.seed, dist.rank))
    q, k, v = x["q"], x["k"], x["v"]
    gamma = x["gamma"].to(dev)
    out = torch.empty_like(v)
    nseg, seg_chunks, launches = hla.forward_plan(w.B, w.H, w.n, w.d, w.dv, w.chunk, normalize=w.normalize)

    def step(evs=None):
        hla.forward(q, k, v, gamma=gamma, chunk=w.chunk, out=out, phase_events=evs)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    K = args.steps
    # the per-phase split comes from a separate run: events recorded between the kernels of a
    # step would serialise their programmatic dependent launches
    KP = min(K, 200)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(KP)]
    for e in evs:  # create the CUDA events outside the timed region
        for ev in e:
            ev.record()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dist.local)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    t_start.record()
    for i in range(K):
        step()
    t_end.record()
    torch.cuda.synchronize()
    wall1 = time.time()
    dist.barrier()
    clk = clocks.stop(wall0, wall1)
    ms_total = dist.max(t_start.elapsed_time(t_end))
    ms_per_step = ms_total / K
    value = weak_scaling_value(dist.world, tokens, ms_per_step)

    # per-phase device time (events on the launching stream), in a run of its own
    for i in range(KP):
        step(evs[i])
    torch.cuda.synchronize()
    ph = {name: 0.0 for name in PHASES}
    for e in evs:
        for j, name in enumerate(PHASES):
            ph[name] += e[j].elapsed_time(e[j + 1])
    ph = {name: t / KP for name, t in ph.items()}

    hbm_gbs, bf16_tflops, peak_kind = peaks()
    # algorithmic bytes per launch: q, k, v read (bf16) and out written (bf16) for the
    # tokens the launch processes
    out_bytes = tokens * (2 * w.d + w.dv) * 2 + tokens * w.dv * 2
    io_mb = tokens * (2 * w.d + 2 * w.dv) * 2 / 1e6
    summary_tokens = w.B * w.H * min(w.n, (nseg - 1) * seg_chunks * w.chunk)
    summ_bytes = summary_tokens * (2 * w.d + w.dv) * 2
    # The masked bf16 forward at d = dv = 64, chunk 128 with more than one segment takes the
    # stored-p path: its summary pass covers every token and also writes p = S q (d bf16 per
    # token) into out, and its output pass reads q, p, v (no k) and writes out (same bytes).
    stored_p = (w.d == 64 and w.dv == 64 and w.chunk == 128 and not w.normalize and nseg > 1
                and os.environ.get("HLA2_KERNEL") != "mma")
    if stored_p:
        summary_tokens = tokens
        summ_bytes = tokens * ((2 * w.d + w.dv) * 2 + w.d * 2)
    if ph["output_pass"] >= ph["segment_summaries"]:
        kname, kbytes, kms = "output_pass", out_bytes, ph["output_pass"]
    else:
        kname, kbytes, kms = "segment_summaries", summ_bytes, ph["segment_summaries"]
    achieved = kbytes / (kms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                "frac": achieved / hbm_gbs, "traffic": recorded_traffic(kname),
                "kernel": kname, "peak_source": peak_kind,
                "algorithmic_bytes_per_launch": kbytes, "ms_per_launch": kms}
    # whole-step fractions against both roofs (flops of the method at chunk 64)
    flops_per_token = 98304
    step_bytes = out_bytes
    whole = {"hbm_frac": step_bytes / (ms_per_step * 1e-3) / 1e9 / hbm_gbs,
             "tensor_frac": tokens * flops_per_token / (ms_per_step * 1e-3) / 1e12 / bf16_tflops,
             "roofline_time_us": max(step_bytes / (hbm_gbs * 1e9), tokens * flops_per_token / (bf16_tflops * 1e12)) * 1e6}

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        qh, kh, vh = (t.to("cpu").pin_memory() for t in (q, k, v))
        oh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        Ke = max(3, min(K, 50))
        for _ in range(2):
            hla.forward(qh, kh, vh, gamma=gamma, chunk=w.chunk, out=oh)
        torch.cuda.synchronize()
        dist.barrier()
        t0 = time.perf_counter()
        for _ in range(Ke):
            hla.forward(qh, kh, vh, gamma=gamma, chunk=w.chunk, out=oh)
        torch.cuda.synchronize()
        dt = dist.max(time.perf_counter() - t0) / Ke
        e2e = {"value": weak_scaling_value(dist.world, tokens, dt * 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": 3 * q.numel() * q.element_size(),
               "d2h_bytes_per_step": out.numel() * out.element_size(), "steps": Ke}

    secondary = None
    if not args.no_secondary and args.n is None:
        secondary = {"decode": measure_decode(dev, dist, hbm_gbs),
                     "decode_compact": measure_decode(dev, dist, hbm_gbs, compact=True),
                     "decode_unmasked": measure_decode(dev, dist, hbm_gbs, masked=False),
                     "decode_mq": measure_decode_mq(dev, dist, hbm_gbs),
                     "train": measure_train(dev, dist, bf16_tflops, hbm_gbs),
                     "train_d64": measure_train(dev, dist, bf16_tflops, hbm_gbs, d=64),
                     "ahla": measure_ahla(dev, dist, hbm_gbs, bf16_tflops),
                     "ahla_backward": measure_ahla_backward(dev, dist, hbm_gbs),
                     "unmasked": measure_unmasked(dev, dist, hbm_gbs),
                     "hla3": measure_hla3(dev, dist, hbm_gbs),
                     "prefill": measure_prefill(dev, dist, hbm_gbs)}
        secondary.update(measure_normed(dev, dist, hbm_gbs))
        secondary.update(measure_normed_backward(dev, dist, hbm_gbs))
        secondary["prefill_d128"] = measure_prefill_d128(dev, dist, hbm_gbs)

    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        val, cores, desc = oracle_sample(target_s=15.0)
        cpu = {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc}

    if dist.rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": dist.world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": CONFIG_NAME, "B": w.B, "H": w.H, "n": w.n, "d": w.d, "dv": w.dv,
                       "chunk": w.chunk, "segments_per_head": nseg, "chunks_per_segment": seg_chunks,
                       "l2": f"inputs + output ({io_mb:.1f} MB) exceed the 129 MB L2; no flush"},
            "roofline": roofline, "whole_step": whole, "phases_ms": ph, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches * K, "clocks": clk, "secondary": secondary,
        }
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    dist = Dist("gloo" if args.impl == "reference" else "nccl")
    try:
        if args.impl == "reference":
            run_reference(args, dist)
        else:
            run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
