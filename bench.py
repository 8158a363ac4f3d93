"""Benchmark: causal prefill tokens/s (+ % of the HBM roofline) and the decode
step (us/token, state GB/s) of the kernelized linear attention library.

One JSON line on stdout (rank 0).  Headline workload: the long causal
prefill B=8, H=16, T=8192, Dk=Dv=128, bf16 q/k/v, fp32 state, relu+eps,
normalized, eps 1e-6 -- the largest single-GPU configuration measured.  The
line also carries every other prefill workload (``workloads``: the 2k
prefill, its masked form, the unnormalized and non-causal 8k passes, the
ONNX linear and gated GQA workloads, the per-key-dimension decay, the
delta rule, the backward pass) and the streaming-decode workload (B=256,
H=32, D=128, state from a 4096-token prefill, 1024 single-token steps) as
the ``decode`` object.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Multi-GPU (torchrun): every rank runs its own copy of the workload on its own
GPU (independent sequences, no collective on the data path): weak scaling.
``--impl reference`` times the CPU oracle (the only reference there is) on
the host cores instead, on a sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import linattn_inputs as inputs  # noqa: E402

METRIC = "causal prefill tokens/s and % roofline; decode step µs/token and state-GB/s"
L2_BYTES = 129 * 1024 * 1024


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks sampled during the timed region

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.25)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed plumbing (weak scaling: independent replicas)

def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# workload definitions

HEADLINE = inputs.LONG_8K


def rotate_sets(w):
    """Input sets the timed prefill calls rotate over: more than 3x L2 of
    inputs in flight, so that every call reads cold data from HBM."""
    return max(2, -(-3 * L2_BYTES // prefill_alg_bytes(w)))


def config_for(w, world=1):
    """The ``config`` object of the JSON line; both arms print the same one."""
    n = rotate_sets(w)
    return {"workload": w.name, "B": w.B, "T": w.T, "H": w.q_heads, "H_kv": w.kv_heads, "Dk": w.Dk, "Dv": w.Dv,
            "feature_map": w.feature_map, "use_normalizer": w.use_normalizer, "eps": w.eps, "rule": w.rule,
            "io_dtype": "bf16" if w.dtype == torch.bfloat16 else "fp32", "state_dtype": "fp32",
            "parallelism": f"{world} independent replica(s)",
            "l2": f"GPU arm: inputs rotate over {n} sets ({n * prefill_alg_bytes(w) / 1e6:.0f} MB > L2)"}


def prefill_kwargs(w):
    return dict(q_heads=w.q_heads, kv_heads=w.kv_heads, feature_map=w.feature_map,
                use_normalizer=w.use_normalizer, epsilon=w.eps, scale=w.scale, update_rule=w.rule)


def prefill_alg_bytes(w, T=None):
    T = w.T if T is None else T
    esz = 2 if w.dtype == torch.bfloat16 else 4
    qy = w.B * T * w.q_heads * (w.Dk + w.Dv) * esz
    kv = w.B * T * w.kv_heads * (w.Dk + w.Dv) * esz
    dec = w.B * T * w.kv_heads * (w.Dk if w.decay_per_dim else 1) * esz if w.rule in ("gated", "gated_delta") else 0
    dec += w.B * T * w.kv_heads * esz if w.rule in ("delta", "gated_delta") else 0  # beta
    msk = w.B * T if w.mask else 0  # one validity byte per (batch, step)
    return qy + kv + dec + msk


def decode_alg_bytes(w):
    esz = 2
    state = w.B * w.kv_heads * (w.Dk * w.Dv + (w.Dk if w.use_normalizer else 0)) * 4
    tok = w.B * (w.q_heads * (w.Dk + w.Dv) + w.kv_heads * (w.Dk + w.Dv)) * esz
    return 2 * state + tok, 2 * state


# ---------------------------------------------------------------------------
# GPU arm

def time_prefill(la, w, steps, warmup, stream):
    """Device time of `steps` causal prefill calls on rotating input sets."""
    nsets = rotate_sets(w)
    sets = []
    for s in range(nsets):
        q, k, v, d = inputs.make_qkv(w, device="cuda", seed=w.seed + s)
        y = torch.empty(w.B, w.T, w.q_heads, w.Dv, dtype=w.dtype, device="cuda")
        sets.append((q, k, v, d, y))
    kw = prefill_kwargs(w)
    ws = torch.empty(max(1, la.la_workspace_bytes(la.make_params(
        batch=w.B, seq_len=w.T, q_heads=w.q_heads, kv_heads=w.kv_heads, key_dim=w.Dk, value_dim=w.Dv,
        io_dtype=w.dtype, feature_map=w.feature_map, use_normalizer=w.use_normalizer, epsilon=w.eps,
        scale=w.scale, update_rule=w.rule), True)), dtype=torch.uint8, device="cuda")

    def step(i):
        q, k, v, d, y = sets[i % nsets]
        la.la_forward_causal(q, k, v, decay=d, out=y, workspace=ws, stream=stream, **kw)

    with torch.cuda.stream(stream):
        for i in range(warmup):
            step(i)
    torch.cuda.synchronize()
    n0 = la.la_launch_count()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for i in range(steps):
            step(warmup + i)
    ev1.record(stream)
    torch.cuda.synchronize()
    launches = la.la_launch_count() - n0
    ms = ev0.elapsed_time(ev1) / steps
    return ms, launches, nsets, sets


def time_prefill_e2e(la, w, steps, warmup, stream):
    """Same call with host-resident inputs, as a serving loop would run it: every
    step copies its q, k, v from pinned host memory to the device, runs the
    call, and copies y back to pinned host memory, all inside the timed region.
    Steps are pipelined over three streams (host->device copies, compute,
    device->host copies) with two device buffer sets, so the copies of one
    step overlap the compute of its neighbours."""
    q, k, v, d = inputs.make_qkv(w, device="cpu", seed=w.seed)
    hq, hk, hv = (t.pin_memory() for t in (q, k, v))
    hd = d.pin_memory() if d is not None else None
    hys = [torch.empty(w.B, w.T, w.q_heads, w.Dv, dtype=w.dtype).pin_memory() for _ in range(2)]
    bufs = []
    p = la.make_params(batch=w.B, seq_len=w.T, q_heads=w.q_heads, kv_heads=w.kv_heads, key_dim=w.Dk,
                       value_dim=w.Dv, io_dtype=w.dtype, feature_map=w.feature_map,
                       use_normalizer=w.use_normalizer, epsilon=w.eps, scale=w.scale, update_rule=w.rule)
    for _ in range(2):
        bufs.append(dict(q=torch.empty_like(q, device="cuda"), k=torch.empty_like(k, device="cuda"),
                         v=torch.empty_like(v, device="cuda"),
                         d=torch.empty_like(d, device="cuda") if d is not None else None,
                         y=torch.empty(w.B, w.T, w.q_heads, w.Dv, dtype=w.dtype, device="cuda"),
                         ws=torch.empty(max(1, la.la_workspace_bytes(p, True)), dtype=torch.uint8, device="cuda")))
    kw = prefill_kwargs(w)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]
    in_done = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def step(i):
        b = i % 2
        u = bufs[b]
        if used[b]:
            s_in.wait_event(comp_done[b])      # inputs of step i-2 consumed
        with torch.cuda.stream(s_in):
            u["q"].copy_(hq, non_blocking=True)
            u["k"].copy_(hk, non_blocking=True)
            u["v"].copy_(hv, non_blocking=True)
            if hd is not None:
                u["d"].copy_(hd, non_blocking=True)
        in_done[b].record(s_in)
        stream.wait_event(in_done[b])
        if used[b]:
            stream.wait_event(out_done[b])     # y of step i-2 copied out
        with torch.cuda.stream(stream):
            la.la_forward_causal(u["q"], u["k"], u["v"], decay=u["d"], out=u["y"], workspace=u["ws"],
                                 stream=stream, **kw)
        comp_done[b].record(stream)
        s_out.wait_event(comp_done[b])
        with torch.cuda.stream(s_out):
            hys[b].copy_(u["y"], non_blocking=True)
        out_done[b].record(s_out)
        used[b] = True

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(s_in)
    stream.wait_event(ev0)
    s_out.wait_event(ev0)
    for i in range(steps):
        step(warmup + i)
    stream.wait_event(out_done[(warmup + steps - 1) % 2])
    stream.wait_event(out_done[(warmup + steps - 2) % 2])
    ev1.record(stream)
    torch.cuda.synchronize()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv) + ((hd,) if hd is not None else ()))
    return ev0.elapsed_time(ev1) / steps, h2d, hys[0].numel() * hys[0].element_size()


def time_decode(la, w, n_steps, warmup, stream):
    """us per decode step of the streaming-decode workload."""
    kw = prefill_kwargs(w)
    # state from a causal prefill over the workload's prompt length (untimed)
    q, k, v, _ = inputs.make_qkv(w, device="cuda", seed=w.seed)
    _, (S, Z) = la.la_forward_causal(q, k, v, return_state=True, stream=stream, **kw)
    del q, k, v
    g = inputs.generator(1000, "cuda")
    total = warmup + n_steps
    tq = inputs.normal((total, w.B, 1, w.q_heads, w.Dk), g, dtype=w.dtype, device="cuda")
    tk = inputs.normal((total, w.B, 1, w.kv_heads, w.Dk), g, dtype=w.dtype, device="cuda")
    tv = inputs.normal((total, w.B, 1, w.kv_heads, w.Dv), g, dtype=w.dtype, device="cuda")
    y = torch.empty(w.B, 1, w.q_heads, w.Dv, dtype=w.dtype, device="cuda")
    with torch.cuda.stream(stream):
        for i in range(warmup):
            la.la_decode_step(tq[i], tk[i], tv[i], S, Z, out=y, stream=stream, **kw)
    torch.cuda.synchronize()
    n0 = la.la_launch_count()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for i in range(warmup, total):
            la.la_decode_step(tq[i], tk[i], tv[i], S, Z, out=y, stream=stream, **kw)
    ev1.record(stream)
    torch.cuda.synchronize()
    return ev0.elapsed_time(ev1) * 1e3 / n_steps, la.la_launch_count() - n0


def time_workload(la, w, steps, warmup, stream, causal=True):
    """Device time of one call (causal or non-causal) on one of the measured
    workloads, inputs resident in HBM and rotated so that the data a call
    reads exceeds L2 (the larger workloads exceed it on their own)."""
    set_bytes = prefill_alg_bytes(w)
    nsets = max(1, -(-3 * L2_BYTES // set_bytes))
    sets = []
    for s in range(nsets):
        q, k, v, d = inputs.make_qkv(w, device="cuda", seed=w.seed + s)
        y = torch.empty(w.B, w.T, w.q_heads, w.Dv, dtype=w.dtype, device="cuda")
        m = inputs.validity_mask(w.mask, w.B, w.T, w.seed + s, "cuda") if w.mask else None
        bt = inputs.make_beta(w, "cuda", w.seed + s) if w.rule in ("delta", "gated_delta") else None
        sets.append((q, k, v, d, y, m, bt))
    kw = prefill_kwargs(w)
    if not causal:
        kw.pop("update_rule")
    p = la.make_params(batch=w.B, seq_len=w.T, q_heads=w.q_heads, kv_heads=w.kv_heads, key_dim=w.Dk,
                       value_dim=w.Dv, io_dtype=w.dtype, feature_map=w.feature_map,
                       use_normalizer=w.use_normalizer, epsilon=w.eps, scale=w.scale, update_rule=w.rule)
    need = la.la_delta_workspace_bytes(p) if w.rule in ("delta", "gated_delta") else la.la_workspace_bytes(p, causal)
    ws = torch.empty(max(1, need), dtype=torch.uint8, device="cuda")

    def step(i):
        q, k, v, d, y, m, bt = sets[i % nsets]
        if causal:
            la.la_forward_causal(q, k, v, decay=d, out=y, workspace=ws, mask=m, beta=bt, stream=stream, **kw)
        else:
            la.la_forward_noncausal(q, k, v, out=y, workspace=ws, mask=m, stream=stream, **kw)

    with torch.cuda.stream(stream):
        for i in range(warmup):
            step(i)
    torch.cuda.synchronize()
    n0 = la.la_launch_count()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for i in range(steps):
            step(warmup + i)
    ev1.record(stream)
    torch.cuda.synchronize()
    launches = la.la_launch_count() - n0
    del sets, ws
    torch.cuda.empty_cache()
    return ev0.elapsed_time(ev1) / steps, launches / steps


def time_backward(la, w, steps, warmup, stream):
    """Device time of la_backward_causal on a workload (linear rule): q, k, v
    and dy resident in HBM, fp32 gradients.  Algorithmic bytes: q, k, v, dy
    read once, dq, dk, dv written once."""
    q, k, v, _ = inputs.make_qkv(w, device="cuda", seed=w.seed)
    dy = inputs.normal((w.B, w.T, w.q_heads, w.Dv), inputs.generator(w.seed + 1, "cuda"), 1.0, dtype=w.dtype,
                       device="cuda")
    kw = prefill_kwargs(w)
    kw.pop("update_rule")
    p = la.make_params(batch=w.B, seq_len=w.T, q_heads=w.q_heads, kv_heads=w.kv_heads, key_dim=w.Dk, value_dim=w.Dv,
                       io_dtype=w.dtype, feature_map=w.feature_map, use_normalizer=w.use_normalizer,
                       epsilon=w.eps, scale=w.scale)
    ws = torch.empty(max(1, la.la_backward_workspace_bytes(p)), dtype=torch.uint8, device="cuda")
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            la.la_backward_causal(q, k, v, dy, workspace=ws, stream=stream, **kw)
    torch.cuda.synchronize()
    n0 = la.la_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(steps):
            la.la_backward_causal(q, k, v, dy, workspace=ws, stream=stream, **kw)
    ev1.record(stream)
    torch.cuda.synchronize()
    launches = (la.la_launch_count() - n0) / steps
    esz = 2 if w.dtype == torch.bfloat16 else 4
    alg = (w.B * w.T * (w.q_heads * (w.Dk + w.Dv) + w.kv_heads * (w.Dk + w.Dv)) * esz
           + w.B * w.T * (w.q_heads * w.Dk + w.kv_heads * (w.Dk + w.Dv)) * 4)
    return ev0.elapsed_time(ev1) / steps, launches, alg


def workload_sweep(la, steps, warmup, stream, hbm_gbs):
    """Every prefill workload of the library (causal and non-causal), each
    with its HBM roofline fraction.  Algorithmic bytes: q, k, v (+ decay)
    read once and y written once (plus one mask byte per step for the
    masked workload, whose tokens/s counts padded steps too)."""
    out = []
    cases = [(inputs.PREFILL_2K, True), (inputs.PREFILL_2K_RIGHTPAD, True), (inputs.LONG_8K, True),
             (inputs.LONG_8K_UNNORM, True), (inputs.LONG_8K, False), (inputs.LONG_8K_UNNORM, False),
             (inputs.ONNX_LINEAR, True), (inputs.ONNX_GATED, True), (inputs.GATED_PERDIM, True),
             (inputs.GATED_DELTA, True)]
    for w, causal in cases:
        ms, lpc = time_workload(la, w, steps, warmup, stream, causal)
        alg = prefill_alg_bytes(w)
        gbs = alg / (ms * 1e-3) / 1e9
        out.append({"workload": w.name, "mode": "causal" if causal else "noncausal", "ms": ms,
                    "tokens_per_s": w.B * w.T / (ms * 1e-3), "alg_bytes": alg, "achieved_GBps": gbs,
                    "roofline_frac": gbs / hbm_gbs, "launches_per_call": lpc})
    # the backward pass of the headline workload (CUDA-core scans)
    w = inputs.PREFILL_2K
    ms, lpc, alg = time_backward(la, w, max(1, min(steps, 5)), min(warmup, 2), stream)
    gbs = alg / (ms * 1e-3) / 1e9
    out.append({"workload": w.name, "mode": "backward", "ms": ms, "tokens_per_s": w.B * w.T / (ms * 1e-3),
                "alg_bytes": alg, "achieved_GBps": gbs, "roofline_frac": gbs / hbm_gbs, "launches_per_call": lpc})
    return out


def oracle_sample(w):
    """A bounded sample of a workload for the CPU oracle: batch row 0 with all
    of its heads over the full sequence (1/B of the work); tokens/s over the
    sample equals tokens/s over the whole workload at the same rate."""
    q, k, v, d = inputs.make_qkv(w, device="cpu", seed=w.seed)
    sl = slice(0, 1)
    return q[sl], k[sl], v[sl], None if d is None else d[sl]


def cpu_baseline(w, budget_s=8.0):
    """The oracle as it stands on the host cores, on a sample of the
    workload (oracle_sample), repeated until the time budget is used."""
    import oracle
    q, k, v, d = oracle_sample(w)
    cores = os.cpu_count() or 1
    n_streams = w.kv_heads
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.causal(q, k, v, q_heads=w.q_heads, kv_heads=w.kv_heads, feature_map=w.feature_map,
                      use_normalizer=w.use_normalizer, eps=w.eps, scale=w.scale, rule=w.rule,
                      decay=d, nthreads=cores)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 50:
            break
    tok_s = reps * w.T / el
    return {"value": tok_s, "unit": "tokens/s", "cores": min(cores, n_streams), "kind": "oracle",
            "sample": f"batch row 0 of the workload (1x{w.T} tokens, all {w.q_heads} heads, 1/{w.B} of it) run "
                      f"{reps} time(s); fp64 recurrence, one thread per (batch, kv-head) stream"}


def measured_traffic(workload):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, or None when the kernel sources changed since that capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "chunk_kernel_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    for rel, digest in rec.get("sources_sha256", {}).items():
        src = os.path.join(ROOT, rel)
        if not os.path.exists(src):
            return None
        with open(src, "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != digest:
                return None
    return rec.get("traffic_bytes_per_launch", {}).get(workload)


def run_gpu(args):
    import kernelized_linear_attention_02_gb300 as la
    world, rank, local = dist_init()
    la.lib()
    w = HEADLINE
    wd = inputs.DECODE
    pk = peaks()
    stream = torch.cuda.Stream()

    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ms, launches, nsets, _ = time_prefill(la, w, args.steps, args.warmup, stream)
        torch.cuda.synchronize()
        barrier(world)
    ms = max_over_ranks(ms, world)
    clocks = clk.summary()
    tokens = w.B * w.T
    value = tokens * world / (ms * 1e-3)
    alg = prefill_alg_bytes(w)
    achieved = alg / (ms * 1e-3) / 1e9
    e2e_ms, h2d, d2h = time_prefill_e2e(la, w, args.steps, args.warmup, stream)
    e2e_ms = max_over_ranks(e2e_ms, world)

    dec = None
    if not args.skip_decode:
        with ClockSampler(local) as dclk:
            us, dlaunch = time_decode(la, wd, args.decode_steps, args.warmup, stream)
        us = max_over_ranks(us, world)
        dbytes, sbytes = decode_alg_bytes(wd)
        dec = {"workload": wd.name, "us_per_step": us, "us_per_token": us / wd.B,
               "state_GBps": sbytes / (us * 1e-6) / 1e9, "alg_GBps": dbytes / (us * 1e-6) / 1e9,
               "roofline_frac": dbytes / (us * 1e-6) / 1e9 / pk["hbm_gbs"], "steps": args.decode_steps,
               "gpu_launches": dlaunch, "clocks": dclk.summary()}

    sweep = None
    if not args.skip_sweep:
        sweep = workload_sweep(la, max(3, min(args.steps, 10)), args.warmup, stream, pk["hbm_gbs"])

    if rank != 0:
        return
    traffic = measured_traffic(w.name)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_for(w, world),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / pk["hbm_gbs"], "traffic": traffic,
                     "peak_source": pk["source"], "alg_bytes_per_call": alg,
                     "scope": f"one la_forward_causal call ({launches / args.steps:.0f} launch(es)); traffic: the "
                              "causal pass, one launch"},
        "e2e": {"value": tokens * world / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "how": "pinned host buffers; per step h2d of q, k, v + la_forward_causal + d2h of y, "
                       "pipelined over three streams with two device buffer sets"},
        "gpu_launches": launches,
        "clocks": clocks,
        "workloads": sweep,
        "decode": dec,
    }
    if world == 1 and not args.skip_cpu:
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line), flush=True)


def run_reference(args):
    """The oracle timed as it stands on the host cores: every step runs the
    bounded sample of the headline workload (oracle_sample)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = HEADLINE
    import oracle
    q, k, v, d = oracle_sample(w)
    cores = os.cpu_count() or 1

    def step():
        oracle.causal(q, k, v, q_heads=w.q_heads, kv_heads=w.kv_heads, feature_map=w.feature_map,
                      use_normalizer=w.use_normalizer, eps=w.eps, scale=w.scale, rule=w.rule,
                      decay=d, nthreads=cores)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = (time.perf_counter() - t0) / args.steps
    value = w.T / el  # tokens of the sample (all heads) per second
    sample = (f"per step batch row 0 of the workload (1x{w.T} tokens, all {w.q_heads} heads, 1/{w.B} of it), "
              f"fp64 oracle, one thread per (batch, kv-head) stream")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 * w.B, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_for(w, world),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": min(cores, w.kv_heads),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_only(args):
    """One workload alone (optionally at another batch size): the entry point
    for profiling a single kernel on a case small enough for a full capture."""
    import dataclasses
    import kernelized_linear_attention_02_gb300 as la
    if torch.cuda.is_available():
        torch.cuda.set_device(0)
    la.lib()
    w = getattr(inputs, args.only)
    if args.batch:
        w = dataclasses.replace(w, B=args.batch)
    if args.seq_len:
        w = dataclasses.replace(w, T=args.seq_len)
    stream = torch.cuda.Stream()
    if args.backward:
        ms, lpc, alg = time_backward(la, w, args.steps, args.warmup, stream)
        gbs = alg / (ms * 1e-3) / 1e9
        print(json.dumps({"workload": w.name, "B": w.B, "mode": "backward", "ms": ms,
                          "tokens_per_s": w.B * w.T / (ms * 1e-3), "alg_bytes": alg, "achieved_GBps": gbs,
                          "roofline_frac": gbs / peaks()["hbm_gbs"], "launches_per_call": lpc}), flush=True)
        return
    causal = not args.noncausal
    ms, lpc = time_workload(la, w, args.steps, args.warmup, stream, causal)
    alg = prefill_alg_bytes(w)
    gbs = alg / (ms * 1e-3) / 1e9
    print(json.dumps({"workload": w.name, "B": w.B, "T": w.T, "mode": "causal" if causal else "noncausal", "ms": ms,
                      "tokens_per_s": w.B * w.T / (ms * 1e-3), "alg_bytes": alg, "achieved_GBps": gbs,
                      "roofline_frac": gbs / peaks()["hbm_gbs"], "launches_per_call": lpc}), flush=True)


def run_decode_only(args):
    """The decode step alone on the streaming-decode shape (B=256, H=32, D=128,
    512 MiB fp32 state), with the state built from a short prompt of
    --prompt tokens: the entry point for profiling the decode kernel on a case
    that fits a full capture.  The step's work does not depend on the prompt
    length."""
    import dataclasses
    import kernelized_linear_attention_02_gb300 as la
    torch.cuda.set_device(0)
    la.lib()
    w = dataclasses.replace(inputs.DECODE, T=args.prompt)
    stream = torch.cuda.Stream()
    us, launches = time_decode(la, w, args.decode_steps, args.warmup, stream)
    dbytes, sbytes = decode_alg_bytes(w)
    pk = peaks()
    print(json.dumps({"workload": w.name, "prompt": w.T, "us_per_step": us, "us_per_token": us / w.B,
                      "state_GBps": sbytes / (us * 1e-6) / 1e9, "alg_GBps": dbytes / (us * 1e-6) / 1e9,
                      "roofline_frac": dbytes / (us * 1e-6) / 1e9 / pk["hbm_gbs"], "gpu_launches": launches}),
          flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--decode-steps", type=int, default=1024)
    ap.add_argument("--skip-decode", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-sweep", action="store_true", help="skip the per-workload roofline sweep")
    ap.add_argument("--only", default=None, help="time one workload of linattn_inputs (e.g. LONG_8K) alone")
    ap.add_argument("--batch", type=int, default=0, help="with --only: batch size override")
    ap.add_argument("--seq-len", type=int, default=0, help="with --only: sequence length override")
    ap.add_argument("--noncausal", action="store_true", help="with --only: the non-causal pass")
    ap.add_argument("--backward", action="store_true", help="with --only: the backward pass (linear rule)")
    ap.add_argument("--decode-only", action="store_true", help="time the decode step alone (see --prompt)")
    ap.add_argument("--prompt", type=int, default=64, help="with --decode-only: prompt tokens that build the state")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.only:
        run_only(args)
    elif args.decode_only:
        run_decode_only(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
