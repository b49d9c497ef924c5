#!/usr/bin/env python
"""Benchmark of the chunkwise Kimi Delta Attention forward on GB300.

One step = one kda_fwd over the whole workload (chunk index, intra-chunk kernel,
state/output recurrence kernel) with the inputs resident in HBM.  Default workload:
dense bf16 prefill B=2, T=4096, H=16, K=V=128, chunk 64.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--cpu-seconds S]

Prints one JSON line (rank 0).  Under torchrun every rank runs an independent replica
of the workload (the path has no exchange step); value = tokens of all ranks divided by
the slowest rank's time.  ``--impl reference`` times the fp64 CPU oracle instead, on a
bounded sample of the same workload, on the host cores of rank 0.
"""
from __future__ import annotations

import argparse
import csv
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

import torch  # noqa: E402

from workloads import DECODE_WORKLOADS, WORKLOADS, make_decode_inputs, make_inputs  # noqa: E402

METRIC = "KDA fwd tokens/s and TFLOP/s (bf16, H=16, K=V=128, T=4096); % of roofline"
UNIT = "tokens/s"
DECODE_METRIC = "KDA decode step tokens/s (one token per sequence)"
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# algorithmic work (per token-head), the measurement plan's counts
# ---------------------------------------------------------------------------

def flops_per_chunk(c: int, K: int, V: int) -> int:
    """Causal/triangular work of one chunk of c tokens (2 flops per MAC): Aqk, L, the
    unit-lower solve, W, U, the three state GEMMs (W S, Qg S, K_bar^T V_new) and
    Aqk V_new."""
    return (c * (c + 1) * K + c * (c - 1) * K + (c - 1) * c * (c + 1) // 3 + c * (c + 1) * K
            + c * (c + 1) * V + 3 * 2 * c * K * V + c * (c + 1) * V)


def algorithmic(inp) -> dict:
    """Bytes and flops the method must move/do for one pass over the inputs."""
    B, T, H, K, V = (inp[x] for x in ("B", "T", "H", "K", "V"))
    esz = 2 if inp["dtype"] == torch.bfloat16 else 4
    th = B * T * H
    in_bytes = th * (esz * (2 * K + V) + 4 * K + 4)
    out_bytes = th * esz * V
    state = inp["N"] * H * K * V * 4
    s_in = state if inp["initial_state"] is not None else 0
    s_out = state
    if inp["cu_seqlens"] is not None:
        lens = (inp["cu_seqlens"][1:] - inp["cu_seqlens"][:-1]).cpu().tolist()
    else:
        lens = [T] * B
    fl = 0
    for L in lens:
        full, tail = divmod(int(L), 64)
        fl += full * flops_per_chunk(64, K, V) + (flops_per_chunk(tail, K, V) if tail else 0)
    fl *= H
    return dict(token_heads=th, tokens=B * T, in_bytes=in_bytes, out_bytes=out_bytes,
                state_in=s_in, state_out=s_out,
                bytes=in_bytes + out_bytes + s_in + s_out, flops=fl)


# ---------------------------------------------------------------------------
# environment helpers
# ---------------------------------------------------------------------------

def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world):
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks/throttle sampling while the GPU is busy."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.sel = ["-i", uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"]
        except Exception:
            self.sel = []

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", *self.sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL,
                stderr=subprocess.DEVNULL)
        except FileNotFoundError:
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
        with open(self.path) as f:
            for r in csv.reader(f):
                if len(r) >= 9:
                    rows.append([x.strip() for x in r])
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x.split()[0])
            except (ValueError, IndexError):
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i - 5] for r in rows for i in range(5, 9) if r[i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if the summary
    was taken on this workload and on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(kernel)
    if not ent or ent.get("workload") != workload:
        return None
    src = os.path.join(ROOT, ent["source"])
    if not os.path.exists(src):
        return None
    with open(src, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    return ent["bytes_per_launch"] if sha == ent.get("source_sha") else None


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and --impl reference)
# ---------------------------------------------------------------------------

def oracle_sample_rate(inp, seconds: float):
    """Time the fp64 oracle on the first T_s tokens of every (sequence, head) chain of
    the workload, T_s sized for about `seconds` of work.  Returns (tokens/s, threads,
    description)."""
    import oracle
    orc = oracle.default_oracle()
    cpu = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in inp.items()}
    B, H = cpu["B"], cpu["H"]

    def run(Ts):
        sl = {k: cpu[k][:, :Ts].contiguous() for k in ("q", "k", "v", "g", "beta")}
        t = time.perf_counter()
        orc.recurrent(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], cpu["scale"],
                      initial_state=cpu["initial_state"] if cpu["cu_seqlens"] is None else None)
        return time.perf_counter() - t

    T = cpu["T"] if cpu["cu_seqlens"] is None else int(cpu["cu_seqlens"][1])
    probe = min(T, 32)
    dt = run(probe)
    Ts = max(1, min(T, int(probe * seconds / max(dt, 1e-6))))
    dt = run(Ts)
    tokens = B * Ts
    desc = (f"fp64 token recurrence on the first {Ts} of {T} tokens of all {B}x{H} "
            f"(sequence, head) chains; tokens/s = {B}*{Ts}/time")
    return tokens / dt, orc.threads_used, desc, dt


def oracle_decode_rate(spec: dict, seconds: float):
    """Time the fp64 oracle on whole decode steps of the decode workload (every
    sequence and head advanced by its one token from its state), repeated for about
    `seconds`.  Returns (tokens/s, threads, description, seconds per step)."""
    import oracle
    orc = oracle.default_oracle()
    d = make_decode_inputs(**spec)
    tok = {x: d[x].unsqueeze(1).contiguous() for x in ("q", "k", "v", "g", "beta")}
    reps, t0 = 0, time.perf_counter()
    while True:
        orc.recurrent(tok["q"], tok["k"], tok["v"], tok["g"], tok["beta"], d["scale"],
                      initial_state=d["state"])
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = (time.perf_counter() - t0) / reps
    desc = (f"fp64 token recurrence, {reps} whole decode steps of {d['N']} sequences x "
            f"{d['H']} heads; tokens/s = {d['N']}/time per step")
    return d["N"] / dt, orc.threads_used, desc, dt


def run_reference_decode(args, rank, world):
    if rank != 0:
        return 0
    spec = DECODE_WORKLOADS[args.workload]
    per_step = min(5.0, max(0.2, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_decode_rate(spec, per_step)
    rates, threads, desc = [], 1, ""
    for _ in range(args.steps):
        r, threads, desc, _ = oracle_decode_rate(spec, per_step)
        rates.append(r)
    value = statistics.median(rates)
    line = {
        "metric": DECODE_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * spec["N"] / value,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference", "config": decode_config(args.workload, spec),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def decode_config(name: str, spec: dict) -> dict:
    return {"workload": f"{name}: N={spec['N']} H={spec['H']} K={spec['K']} V={spec['V']}",
            "l2": "flushed between timed steps (write of 4x L2)"}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    w = WORKLOADS[args.workload]
    inp = make_inputs(w)
    per_step = min(10.0, max(0.2, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample_rate(inp, per_step)
    rates, times = [], []
    threads, desc = 1, ""
    for _ in range(args.steps):
        r, threads, desc, dt = oracle_sample_rate(inp, per_step)
        rates.append(r)
        times.append(dt)
    value = statistics.median(rates)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * inp["B"] * inp["T"] / value,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": workload_config(w, inp),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, inp):
    return {"workload": f"{w.name}: B={inp['B']} T={inp['T']} H={inp['H']} K={inp['K']} "
                        f"V={inp['V']} C={inp['chunk_size']} {w.dtype_name}",
            "global_batch": inp["B"], "seq_len": inp["T"], "heads": inp["H"],
            "parallelism": "replicas",
            "l2": "flushed between timed steps (write of 4x L2)"}


# ---------------------------------------------------------------------------
# our CUDA path
# ---------------------------------------------------------------------------

def run_ours(args, rank, world, local):
    import kimi_delta_attention_11_gb300 as kda
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    kda.load_library()
    w = WORKLOADS[args.workload]
    host = make_inputs(w)
    inp = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in host.items()}
    alg = algorithmic(host)
    B, T, H, K, V, N = (inp[x] for x in ("B", "T", "H", "K", "V", "N"))
    num_seqs = N if inp["cu_seqlens"] is not None else 0
    ws = torch.empty(kda.workspace_bytes(B, T, H, K, V, num_seqs, inp["dtype"]),
                     dtype=torch.uint8, device=dev)
    o = torch.empty((B, T, H, V), dtype=inp["dtype"], device=dev)
    fin = torch.empty((N, H, K, V), dtype=torch.float32, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(4 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(evs=None):
        kda.fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                initial_state=inp["initial_state"], cu_seqlens=inp["cu_seqlens"],
                workspace=ws, out=o, final_state=fin, events=evs)

    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()

    # timed region: K steps of kda_fwd as a user calls it (the pipelined schedule where it
    # applies), a CUDA event pair on the launching stream around each step; the L2 flush
    # between steps stays outside the events
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        ev_a[i].record(stream)
        step()
        ev_b[i].record(stream)
    barrier(world)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    step_ms = sum(a.elapsed_time(b) for a, b in zip(ev_a, ev_b)) / args.steps
    ms = max_over_ranks(step_ms, world, dev)

    # per-kernel durations: the same kernels run back to back, one launch each over the
    # whole problem (kda_fwd_profiled), events between them on the launching stream
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for e in (x for row in evs for x in row):   # torch creates the CUDA event on first record
        e.record(stream)
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        step(evs[i])
    torch.cuda.synchronize()
    stage_ms = [[e[j].elapsed_time(e[j + 1]) for j in range(3)] for e in evs]

    # end to end through the public call with host buffers (pinned), copies timed
    pinned = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in host.items()}
    o_h = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    f_h = torch.empty(fin.shape, dtype=fin.dtype).pin_memory()
    dbuf = {k: torch.empty_like(inp[k]) for k in ("q", "k", "v", "g", "beta")}
    s0 = torch.empty_like(inp["initial_state"]) if inp["initial_state"] is not None else None
    cu = torch.empty_like(inp["cu_seqlens"]) if inp["cu_seqlens"] is not None else None
    h2d = sum(pinned[k].numel() * pinned[k].element_size() for k in dbuf)
    h2d += (s0.numel() * 4 if s0 is not None else 0) + (cu.numel() * 4 if cu is not None else 0)
    d2h = o_h.numel() * o_h.element_size() + f_h.numel() * 4

    def e2e_step():
        for k in dbuf:
            dbuf[k].copy_(pinned[k], non_blocking=True)
        if s0 is not None:
            s0.copy_(pinned["initial_state"], non_blocking=True)
        if cu is not None:
            cu.copy_(pinned["cu_seqlens"], non_blocking=True)
        kda.fwd(dbuf["q"], dbuf["k"], dbuf["v"], dbuf["g"], dbuf["beta"], inp["scale"],
                initial_state=s0, cu_seqlens=cu, workspace=ws, out=o, final_state=fin)
        o_h.copy_(o, non_blocking=True)
        f_h.copy_(fin, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    e_ms = []
    for _ in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        b.synchronize()
        e_ms.append(a.elapsed_time(b))
    clocks = sampler.stop()
    e2e_ms = max_over_ranks(sum(e_ms) / len(e_ms), world, dev)

    # parity spot check of the last timed output against itself being finite
    assert torch.isfinite(o.float()).all().item(), "non-finite output"

    if rank != 0:
        return 0
    tokens_all = alg["tokens"] * world
    value = tokens_all / (ms * 1e-3)
    tc = inp["dtype"] == torch.bfloat16 and K == 128 and V == 128
    # the recurrence runs value-sliced (two CTAs per chain) when 2 x chains fit the SMs
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    chains = (N if inp["cu_seqlens"] is not None else B) * H
    ho_tc = "kda_h_o_sliced_tc" if 2 * chains <= sms else "kda_h_o_tc"
    names = (["kda_chunk_index", "kda_intra_tc", ho_tc] if tc
             else ["kda_chunk_index", "kda_intra_simt", "kda_h_o_simt"])
    avg = [sum(s[j] for s in stage_ms) / args.steps for j in range(3)]
    dom = max(range(3), key=lambda j: avg[j])
    kb = {names[0]: 0, names[1]: alg["in_bytes"],
          names[2]: alg["out_bytes"] + alg["state_in"] + alg["state_out"]}
    peak, peak_kind = measured_peaks()
    path_achieved = alg["bytes"] / (ms * 1e-3) / 1e9
    launches_per_step = kda.launch_count(B, T, H, K, V, num_seqs, inp["dtype"])
    sched = kda.schedule(B, T, H, K, V, num_seqs, inp["dtype"])
    # the fused schedule's single kernel is the whole step and moves the whole path's
    # algorithmic bytes; the scan's four launches are rated as one path
    fused = sched in ("fused", "scan")
    if fused:
        dom_name = "kda_fused_tc" if sched == "fused" else "scan schedule (4 launches)"
        achieved = path_achieved
    else:
        dom_name = names[dom]
        achieved = kb[names[dom]] / (avg[dom] * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype_name, "data": "synthetic",
        "config": workload_config(w, host),
        "tflops": alg["flops"] * world / (ms * 1e-3) / 1e12,
        "roofline": {"bound": "hbm", "kernel": dom_name, "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "traffic": ncu_traffic(dom_name, w.name)},
        "path_roofline": {"algorithmic_bytes": alg["bytes"], "achieved_GBps": path_achieved,
                          "frac_of_measured_hbm": path_achieved / peak,
                          "algorithmic_flops": alg["flops"]},
        "stage_ms": dict(zip(names, avg)),
        "schedule": sched,
        "stage_schedule": ("the two-kernel schedule, kernels back to back (the timed steps run "
                           f"the {sched} schedule)") if fused else
                          ("kernels back to back, one launch each (the timed steps overlap "
                           "them when the call is pipelined)"),
        "e2e": {"value": tokens_all / (e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "wall_s_timed": wall,
    }
    if world == 1 and not args.no_cpu_baseline:
        rate, threads, desc, _ = oracle_sample_rate(host, args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
                                "sample": desc}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# decode step (a second workload on the same state)
# ---------------------------------------------------------------------------

def run_decode(args, rank, world, local):
    """Times kda_decode: one token for each of N sequences; HBM-bound on the state."""
    import kimi_delta_attention_11_gb300 as kda
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    kda.load_library()
    spec = DECODE_WORKLOADS[args.workload]
    inp = make_decode_inputs(device=str(dev), **spec)
    N, H, K, V, dt = (inp[x] for x in ("N", "H", "K", "V", "dtype"))
    esz = 2 if dt == torch.bfloat16 else 4
    state_bytes = N * H * K * V * 4
    step_bytes = 2 * state_bytes + N * H * (esz * (2 * K + 2 * V) + 4 * K + 4)
    o = torch.empty((N, H, V), dtype=dt, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(4 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kda.decode(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state"],
                   inp["scale"], out=o)

    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(args.warmup):
        flush.zero_()
        step()
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        ev_a[i].record(stream)
        step()
        ev_b[i].record(stream)
    barrier(world)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in zip(ev_a, ev_b)) / args.steps, world, dev)
    clocks = sampler.stop()
    assert torch.isfinite(o.float()).all().item() and torch.isfinite(inp["state"]).all().item()
    if rank != 0:
        return 0
    peak, peak_kind = measured_peaks()
    achieved = step_bytes / (ms * 1e-3) / 1e9
    line = {
        "metric": DECODE_METRIC, "value": N * world / (ms * 1e-3),
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if dt == torch.bfloat16 else "f32", "data": "synthetic",
        "config": decode_config(args.workload, spec),
        "roofline": {"bound": "hbm", "kernel": "kda_decode_kernel", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "traffic": ncu_traffic("kda_decode", args.workload),
                     "bytes_per_step": step_bytes},
        "gpu_launches": args.steps, "clocks": clocks, "wall_s_timed": wall,
    }
    if world == 1 and not args.no_cpu_baseline:
        r, threads, desc, _ = oracle_decode_rate(spec, min(args.cpu_seconds, 5.0))
        line["cpu_baseline"] = {"value": r, "unit": "tokens/s", "cores": threads,
                                "kind": "oracle", "sample": desc}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[1])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + sorted(DECODE_WORKLOADS),
                    default="dense_bf16")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_info()
    if args.workload in DECODE_WORKLOADS:
        if args.impl == "reference":
            return run_reference_decode(args, rank, world)
        init_dist(world)
        try:
            return run_decode(args, rank, world, local)
        finally:
            if world > 1 and torch.distributed.is_initialized():
                torch.distributed.destroy_process_group()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    init_dist(world)
    try:
        return run_ours(args, rank, world, local)
    finally:
        if world > 1 and torch.distributed.is_initialized():
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
