"""Benchmark of the KDA mixer step on GB300 (one JSON line on stdout, rank 0).

Headline (``value``): single-token decode throughput of one KDA mixer step, tokens/s, on the
decode_b64 workload (B=64 sequences, H=8 heads, dk=dv=128, FP32 pool of 256 slots, 64 decode
steps, seed 1), i.e. B / (device time per decode launch).  One bench step = the workload's 64
decode launches for each of 8 layer instances (separate slot pools, same weights and inputs),
interleaved layer-fastest and captured as one CUDA graph: the 8 x 32 MiB of touched state
exceeds the 126 MB L2, so every launch streams its state from HBM (inputs larger than L2, no
flush), and launches follow each other as they do in a served model.  Inputs are resident in
HBM before timing; CUDA events bracket the graph replays on the launching stream.
The same workload is also timed cold (``rows.decode_b64_cold``): L2 flushed before every
single launch (256 MiB written, then 256 MiB read), each launch bracketed by its own events,
which adds the full launch latency to every launch.

Also reported on the same line:
  roofline      achieved HBM GB/s of the decode kernel (algorithmic bytes / mean launch time)
                against the measured copy bandwidth (MEASURED_PEAKS.json), with the ncu DRAM
                traffic per launch when a capture of the current kernel exists;
  e2e           the same workload through the public API with pinned host buffers: each step
                copies its inputs host->device, runs the 64 launches and copies the outputs back;
  cpu_baseline  the FP64 oracle on the host cores on the same workload (and on one core);
  rows          the other measured paths: decode_small, decode_b256 (BF16 pool), verify_b64 +
                commit, prefill_b4, each with its own device time, tokens/s, GB/s and roofline
                fraction.
``--impl reference`` times the FP64 oracle instead (the reference arm of this comparison).

Output: one JSON line on stdout (the figures above, each row as [us per launch, GB/s, fraction
of measured HBM, ncu DRAM bytes per launch], short enough to survive a 1.5 KB log tail), and
before it, on stderr, the same run with every figure's description and timing mode.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import numpy as np  # noqa: E402

HEADLINE = "decode_b64"
METRIC = "KDA decode tokens/s (decode_b64) and achieved HBM GB/s; prefill tokens/s (prefill_b4)"


def base_config():
    """The headline workload, as both arms (this library and the FP64 oracle) report it."""
    return {"workload": HEADLINE, "B": 64, "H": 8, "dk": 128, "dv": 128, "decode_steps": 64,
            "pool_slots": 256, "state_dtype": "f32"}
L2_FLUSH_BYTES = 256 << 20
NAMES = ("q", "k", "v", "f_a", "beta", "gate")


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ----------------------------------------------------------------------------- algorithmic bytes

def decode_bytes(B, H, state_bytes, T=1):
    """Bytes a decode launch must move: state read + write, conv window read + write, the
    token inputs and output, the layer weights."""
    C = H * 128
    state = B * H * 128 * 128 * state_bytes * 2
    conv = B * 3 * 3 * C * 2 * 2
    io = B * T * (4 * C * 2 + C * 2 + H * 2 + 128 * 2)   # q,k,v,gate in, out, beta, f_a
    weights = C * 128 * 2 + 3 * C * 4 * 2 + H * 4 + C * 4 + 128 * 4 + B * 4
    return state + conv + io + weights


def verify_bytes(B, H, T, state_bytes):
    C = H * 128
    state_in = B * H * 128 * 128 * state_bytes
    records = B * T * H * 128 * 128 * 4
    conv_in = B * 3 * 3 * C * 2
    conv_rec = B * T * 3 * 3 * C * 2
    io = B * T * (4 * C * 2 + C * 2 + H * 2 + 128 * 2)
    weights = C * 128 * 2 + 3 * C * 4 * 2 + H * 4 + C * 4 + 128 * 4 + B * 4
    return state_in + records + conv_in + conv_rec + io + weights


def commit_bytes(accepted, H, state_bytes):
    n = int(np.count_nonzero(accepted))
    C = H * 128
    return n * (H * 128 * 128 * (4 + state_bytes) + 2 * 3 * 3 * C * 2) + accepted.size * 8


def prefill_bytes(B, L, H, state_bytes):
    C = H * 128
    io = B * L * (4 * C * 2 + C * 2 + H * 2 + 128 * 2)
    state = B * H * 128 * 128 * state_bytes * 2
    weights = C * 128 * 2 + 3 * C * 4 * 2 + H * 4 + C * 4 + 128 * 4
    return io + state + weights + B * 3 * 3 * C * 2 * 2


def prefill_flops(B, L, H, chunk=64):
    """Dense-contraction flops of the chunked form per chunk-head (C = chunk, d = 128):
    f_b projection 2Cdr, gated K K^T and Q K^T 2*2C^2d, W and U 2*2C^2d, W S and Q S 2*2Cd^2,
    intra-chunk attention times V' 2C^2d, state update 2Cd^2."""
    d, C = 128, chunk
    per = 2 * C * d * 128 + 4 * C * C * d + 4 * C * C * d + 4 * C * d * d + 2 * C * C * d + 2 * C * d * d
    n_chunks = (L + C - 1) // C
    return per * n_chunks * B * H


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if not self.path or not os.path.exists(self.path):
            return out
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return out
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i in range(4) if r[i].lower() == "active"})
        out.update(sm_mhz=statistics.median(r[0] for r in rows), sm_max_mhz=max(r[1] for r in rows),
                   reasons=reasons, samples=len(rows))
        return out


# ----------------------------------------------------------------------------- helpers

def source_digest(rel):
    """sha1 over a CUDA source and, recursively, every in-tree header it includes with quotes
    (each once, in the order first met), so that an edit to a shared header also counts as a
    change of the kernel."""
    import hashlib
    import re

    h, seen = hashlib.sha1(), set()

    def walk(path):
        path = os.path.normpath(path)
        if path in seen or not os.path.isfile(path):
            return
        seen.add(path)
        with open(path, "rb") as f:
            text = f.read()
        h.update(text)
        for inc in re.findall(rb'^\s*#\s*include\s+"([^"]+)"', text, re.M):
            walk(os.path.join(os.path.dirname(path), inc.decode()))

    walk(os.path.join(ROOT, rel))
    return h.hexdigest()


def ncu_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu capture of this kernel (profiles/traffic.json),
    or None when there is none or the kernel's source or headers changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            entry = json.load(f).get(kernel_key)
        return int(entry["bytes"]) if source_digest(entry["source"]).startswith(entry["sha1"]) else None
    except Exception:
        return None


def decode_kernel_key(torch, B, H, state_dtype):
    """Which single-token decode kernel the library runs for this shape (its traffic entry):
    a cluster of four CTAs per tile while 4 x B x H CTAs fit on the SMs; beyond that, BF16 pools
    the BF16 decode kernel, FP32 pools the tile kernel while one resident wave of it (2 CTAs per
    SM) holds all B x H tiles and the paired-tile kernel beyond."""
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    if 4 * B * H <= sms:
        return "decode_cluster_" + state_dtype
    if state_dtype == "bf16":
        return "decode_bf16"
    return "decode_f32_pair" if B * H > 2 * sms else "decode_f32"


def roofline(bytes_per_launch, ms_per_launch, hbm_peak, src, kernel_key):
    achieved = bytes_per_launch / (ms_per_launch * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(achieved / hbm_peak, 4), "peak_source": src + " (MEASURED_PEAKS.json hbm_gbs)" if src == "measured" else "fallback 6.8 TB/s",
            "frac_of_nominal_8TBs": round(achieved / 8000.0, 4),
            "traffic": ncu_traffic(kernel_key), "bytes_algorithmic": int(bytes_per_launch)}


class Flusher:
    """Evicts L2 before a timed launch: writes a buffer twice the size of L2, then reads a
    second one, so that the dirty lines of the write are written back before the timed kernel
    starts (otherwise their write-back would be charged to it) and L2 is left holding clean
    lines of unrelated data."""

    def __init__(self, torch):
        self.torch = torch
        self.wbuf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
        self.rbuf = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    def __call__(self):
        self.wbuf.fill_(1.0)
        self.rbuf.sum()


def time_launches(torch, launches, flush, stream=None):
    """Runs each callable with an L2 flush before it; returns per-launch device ms."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in launches]
    ends = [torch.cuda.Event(enable_timing=True) for _ in launches]
    for fn, s, e in zip(launches, starts, ends):
        if flush is not None:
            flush()
        s.record()
        fn()
        e.record()
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


# ----------------------------------------------------------------------------- GPU rows

def setup_case(name, **kw):
    from gpu_io import device_inputs, device_layer, device_pool
    from kda_inputs import make
    import torch

    case = make(name, **kw)
    return case, device_layer(case), device_pool(case), device_inputs(case), torch.from_numpy(case.slot_ids).cuda()


def bench_decode(torch, K, name, steps, warmup, flush, hbm, src):
    case, layer, pool, ins, slots = setup_case(name)
    n_steps = ins["q"].shape[0]
    outs = torch.empty(n_steps, case.B, layer.H * 128, dtype=torch.bfloat16, device="cuda")
    launches = [(lambda s=s: K.kda_decode(layer, pool, slots, *(ins[n][s] for n in NAMES), out=outs[s]))
                for s in range(n_steps)]
    for _ in range(warmup):
        time_launches(torch, launches, flush)
    times = []
    for _ in range(steps):
        times.extend(time_launches(torch, launches, flush))
    ms_launch = statistics.mean(times)
    sb = 2 if case.pool.state_dtype == "bf16" else 4
    nbytes = decode_bytes(case.B, layer.H, sb)
    return {
        "workload": name, "B": case.B, "H": layer.H, "state_dtype": case.pool.state_dtype,
        "launches_per_step": n_steps, "tokens_per_step": case.B * n_steps,
        "us_per_launch": round(ms_launch * 1e3, 3),
        "us_per_launch_median": round(statistics.median(times) * 1e3, 3),
        "ms_per_step": ms_launch * n_steps,
        "tokens_per_s": case.B / (ms_launch * 1e-3),
        "roofline": roofline(nbytes, ms_launch, hbm, src, decode_kernel_key(torch, case.B, case.layer.H, case.pool.state_dtype)),
        "kernel_launches": len(times),
    }, (case, layer, pool, ins, slots)


def max_over_ranks(torch, dist, x, device):
    """The largest of the ranks' values of x (x itself when the job has one rank)."""
    if dist is None:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank_step, world, ms_step_max):
    """Whole-job throughput: the units every rank processed in a step over the slowest rank's
    step time (each rank runs the same workload on its own GPU: weak scaling)."""
    return units_per_rank_step * world / (ms_step_max * 1e-3)


def access_pattern_ceiling(torch, state_bytes, layers, n_steps, steps=5, warmup=3):
    """The decode graph's memory traffic without its arithmetic: each launch reads and writes
    back `state_bytes` in place (a torch elementwise multiply) in buffer l of `layers`, in the
    graph's order and count.  Context for the roofline: what this access pattern reaches."""
    bufs = [torch.ones(state_bytes // 4, device="cuda") for _ in range(layers)]

    def step():
        for _ in range(n_steps):
            for b in bufs:
                b.mul_(1.0)

    step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            step()
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(warmup):
        graph.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / steps / (n_steps * layers) * 1e3
    del bufs, graph
    return {"us_per_launch": round(us, 3), "GB_per_s": round(2 * state_bytes / (us * 1e-6) / 1e9, 1),
            "what": "in-place read + write of each launch's state bytes (contiguous, torch elementwise) "
                    "through the same rotation of layer buffers, one CUDA graph of the same launch count"}


def bench_decode_steady(torch, K, name, layers, steps, warmup, hbm, src, sync_ranks=None):
    """The workload's n_steps decode launches for each of `layers` layer instances (separate
    slot pools, same weights and inputs), interleaved layer-fastest and captured as one CUDA
    graph, replayed back to back.  The touched state of all layers (layers x touched state)
    exceeds the 126 MB L2, so each launch streams its state from HBM without an explicit flush,
    and launch overhead is pipelined as it is in a served model.  Per-launch time = step time /
    (n_steps x layers)."""
    from gpu_io import device_pool

    case, layer, pool0, ins, slots = setup_case(name)
    pools = [pool0] + [device_pool(case) for _ in range(layers - 1)]
    n_steps = ins["q"].shape[0]
    outs = torch.empty(layers, n_steps, case.B, layer.H * 128, dtype=torch.bfloat16, device="cuda")

    def step():
        for s in range(n_steps):
            for li in range(layers):
                K.kda_decode(layer, pools[li], slots, *(ins[n][s] for n in NAMES), out=outs[li, s])

    step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            step()
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    if sync_ranks:
        sync_ranks()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    if sync_ranks:
        sync_ranks()
    assert K.kda_get_error(pool0) == 0
    ms_step = e0.elapsed_time(e1) / steps
    launches = n_steps * layers
    working_set = layers * case.B * layer.H * 128 * 128 * (2 if case.pool.state_dtype == "bf16" else 4)
    ms_launch = ms_step / launches
    sb = 2 if case.pool.state_dtype == "bf16" else 4
    nbytes = decode_bytes(case.B, layer.H, sb)
    ceiling = access_pattern_ceiling(torch, case.B * layer.H * 128 * 128 * sb, layers, n_steps)
    return {
        "workload": name, "B": case.B, "H": layer.H, "state_dtype": case.pool.state_dtype,
        "layers": layers, "launches_per_step": launches, "tokens_per_step": case.B * launches,
        "access_pattern_ceiling": ceiling,
        "us_per_launch": round(ms_launch * 1e3, 3), "ms_per_step": ms_step,
        "tokens_per_s": case.B / (ms_launch * 1e-3),
        "roofline": roofline(nbytes, ms_launch, hbm, src, decode_kernel_key(torch, case.B, case.layer.H, case.pool.state_dtype)),
        "kernel_launches": launches * steps,
        "timing": "one CUDA graph per step, events around the replays, no flush",
        "state_working_set_bytes": working_set,
        "l2_resident": working_set < torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size,
    }


def bench_verify(torch, K, steps, warmup, flush, hbm, src):
    case, layer, pool, ins, slots = setup_case("verify_b64")
    B, T = case.B, ins["q"].shape[1]
    out = torch.empty(B, T, layer.H * 128, dtype=torch.bfloat16, device="cuda")
    rec = torch.empty(B, T, layer.H, 128, 128, dtype=torch.float32, device="cuda")
    recw = torch.empty(B, T, 3, 3, layer.H * 128, dtype=torch.bfloat16, device="cuda")
    acc = torch.from_numpy(case.accepted).cuda()
    snap = (pool.state.clone(), pool.conv_state.clone())

    def ver():
        K.kda_verify(layer, pool, slots, *(ins[n] for n in NAMES), out=out, rec_state=rec, rec_conv=recw)

    def com():
        K.kda_commit(pool, slots, acc, rec, recw)

    tv, tc = [], []
    for i in range(warmup + steps):
        pool.state.copy_(snap[0])
        pool.conv_state.copy_(snap[1])
        a, c = time_launches(torch, [ver, com], flush)
        if i >= warmup:
            tv.append(a)
            tc.append(c)
    mv, mc = statistics.mean(tv), statistics.mean(tc)
    vb = verify_bytes(B, layer.H, T, 4)
    cb = commit_bytes(case.accepted, layer.H, 4)
    return {
        "workload": "verify_b64", "B": B, "H": layer.H, "T": T,
        "verify_us": round(mv * 1e3, 3), "commit_us": round(mc * 1e3, 3),
        "draft_tokens_per_s": B * T / ((mv + mc) * 1e-3),
        "verify_roofline": roofline(vb, mv, hbm, src, "verify_f32"),
        "commit_roofline": roofline(cb, mc, hbm, src, "commit_f32"),
    }


def _graph(torch, fn):
    """fn() captured once as a CUDA graph (after one eager run, which does the library's set-up)."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    return g


def _replay_ms(torch, g, steps, warmup):
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def bench_verify_steady(torch, K, layers, reps, steps, warmup, hbm, src):
    """verify_b64 on `layers` layer instances (separate pools and record buffers, same weights
    and inputs), `reps` rounds of one verify per layer captured as one CUDA graph and replayed
    back to back: 8 x (32 MiB of state + 128 MiB of records) exceeds L2, so every launch moves
    its bytes through HBM; programmatic dependent launch overlaps each launch's start with the
    previous one's tail, as in a served model."""
    from gpu_io import device_pool

    case, layer, pool0, ins, slots = setup_case("verify_b64")
    B, T, H = case.B, ins["q"].shape[1], layer.H
    pools = [pool0] + [device_pool(case) for _ in range(layers - 1)]
    bufs = [(torch.empty(B, T, H * 128, dtype=torch.bfloat16, device="cuda"),
             torch.empty(B, T, H, 128, 128, dtype=torch.float32, device="cuda"),
             torch.empty(B, T, 3, 3, H * 128, dtype=torch.bfloat16, device="cuda")) for _ in range(layers)]

    def step():
        for _ in range(reps):
            for li in range(layers):
                o, r, w = bufs[li]
                K.kda_verify(layer, pools[li], slots, *(ins[n] for n in NAMES), out=o, rec_state=r, rec_conv=w)

    g = _graph(torch, step)
    ms = _replay_ms(torch, g, steps, warmup)
    assert K.kda_get_error(pool0) == 0
    us = ms * 1e3 / (reps * layers)
    del g, bufs
    return {"workload": "verify_b64", "layers": layers, "launches_per_step": reps * layers,
            "us_per_launch": round(us, 3), "draft_tokens_per_s": B * T / (us * 1e-6),
            "roofline": roofline(verify_bytes(B, H, T, 4), us * 1e-3, hbm, src, "verify_f32"),
            "timing": "one CUDA graph of verify launches over 8 layer instances, events around the replays, no flush"}


def bench_resume_steady(torch, K, layers, reps, steps, warmup, hbm, src):
    """The step after verify_b64 in steady state: kda_decode_resume (the accepted lengths'
    records committed inside the decode) on `layers` layer instances, as one CUDA graph."""
    from gpu_io import bf16_dev, device_pool
    from kda_inputs import make_verify

    case, layer, pool0, ins, slots = setup_case("verify_b64")
    B, T, H = case.B, ins["q"].shape[1], layer.H
    pools = [pool0] + [device_pool(case) for _ in range(layers - 1)]
    prev = [K.kda_verify(layer, pl, slots, *(ins[n] for n in NAMES)) for pl in pools]
    acc = torch.from_numpy(case.accepted).cuda()
    nxt = make_verify(seed=case.seed + 100, B=B, H=H, T=1, num_slots=B).inputs
    stepin = {n: bf16_dev(nxt[n][:, 0]) for n in NAMES}
    outs = [torch.empty(B, H * 128, dtype=torch.bfloat16, device="cuda") for _ in range(layers)]

    def step():
        for _ in range(reps):
            for li in range(layers):
                _, r, w = prev[li]
                K.kda_decode_resume(layer, pools[li], slots, (acc, r, w), *(stepin[n] for n in NAMES), out=outs[li])

    g = _graph(torch, step)
    ms = _replay_ms(torch, g, steps, warmup)
    assert K.kda_get_error(pool0) == 0
    us = ms * 1e3 / (reps * layers)
    del g
    return {"workload": "decode_resume after verify_b64", "layers": layers, "launches_per_step": reps * layers,
            "us_per_launch": round(us, 3),
            "roofline": roofline(decode_bytes(B, H, 4), us * 1e-3, hbm, src, "decode_resume_f32"),
            "timing": "one CUDA graph of decode_resume launches over 8 layer instances, events around the replays, no flush"}


def bench_resume(torch, K, steps, warmup, flush, hbm, src):
    """The step after a verify_b64 step: kda_commit + kda_decode against kda_decode_resume
    (the commit fused into the decode), each timed from a flushed L2 as one region."""
    from kda_inputs import make_verify

    case, layer, pool, ins, slots = setup_case("verify_b64")
    B, T, H = case.B, ins["q"].shape[1], layer.H
    out, rec, recw = K.kda_verify(layer, pool, slots, *(ins[n] for n in NAMES))
    acc = torch.from_numpy(case.accepted).cuda()
    nxt = make_verify(seed=case.seed + 100, B=B, H=H, T=1, num_slots=B).inputs
    from gpu_io import bf16_dev
    step = {n: bf16_dev(nxt[n][:, 0]) for n in NAMES}
    o = torch.empty(B, H * 128, dtype=torch.bfloat16, device="cuda")
    snap = (pool.state.clone(), pool.conv_state.clone())

    def unfused():
        K.kda_commit(pool, slots, acc, rec, recw)
        K.kda_decode(layer, pool, slots, *(step[n] for n in NAMES), out=o)

    def fused():
        K.kda_decode_resume(layer, pool, slots, (acc, rec, recw), *(step[n] for n in NAMES), out=o)

    tu, tf = [], []
    for i in range(warmup + steps):
        pool.state.copy_(snap[0])
        pool.conv_state.copy_(snap[1])
        (a,) = time_launches(torch, [unfused], flush)
        pool.state.copy_(snap[0])
        pool.conv_state.copy_(snap[1])
        (f,) = time_launches(torch, [fused], flush)
        if i >= warmup:
            tu.append(a)
            tf.append(f)
    mu, mf = statistics.mean(tu), statistics.mean(tf)
    return {
        "workload": "verify_b64 accepted lengths, then one decode step",
        "B": B, "H": H, "prev_T": T,
        "commit_plus_decode_us": round(mu * 1e3, 3), "decode_resume_us": round(mf * 1e3, 3),
        "saved_us": round((mu - mf) * 1e3, 3),
        "decode_resume_roofline": roofline(decode_bytes(B, H, 4), mf, hbm, src, "decode_resume_f32"),
    }


def bench_prefill(torch, K, steps, warmup, flush, hbm, src, tflops, tsrc):
    case, layer, pool, ins, slots = setup_case("prefill_b4")
    B, L = case.B, ins["q"].shape[1]
    out = torch.empty(B, L, layer.H * 128, dtype=torch.bfloat16, device="cuda")
    ws_bytes = K.kda_prefill_workspace_size(layer, B, L, case.chunk)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    zero_state, zero_conv = pool.state.clone(), pool.conv_state.clone()

    def run():
        K.kda_prefill(layer, pool, slots, *(ins[n] for n in NAMES), chunk=case.chunk, out=out,
                      workspace=ws)

    times = []
    for i in range(warmup + steps):
        pool.state.copy_(zero_state)
        pool.conv_state.copy_(zero_conv)
        (t,) = time_launches(torch, [run], flush)
        if i >= warmup:
            times.append(t)
    ms = statistics.mean(times)
    nb = prefill_bytes(B, L, layer.H, 4)
    fl = prefill_flops(B, L, layer.H, case.chunk)
    return {
        "workload": "prefill_b4", "B": B, "L": L, "H": layer.H, "chunk": case.chunk,
        "ms": round(ms, 4), "tokens_per_s": B * L / (ms * 1e-3),
        "workspace_bytes": int(ws_bytes),
        "roofline_hbm": roofline(nb, ms, hbm, src, "prefill_f32"),
        "roofline_tensor": {"bound": "tensor", "achieved": round(fl / (ms * 1e-3) / 1e12, 2),
                            "peak": tflops, "unit": "TFLOP/s", "frac": round(fl / (ms * 1e-3) / 1e12 / tflops, 4),
                            "flops_algorithmic": int(fl), "peak_source": tsrc},
    }


def bench_e2e(torch, K, steps, warmup):
    """decode_b64 through the public API with pinned host buffers.  Every step copies its 64
    decode steps' inputs host -> device, runs the 64 kda_decode calls and reads the outputs
    back; all of it lies inside the timed region.  The headline replays the 64 calls from CUDA
    graphs captured once through the same API, with the inputs double-buffered: step i + 1's
    inputs upload on a copy stream while step i computes (the way a serving loop overlaps its
    host traffic).  The eager figure issues each call from Python with no overlap."""
    from gpu_io import device_layer, device_pool
    from kda_inputs import make

    case = make(HEADLINE)
    layer, pool = device_layer(case), device_pool(case)
    slots = torch.from_numpy(case.slot_ids).cuda()
    host = {n: torch.from_numpy(np.ascontiguousarray(case.inputs[n]).view(np.int16)).view(torch.bfloat16).pin_memory()
            for n in NAMES}
    devs = [{n: torch.empty_like(host[n], device="cuda") for n in NAMES} for _ in range(2)]
    n_steps = host["q"].shape[0]
    out_dev = torch.empty(n_steps, case.B, layer.H * 128, dtype=torch.bfloat16, device="cuda")
    out_host = torch.empty_like(out_dev, device="cpu").pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_host.numel() * out_host.element_size()

    def calls(dev):
        for s in range(n_steps):
            K.kda_decode(layer, pool, slots, *(dev[n][s] for n in NAMES), out=out_dev[s])

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        calls(devs[0])               # first use outside capture (the library's setup runs here)
    torch.cuda.current_stream().wait_stream(side)
    graphs = []
    for dev in devs:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            calls(dev)
        graphs.append(g)
    compute = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    uploaded = [torch.cuda.Event(), torch.cuda.Event()]
    consumed = [torch.cuda.Event(), torch.cuda.Event()]

    def upload(i):                   # step i's inputs into buffer i % 2, on the copy stream
        buf = i % 2
        with torch.cuda.stream(copy):
            copy.wait_event(consumed[buf])       # the graph that last read this buffer is done
            for n in NAMES:
                devs[buf][n].copy_(host[n], non_blocking=True)
            uploaded[buf].record(copy)

    def run_pipelined(n):
        begin = torch.cuda.Event()
        begin.record(compute)        # no upload starts before the timed region does
        copy.wait_event(begin)
        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload(i + 1)
            compute.wait_event(uploaded[i % 2])
            graphs[i % 2].replay()
            consumed[i % 2].record(compute)
            out_host.copy_(out_dev, non_blocking=True)

    def step_serial():                # graph replay, copies not overlapped
        for n in NAMES:
            devs[0][n].copy_(host[n], non_blocking=True)
        graphs[0].replay()
        out_host.copy_(out_dev, non_blocking=True)

    def step_eager():
        for n in NAMES:
            devs[0][n].copy_(host[n], non_blocking=True)
        calls(devs[0])
        out_host.copy_(out_dev, non_blocking=True)

    prepared = [K.prepare_decode(layer, pool, slots, *(devs[0][n][s] for n in NAMES), out=out_dev[s])
                for s in range(n_steps)]

    def step_prepared():               # the same calls, checked once and bound to the buffers
        for n in NAMES:
            devs[0][n].copy_(host[n], non_blocking=True)
        for call in prepared:
            call()
        out_host.copy_(out_dev, non_blocking=True)

    def timed(step):
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(steps):
            step()
        t1.record()
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / steps

    for ev in consumed:
        ev.record(compute)
    run_pipelined(warmup)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    run_pipelined(steps)
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / steps

    ms_serial = timed(step_serial)
    ms_eager = timed(step_eager)
    ms_prep = timed(step_prepared)
    return {"value": case.B * n_steps / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
            "tokens_per_step": case.B * n_steps,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "mode": "64 public-API kda_decode calls replayed from CUDA graphs; every step's inputs uploaded "
                    "(double-buffered, overlapping the previous step) and outputs read back inside the timed region",
            "serial": {"value": case.B * n_steps / (ms_serial * 1e-3), "ms_per_step": ms_serial,
                       "mode": "the same graph replay with the copies not overlapped"},
            "eager": {"value": case.B * n_steps / (ms_eager * 1e-3), "ms_per_step": ms_eager,
                      "mode": "64 kda_decode calls from Python per step, copies not overlapped"},
            "prepared": {"value": case.B * n_steps / (ms_prep * 1e-3), "ms_per_step": ms_prep,
                         "mode": "64 prepare_decode calls (checked once, bound to the buffers) from Python "
                                 "per step, copies not overlapped"}}


# ----------------------------------------------------------------------------- oracle (CPU) arm

def oracle_decode_run(min_seconds=5.0):
    """The FP64 oracle, as it stands, on the decode_b64 workload (whole workload, repeated until
    `min_seconds` of CPU time have passed)."""
    import oracle
    from case_io import gathered_state, gathered_window, oracle_layer, storage_mode
    from kda_inputs import make

    case = make(HEADLINE)
    L = oracle_layer(case)
    S0, W0 = gathered_state(case), gathered_window(case)
    ins = [case.inputs[n] for n in NAMES]
    tokens, reps = 0, 0
    t0 = time.perf_counter()
    while True:
        oracle.decode(L, S0, W0, *ins, storage=storage_mode(case))
        reps += 1
        tokens += case.B * ins[0].shape[0]
        if time.perf_counter() - t0 >= min_seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": tokens / dt, "unit": "tokens/s", "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"decode_b64 whole workload (64 steps x 64 sequences x 8 heads) x{reps}, FP64 C oracle, OpenMP over (sequence, head)",
            "seconds": round(dt, 3)}


def oracle_single_core():
    """The same oracle pinned to one OpenMP thread: one pass over the decode_b64 workload."""
    import oracle

    cores = oracle.max_threads()
    oracle.set_threads(1)
    try:
        r = oracle_decode_run(min_seconds=0.0)
    finally:
        oracle.set_threads(cores)
    return {"value": r["value"], "unit": "tokens/s", "cores": 1, "seconds": r["seconds"],
            "sample": "decode_b64 whole workload once, one thread"}


def run_reference(args, rank):
    if rank != 0:
        return 0
    t0 = time.perf_counter()
    ms = []
    for _ in range(args.warmup):
        oracle_decode_run(min_seconds=0.0)
    for _ in range(args.steps):
        r = oracle_decode_run(min_seconds=0.0)
        ms.append(4096 / r["value"] * 1e3)
    ms_step = statistics.mean(ms)
    value = 4096 / (ms_step * 1e-3)
    cb = {"value": value, "unit": "tokens/s", "cores": __import__("oracle").max_threads(), "kind": "oracle",
          "sample": "decode_b64 whole workload per step (64 steps x 64 sequences x 8 heads), FP64 C oracle"}
    line = {"impl": "reference", "metric": METRIC, "value": value,
            "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded, kda_inputs)",
            "config": dict(base_config(), parallelism="host cores (rank 0)"),
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(time.perf_counter() - t0, 2)}
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------- output

ROW_FIELDS = "us/launch, GB/s, frac of measured HBM, ncu DRAM B/launch"


def _r(x, nd=1):
    return None if x is None else round(float(x), nd)


def _row(us, rl):
    return [_r(us, 2), _r(rl["achieved"]), _r(rl["frac"], 3), rl.get("traffic")]


def compact_rows(rows):
    """Each measured row as [us, GB/s, frac, traffic] (prefill: ms, tokens/s, HBM and tensor
    fractions)."""
    out = {"fields": ROW_FIELDS}
    for name in ("decode_b64_cold", "decode_b256", "decode_b256_cold", "decode_small", "decode_small_cold"):
        if name in rows:
            out[name] = _row(rows[name]["us_per_launch"], rows[name]["roofline"])
    if "verify_b64" in rows:
        v = rows["verify_b64"]
        out["verify_b64"] = _row(v["verify_us"], v["verify_roofline"])
        out["commit_b64"] = _row(v["commit_us"], v["commit_roofline"])
    for name in ("verify_b64_steady", "decode_resume_b64_steady"):
        if name in rows:
            out[name] = _row(rows[name]["us_per_launch"], rows[name]["roofline"])
    if "resume_b64" in rows:
        r = rows["resume_b64"]
        out["decode_resume_b64"] = _row(r["decode_resume_us"], r["decode_resume_roofline"])
        out["commit_plus_decode_us"] = _r(r["commit_plus_decode_us"], 2)
    if "prefill_b4" in rows:
        p = rows["prefill_b4"]
        out["prefill_b4"] = {"ms": _r(p["ms"], 4), "tokens_per_s": _r(p["tokens_per_s"], 0),
                             "hbm_frac": _r(p["roofline_hbm"]["frac"], 4), "dram_B": p["roofline_hbm"].get("traffic"),
                             "tflops": _r(p["roofline_tensor"]["achieved"], 2),
                             "tensor_frac": _r(p["roofline_tensor"]["frac"], 4)}
    return out


def compact_line(args, world, value, ms_step, head, e2e, clocks, rows, cpu):
    rl = head["roofline"]
    line = {
        "metric": METRIC, "value": _r(value, 0), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": _r(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded, kda_inputs)",
        "config": {**base_config(), "layer_instances": head["layers"],
                   "l2": "inputs larger than L2 (8 x 32 MiB of state per step), no flush",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "us_per_launch": head["us_per_launch"],
        "roofline": {"bound": "hbm", "achieved": rl["achieved"], "peak": rl["peak"], "unit": "GB/s",
                     "frac": rl["frac"], "traffic": rl["traffic"]},
        "e2e": {"value": _r(e2e["value"], 0), "unit": "tokens/s", "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
                "d2h_bytes_per_step": e2e["d2h_bytes_per_step"],
                "serial": _r(e2e["serial"]["value"], 0), "eager": _r(e2e["eager"]["value"], 0),
                "prepared": _r(e2e["prepared"]["value"], 0)},
        "gpu_launches": head["kernel_launches"],
        "clocks": {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
    }
    if rows:
        line["rows"] = compact_rows(rows)
    if cpu is not None:
        line["cpu_baseline"] = {"value": _r(cpu["value"], 0), "unit": "tokens/s", "cores": cpu["cores"],
                                "kind": "oracle", "sample": "decode_b64 workload, whole, repeated ~5 s (FP64 C, OpenMP)",
                                "one_core": _r(cpu["single_core"]["value"], 0)}
    return line


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-rows", action="store_true", help="headline only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default=None,
                    choices=["decode_small", "decode_b64", "decode_b256", "decode_b64_steady",
                             "decode_b256_steady", "decode_small_steady", "verify_b64", "resume_b64", "prefill_b4",
                             "verify_b64_steady", "decode_resume_b64_steady"],
                    help="time one workload and print its row (used for profiling captures)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return run_reference(args, rank)

    import torch

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import verify_kda_decode_gb300 as K

    hbm, tfl, tfl_sus, src = peaks()
    flush = Flusher(torch)
    if args.only:
        if args.only == "verify_b64_steady":
            row = bench_verify_steady(torch, K, 8, 4, args.steps, args.warmup, hbm, src)
        elif args.only == "decode_resume_b64_steady":
            row = bench_resume_steady(torch, K, 8, 8, args.steps, args.warmup, hbm, src)
        elif args.only.endswith("_steady"):
            name = args.only[: -len("_steady")]
            row = bench_decode_steady(torch, K, name, 2 if name == "decode_b256" else 8, args.steps, args.warmup, hbm, src)
        elif args.only.startswith("decode"):
            row, _ = bench_decode(torch, K, args.only, args.steps, args.warmup, flush, hbm, src)
        elif args.only == "verify_b64":
            row = bench_verify(torch, K, args.steps, args.warmup, flush, hbm, src)
        elif args.only == "resume_b64":
            row = bench_resume(torch, K, args.steps, args.warmup, flush, hbm, src)
        else:
            row = bench_prefill(torch, K, args.steps, args.warmup, flush, hbm, src, tfl, src)
        print(json.dumps({"only": args.only, "row": row}))
        return 0
    def sync_ranks():
        if dist:
            dist.barrier()
        torch.cuda.synchronize()

    with ClockSampler(local) as clk:
        sync_ranks()
        head = bench_decode_steady(torch, K, HEADLINE, 8, args.steps, args.warmup, hbm, src, sync_ranks)
        rows = {}
        if not args.no_rows:
            rows["decode_b64_cold"], _ = bench_decode(torch, K, HEADLINE, max(3, args.steps // 2), 3, flush, hbm, src)
            rows["decode_b256"] = bench_decode_steady(torch, K, "decode_b256", 2, args.steps, 3, hbm, src)
            rows["decode_b256_cold"], _ = bench_decode(torch, K, "decode_b256", max(3, args.steps // 2), 3, flush, hbm, src)
            rows["decode_small_cold"], _ = bench_decode(torch, K, "decode_small", max(3, args.steps // 2), 3, flush, hbm, src)
            rows["decode_small"] = bench_decode_steady(torch, K, "decode_small", 8, args.steps, 3, hbm, src)
            rows["verify_b64"] = bench_verify(torch, K, args.steps, 3, flush, hbm, src)
            rows["verify_b64_steady"] = bench_verify_steady(torch, K, 8, 4, max(3, args.steps // 2), 3, hbm, src)
            rows["resume_b64"] = bench_resume(torch, K, args.steps, 3, flush, hbm, src)
            rows["decode_resume_b64_steady"] = bench_resume_steady(torch, K, 8, 8, max(3, args.steps // 2), 3, hbm, src)
            rows["prefill_b4"] = bench_prefill(torch, K, max(2, args.steps // 5), 3, flush, hbm, src, tfl, src)
        e2e = bench_e2e(torch, K, args.steps, 3)
    clocks = clk.summary()

    ms_step = max_over_ranks(torch, dist, head["ms_per_step"], "cuda")
    value = job_throughput(head["tokens_per_step"], world, ms_step)
    e2e["ms_per_step"] = max_over_ranks(torch, dist, e2e["ms_per_step"], "cuda")
    e2e["value"] = job_throughput(e2e["tokens_per_step"], world, e2e["ms_per_step"])
    if rank != 0:
        return 0
    detail = {
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded, kda_inputs)",
        "config": {**base_config(), "layer_instances": head["layers"],
                   "launches_per_bench_step": head["launches_per_step"],
                   "timing": "one CUDA graph of 64 steps x 8 layer instances per bench step; CUDA events around the replays",
                   "l2": "inputs larger than L2: 8 x 32 MiB of touched state per step, no flush",
                   "value_definition": "B / device time per decode launch (tokens/s of one KDA mixer step)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "us_per_launch": head["us_per_launch"],
        "roofline": head["roofline"],
        "access_pattern_ceiling": head["access_pattern_ceiling"],
        "e2e": e2e,
        "gpu_launches": head["kernel_launches"],
        "clocks": {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "rows": rows,
    }
    cpu = None
    if not args.no_cpu_baseline:
        cpu = oracle_decode_run()
        cpu["single_core"] = oracle_single_core()
        detail["cpu_baseline"] = cpu
    # every figure, with its description, on stderr; the one JSON line on stdout stays short
    # enough that a log tail of 1.5 KB still holds all of it
    print(json.dumps(detail), file=sys.stderr)
    print(json.dumps(compact_line(args, world, value, ms_step, head, e2e, clocks, rows, cpu)))
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
