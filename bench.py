#!/usr/bin/env python
"""Benchmark: per-window int8 recurrent-state decode for one GDN layer on GB300.

Workload (default): one Gated DeltaNet linear-attention layer shaped like
Qwen3.5-9B's, batch 512 requests x 32 heads = 16,384 head-states of 128 x 128,
W = 16, C = 4, seeded synthetic inputs, initial state from 512 warm-up tokens
with planted outlier lines.

One step = one window of W = 16 decode tokens for every head-state: 15
append-only launches and one fused append+fold launch of ``lq_decode_step``,
so every step of the hot path (decay products, fused dequantize+matvec,
compensator and record terms, the delta-rule correction and the fold) runs once
per head-state per token. The metric is head-tokens/s (head-states x tokens per
second) plus the achieved HBM bandwidth of the dominant kernel against the
measured copy bandwidth.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Rank 0 prints ONE JSON line. Under torchrun rank r decodes its own block of
requests (head-states r*N .. (r+1)*N-1 of the same seeded stream) on its own
GPU: head-states are independent, so this is weak scaling with no collective
on the data path; the timed region is bracketed by barriers and the time is
the maximum over ranks.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "head-tokens/s and achieved HBM GB/s (% of GB300 peak) at batch 32/128/512"
UNIT = "head-tokens/s"
FALLBACK_HBM_GBS = 6800.0
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "k_append_gdn_batch128.md")
PROFILE_STEP = os.path.join(ROOT, "profiles", "k_step_gdn_batch128.md")
CSRC = os.path.join(ROOT, "quantized_linear_attention_gb300", "csrc")


def kernel_sources_sha256():
    """One hash over every CUDA source and header of the library (sorted by name), so a
    profile summary taken on other kernels is recognised as stale."""
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")):
            h.update(name.encode())
            with open(os.path.join(CSRC, name), "rb") as f:
                h.update(f.read())
    return h.hexdigest()


# ----------------------------------------------------------------------------- bytes
def alg_bytes_append(p, C=4, kda=False, D=128, bits=8):
    """Algorithmic bytes one head-state moves in an append at window phase p
    (p records held before the token): every input read once, every output written once."""
    alen = D if kda else 1
    rec = 4 * D + 4 * D + 4 * alen  # k, u, alpha of one record
    reads = D * D * bits // 8 + 4 * D + 4 * D + 4 * C + 4 * C * D  # boundary: codes, sigma, lambda, ids, lines
    reads += p * rec + 4  # buffered records, record count
    reads += 4 * D * 3 + 4 * alen + 4  # q, k, v, alpha, beta
    writes = rec + 4 * D + 4  # new record, o, record count
    return reads + writes


def alg_bytes_fold_extra(C=4, D=128, bits=8):
    """Bytes the fold adds to the append that fills the window: the new boundary."""
    return D * D * bits // 8 + 4 * D + 4 * D + 4 * C + 4 * C * D


def alg_bytes_fp32(kda=False, D=128):
    """Per head-token of the fp32-state baseline: the whole state read and written,
    the token's inputs read, o written."""
    return 2 * 4 * D * D + 4 * D * 3 + 4 * (D if kda else 1) + 4 + 4 * D


def alg_bytes_window(W=16, C=4, kda=False, bits=8):
    """Per head-state per window: W-1 appends and one fused append+fold."""
    return sum(alg_bytes_append(p, C, kda, bits=bits) for p in range(W)) + alg_bytes_fold_extra(C, bits=bits)


# ----------------------------------------------------------------------------- environment
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def shard_offset(wl, rank: int) -> int:
    """First global head-state index of rank ``rank``'s block (N = wl.n_states per rank)."""
    return rank * wl.n_states


def job_value(n_states: int, W: int, steps: int, world: int, t_ms: float) -> float:
    """Whole-job head-tokens/s: every rank decodes n_states x W tokens per step."""
    return world * n_states * W * steps / (t_ms / 1e3)


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Maximum of a float over all ranks (identity when world == 1)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def profile_traffic(n_states, summary=PROFILE_SUMMARY):
    """(DRAM bytes per launch at n_states, note) from a committed ncu summary (the
    dominant kernel's by default), scaled from the captured head-states (traffic
    grows in proportion to them), or (None, why) when there is none or the kernel
    source changed since it was taken."""
    try:
        text = open(summary).read()
    except OSError:
        return None, "no ncu summary committed"
    fields = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("kernel_sources_sha256") != kernel_sources_sha256():
        return None, "kernel changed since the ncu capture"
    try:
        per = float(fields["dram_bytes_per_launch"])
        cap = int(fields["captured_head_states"])
    except (KeyError, ValueError):
        return None, "summary lacks dram_bytes_per_launch / captured_head_states"
    how = "phase-averaged, " if summary == PROFILE_SUMMARY else ""
    return round(per * n_states / cap), f"ncu capture at {cap} head-states, {how}scaled to {n_states}"


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the timed region runs."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=0, period_ms=50):
        self.tmp = tempfile.NamedTemporaryFile(prefix="lq_clocks_", suffix=".csv", delete=False)
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 f"-lms={period_ms}"], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        self.t0 = self.t1 = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.tmp.close()
        try:
            text = open(self.tmp.name).read()
        finally:
            os.unlink(self.tmp.name)
        return self.summarize(text, self.t0, self.t1)

    @staticmethod
    def summarize(text, t0=None, t1=None):
        rows = []
        for rec in csv.reader(io.StringIO(text)):
            if len(rec) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(rec[0].strip().split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(rec[2]), float(rec[3]), [x.strip() for x in rec[5:]]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 is not None and t0 - 1 <= r[0] <= (t1 or r[0]) + 1]
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3][1:5]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "in_timed_region": bool(inside)}


# ----------------------------------------------------------------------------- our arm
def run_config(wl, world):
    """The config object both arms print (the reference arm times the same workload)."""
    return dict(workload_config(wl, 4 * wl.W),
                parallelism=f"dp{world}: {wl.n_states} head-states per rank, disjoint request blocks, no collective")


def host_cpu_model():
    """The host CPU's model name (lscpu), for the CPU-baseline record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return os.uname().machine


def workload_config(wl, pool_tokens):
    return {"workload": wl.name, "n_states": wl.n_states, "batch": wl.requests, "layers": wl.layers,
            "heads": wl.heads, "d_k": wl.dk, "d_v": wl.dv, "W": wl.W, "C": wl.C,
            "decay": "per-key (KDA)" if wl.kda else "scalar (GDN)", "tokens_per_step": wl.W,
            "state_storage": "int8 codes + fp32 scales, compensators, records",
            "l2": f"inputs larger than L2: the state buffer and a {pool_tokens}-token input pool exceed 129 MB; "
                  f"no flush"}


class Pool:
    """A pool of token inputs resident in HBM (or pinned on the host for the end-to-end leg)."""

    def __init__(self, wl, n_tokens, device, pinned=False, on_device=True, state0=0):
        import numpy as np
        import torch

        from quantized_linear_attention_gb300 import workload as wlm

        tk = wlm.tokens(wl, 0, n_tokens, state0, wl.n_states)
        self.n_tokens = n_tokens
        self.host = [torch.from_numpy(np.ascontiguousarray(x)) for x in (tk.q, tk.k, tk.v, tk.alpha, tk.beta)]
        if pinned:
            self.host = [h.pin_memory() for h in self.host]
        self.dev = [h.to(device) for h in self.host] if on_device else None

    def token(self, t):
        t %= self.n_tokens
        return [x[t] for x in self.dev]


def setup_state(wl, device, state0=0, bits=8, comp_fit=0, comp_block=0):
    import torch

    from quantized_linear_attention_gb300 import lq
    from quantized_linear_attention_gb300 import workload as wlm

    cfg = lq.config(window=wl.W, n_comp=wl.C, kda=wl.kda, code_bits=bits, comp_fit=comp_fit, comp_block=comp_block)
    S0, _ = wlm.initial_state(wl, state0, wl.n_states)
    state = lq.alloc_state(cfg, wl.n_states, device)
    lq.state_init(cfg, state, wl.n_states, None if S0 is None else torch.from_numpy(S0).to(device))
    del S0
    return cfg, state


def time_main(wl, args, device, world, rank=0, bits=8, steps=None, comp_fit=0, comp_block=0):
    """Two timed passes over whole windows. The headline pass records one CUDA event
    before and one after its K windows (an event between launches costs about 2 us
    a launch on the stream). The breakdown pass records an event between every two
    launches, for the append and fold-step times."""
    import torch

    from quantized_linear_attention_gb300 import lq

    W, N = wl.W, wl.n_states
    s0 = shard_offset(wl, rank)
    cfg, state = setup_state(wl, device, s0, bits, comp_fit, comp_block)
    pool = Pool(wl, 4 * W, device, state0=s0)
    o = torch.empty((N, wl.dv), dtype=torch.float32, device=device)

    def launch(t):
        q, k, v, a, b = pool.token(t)
        lq.decode_step(cfg, state, N, q, k, v, a, b, o, phase=t % W)

    tok = 0
    for _ in range(args.warmup):
        for _ in range(W):
            launch(tok)
            tok += 1
    torch.cuda.synchronize()
    K = args.steps if steps is None else steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(device.index or 0)
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    sampler.mark_start()
    e0.record()
    for _ in range(K * W):
        launch(tok)
        tok += 1
    e1.record()
    torch.cuda.synchronize()
    sampler.mark_end()
    barrier(world)
    clocks = sampler.stop()
    total_ms = e0.elapsed_time(e1)
    Kb = min(K, 100)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(Kb * W + 1)]
    ev[0].record()
    for i in range(Kb * W):
        launch(tok)
        tok += 1
        ev[i + 1].record()
    torch.cuda.synchronize()
    status, bad = lq.get_status(state)
    if status != lq.OK:
        raise RuntimeError(f"device status {lq.STATUS_NAMES.get(status)} at head-state {bad}")
    if not torch.isfinite(o).all():
        raise RuntimeError("non-finite output")
    d = [ev[i].elapsed_time(ev[i + 1]) for i in range(Kb * W)]
    app = [d[i] for i in range(Kb * W) if i % W != W - 1]
    fold = [d[i] for i in range(Kb * W) if i % W == W - 1]
    del state, pool
    torch.cuda.empty_cache()
    return total_ms, app, fold, clocks


def two_passes(launch, tok, n_head, n_break):
    """Run n_head launches between two CUDA events (the throughput), then n_break
    launches with an event between every two (the per-launch times). Returns
    (total ms of the first pass, per-launch ms of the second, next token)."""
    import torch

    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n_head):
        launch(tok)
        tok += 1
    e1.record()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_break + 1)]
    ev[0].record()
    for i in range(n_break):
        launch(tok)
        tok += 1
        ev[i + 1].record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1), [ev[i].elapsed_time(ev[i + 1]) for i in range(n_break)], tok


def time_staggered(wl, device, steps=50, warmup=3):
    """Head-states at W different window phases: group g (states g*N/W ..) is re-admitted
    by lq_state_init_range before token g, then every token is one lq_decode_step with
    LQ_PHASE_ANY (append, then fold the windows it filled). Returns per-token ms."""
    import torch

    from quantized_linear_attention_gb300 import lq

    W, N = wl.W, wl.n_states
    G = N // W
    cfg, state = setup_state(wl, device)
    pool = Pool(wl, 4 * W, device)
    o = torch.empty((N, wl.dv), dtype=torch.float32, device=device)

    def launch(t):
        q, k, v, a, b = pool.token(t)
        lq.decode_step(cfg, state, N, q, k, v, a, b, o, phase=lq.PHASE_ANY)

    for t in range(W):
        if t > 0:  # a new request in these slots: its state starts from zero
            lq.state_init_range(cfg, state, N, t * G, G if t < W - 1 else N - t * G, None)
        launch(t)
    tok = W
    for _ in range(warmup * W):
        launch(tok)
        tok += 1
    total, d, tok = two_passes(launch, tok, steps * W, min(steps, 20) * W)
    status, bad = lq.get_status(state)
    if status != lq.OK:
        raise RuntimeError(f"device status {lq.STATUS_NAMES.get(status)} at head-state {bad}")
    counts = lq.state_views(cfg, state, N)["counts"]
    phases = torch.bincount(counts.long(), minlength=W).tolist()
    del state, pool
    torch.cuda.empty_cache()
    return total, d, phases


def time_two_record(wl, device, steps=50, warmup=3):
    """Two-record tokens (DeltaProduct with two steps): W/2 lq_decode_step2 calls per
    window at stated phases 0, 2, ..., W-2; the last one also folds (second kernel).
    Sub-step 1 takes generator token 2t, sub-step 2 and the query token 2t+1."""
    import torch

    from quantized_linear_attention_gb300 import lq

    W, N = wl.W, wl.n_states
    per_win = W // 2
    cfg, state = setup_state(wl, device)
    pool = Pool(wl, 4 * W, device)
    o = torch.empty((N, wl.dv), dtype=torch.float32, device=device)

    def launch(t):
        q, k2, v2, _, b2 = pool.token(2 * t + 1)
        _, k1, v1, a, b1 = pool.token(2 * t)
        lq.decode_step2(cfg, state, N, q, k1, v1, b1, k2, v2, b2, a, o, phase=(2 * t) % W)

    tok = 0
    for _ in range(warmup * per_win):
        launch(tok)
        tok += 1
    total, d, tok = two_passes(launch, tok, steps * per_win, min(steps, 20) * per_win)
    status, bad = lq.get_status(state)
    if status != lq.OK:
        raise RuntimeError(f"device status {lq.STATUS_NAMES.get(status)} at head-state {bad}")
    app = [d[i] for i in range(len(d)) if i % per_win != per_win - 1]
    fold = [d[i] for i in range(len(d)) if i % per_win == per_win - 1]
    del state, pool
    torch.cuda.empty_cache()
    return total, app, fold, steps * per_win


def time_rwkv(device, steps=50, warmup=3):
    """RWKV7 tokens at batch 512 (16,384 head-states, per-key decay): W/2
    lq_decode_step_rwkv7 calls per window at stated phases; the last also folds.
    Token t takes decay and erase direction from generator token 2t, the rest
    from token 2t+1 (the erase direction normalized)."""
    import torch

    from quantized_linear_attention_gb300 import lq
    from quantized_linear_attention_gb300 import workload as wlm

    wl = wlm.custom(4000, 16384, 0, kda=True, n_warm=64, plant=True)
    W, N = wl.W, wl.n_states
    per_win = W // 2
    cfg, state = setup_state(wl, device)
    pool = Pool(wl, 4 * W, device)
    kh_pool = [torch.nn.functional.normalize(pool.token(2 * t)[1], dim=-1) for t in range(2 * W)]
    o = torch.empty((N, wl.dv), dtype=torch.float32, device=device)

    def launch(t):
        _, _, _, w, _ = pool.token(2 * t)
        r, k, v, a, _ = pool.token(2 * t + 1)
        lq.decode_step_rwkv7(cfg, state, N, r, w, kh_pool[t % (2 * W)], a, k, v, o, phase=(2 * t) % W)

    tok = 0
    for _ in range(warmup * per_win):
        launch(tok)
        tok += 1
    total, d, tok = two_passes(launch, tok, steps * per_win, min(steps, 20) * per_win)
    status, bad = lq.get_status(state)
    if status != lq.OK:
        raise RuntimeError(f"device status {lq.STATUS_NAMES.get(status)} at head-state {bad}")
    app = [d[i] for i in range(len(d)) if i % per_win != per_win - 1]
    fold = [d[i] for i in range(len(d)) if i % per_win == per_win - 1]
    del state, pool
    torch.cuda.empty_cache()
    return total, app, fold, steps * per_win


def time_graphed(wl, steps, device):
    """Small batches are launch-bound: capture the W-1 appends and the fold step as
    two CUDA graphs per pool window and time their replays."""
    import torch

    from quantized_linear_attention_gb300 import lq

    W, N = wl.W, wl.n_states
    cfg, state = setup_state(wl, device)
    n_pool_windows = 4
    pool = Pool(wl, n_pool_windows * W, device)
    o = torch.empty((N, wl.dv), dtype=torch.float32, device=device)
    graphs = []
    side = torch.cuda.Stream(device)
    for wi in range(n_pool_windows):
        ga, gf = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(ga, stream=side, capture_error_mode="relaxed"):
            for p in range(W - 1):
                q, k, v, a, b = pool.token(wi * W + p)
                lq.decode_step(cfg, state, N, q, k, v, a, b, o, phase=p)
        with torch.cuda.graph(gf, stream=side, capture_error_mode="relaxed"):
            q, k, v, a, b = pool.token(wi * W + W - 1)
            lq.decode_step(cfg, state, N, q, k, v, a, b, o, phase=W - 1)
        graphs.append((ga, gf))
    for i in range(3):
        ga, gf = graphs[i % n_pool_windows]
        ga.replay()
        gf.replay()
    torch.cuda.synchronize()
    e = [torch.cuda.Event(enable_timing=True) for _ in range(2 * steps + 1)]
    e[0].record()
    for i in range(steps):
        ga, gf = graphs[i % n_pool_windows]
        ga.replay()
        e[2 * i + 1].record()
        gf.replay()
        e[2 * i + 2].record()
    torch.cuda.synchronize()
    status, _ = lq.get_status(state)
    if status != lq.OK:
        raise RuntimeError(f"device status {lq.STATUS_NAMES.get(status)}")
    total = e[0].elapsed_time(e[-1])
    app = statistics.median(e[2 * i].elapsed_time(e[2 * i + 1]) for i in range(steps)) / (W - 1)
    fold = statistics.median(e[2 * i + 1].elapsed_time(e[2 * i + 2]) for i in range(steps))
    del graphs, state, pool
    torch.cuda.empty_cache()
    return total, app, fold


def time_fp32(wl, device, tokens=48, warmup=4):
    """The fp32-state baseline (lq_fp32_decode_step) on the same head-states and
    tokens: mean time of one decode token over `tokens` launches."""
    import torch

    from quantized_linear_attention_gb300 import lq
    from quantized_linear_attention_gb300 import workload as wlm

    N = wl.n_states
    cfg = lq.config(kda=wl.kda)
    S0, _ = wlm.initial_state(wl)
    S = torch.from_numpy(S0).to(device) if S0 is not None else torch.zeros((N, wl.dv, wl.dk), device=device)
    del S0
    pool = Pool(wl, 16, device)
    o = torch.empty((N, wl.dv), dtype=torch.float32, device=device)

    def launch(t):
        q, k, v, a, b = pool.token(t)
        lq.fp32_decode_step(cfg, S, N, q, k, v, a, b, o)

    for t in range(warmup):
        launch(t)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for t in range(tokens):
        launch(t)
    e1.record()
    torch.cuda.synchronize()
    if not torch.isfinite(o).all():
        raise RuntimeError("non-finite fp32 baseline output")
    ms = e0.elapsed_time(e1) / tokens
    del S, pool, o
    torch.cuda.empty_cache()
    return ms


def time_e2e(wl, steps, device, ring=8):
    """End to end through the C ABI with host buffers: every token's inputs are
    copied from pinned host memory and every token's output is copied back, all
    inside the timed region. The copies run on two side streams and overlap the
    decode calls, as a serving loop would: host-to-device for token t+1 while
    token t decodes, device-to-host of each output once its token is done
    (a ring of `ring` token slots on the device, ordered by events). A token's
    inputs take longer to copy (about 125 us at 205 GB/s) than its append takes
    to run (90 us), so the copies must run ahead through the window's fold
    token: 8 slots let them, 4 did not."""
    import torch

    from quantized_linear_attention_gb300 import lq

    W, N = wl.W, wl.n_states
    cfg, state = setup_state(wl, device)
    n_pool = 2 * W
    pool = Pool(wl, n_pool, device, pinned=True, on_device=False)
    stage = [[torch.empty(tuple(h.shape[1:]), dtype=h.dtype, device=device) for h in pool.host] for _ in range(ring)]
    o_dev = [torch.empty((N, wl.dv), dtype=torch.float32, device=device) for _ in range(ring)]
    o_host = torch.empty((W, N, wl.dv), dtype=torch.float32).pin_memory()
    h2d = W * sum(x.numel() * x.element_size() for x in stage[0])
    d2h = o_host.numel() * o_host.element_size()
    comp = torch.cuda.current_stream(device)
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev_in = [torch.cuda.Event() for _ in range(ring)]
    ev_done = [torch.cuda.Event() for _ in range(ring)]
    ev_out = [torch.cuda.Event() for _ in range(ring)]
    used = [False] * ring

    def load(g):
        slot = g % ring
        with torch.cuda.stream(s_in):
            if used[slot]:
                s_in.wait_event(ev_done[slot])  # the slot's previous inputs have been consumed
            for x, h in zip(stage[slot], pool.host):
                x.copy_(h[g % n_pool], non_blocking=True)
            ev_in[slot].record(s_in)

    def decode(g):
        slot = g % ring
        comp.wait_event(ev_in[slot])
        if used[slot]:
            comp.wait_event(ev_out[slot])  # the slot's previous output has left the device
        x = stage[slot]
        lq.decode_step(cfg, state, N, x[0], x[1], x[2], x[3], x[4], o_dev[slot], phase=g % W)
        ev_done[slot].record(comp)
        used[slot] = True
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[slot])
            o_host[g % W].copy_(o_dev[slot], non_blocking=True)
            ev_out[slot].record(s_out)

    def run(g0, n_tok):
        for g in range(g0, min(g0 + ring - 1, g0 + n_tok)):
            load(g)
        for g in range(g0, g0 + n_tok):
            if g + ring - 1 < g0 + n_tok:
                load(g + ring - 1)
            decode(g)

    run(0, 3 * W)  # warm-up windows
    torch.cuda.synchronize()
    e0, e1, e_end = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    e0.record(comp)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    run(3 * W, steps * W)
    e_end.record(s_out)
    comp.wait_event(e_end)
    e1.record(comp)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    status, _ = lq.get_status(state)
    if status != lq.OK:
        raise RuntimeError(f"device status {lq.STATUS_NAMES.get(status)}")
    del state, stage, o_dev
    torch.cuda.empty_cache()
    return ms, h2d, d2h


def cpu_baseline(wl, budget_s=12.0):
    """The oracle as it stands, on all host cores, over a bounded sample: M
    head-states x one window (16 tokens, fold included)."""
    import oracle
    from quantized_linear_attention_gb300 import workload as wlm

    cores = os.cpu_count() or 1
    W = wl.W

    def run(M, threads):
        S0, _ = wlm.initial_state(wl, 0, M)
        tk = wlm.tokens(wl, 0, W, 0, M)
        st = oracle.OracleState(M, W=W, C=wl.C, decay_per_key=wl.kda)
        st.init(S0)
        t0 = time.perf_counter()
        st.run(tk.q, tk.k, tk.v, tk.alpha, tk.beta, nthreads=threads, want_o=True)
        return time.perf_counter() - t0

    m0 = min(wl.n_states, max(cores, 32))
    rate = m0 * W / run(m0, cores)
    M = int(min(wl.n_states, max(m0, rate * budget_s / W)))
    dt = run(M, cores)
    m1 = min(wl.n_states, 16)
    rate1 = m1 * W / run(m1, 1)
    M1 = int(min(wl.n_states, max(m1, rate1 * budget_s / 3 / W)))
    dt1 = run(M1, 1)
    return {"value": round(M * W / dt, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
            "single_core": round(M1 * W / dt1, 1), "host_cpu": f"{host_cpu_model()} ({os.uname().machine})",
            "sample": f"{M} (1 core: {M1}) of {wl.n_states} head-states x {W} tokens (one window, fold included) "
                      f"of {wl.name}; {dt:.1f} s on {cores} threads, {dt1:.1f} s on 1"}


def run_ours(args):
    import torch

    from quantized_linear_attention_gb300 import lq
    from quantized_linear_attention_gb300 import workload as wlm

    rank, world, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=device)
    lq.load()
    wl = wlm.WORKLOADS[args.workload]
    W, N, K = wl.W, wl.n_states, args.steps
    total_ms, app, fold, clocks = time_main(wl, args, device, world, rank)
    t_ms = max_over_ranks(total_ms, world, device)
    value = job_value(N, W, K, world, t_ms)

    peaks, peak_kind = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    app_bytes = N * statistics.mean(alg_bytes_append(p, wl.C, wl.kda) for p in range(W - 1))
    app_ms = statistics.mean(app)
    fold_ms = statistics.mean(fold)
    achieved = app_bytes / (app_ms / 1e3) / 1e9
    traffic, traffic_note = profile_traffic(N)
    fold_bytes = N * (alg_bytes_append(W - 1, wl.C, wl.kda) + alg_bytes_fold_extra(wl.C))
    win_bytes = N * alg_bytes_window(W, wl.C, wl.kda)
    step_traffic, _ = profile_traffic(N, PROFILE_STEP)
    win_dram = None
    if traffic is not None and step_traffic is not None:  # 15 appends (phase-averaged) and the fold step
        win_dram = round(((W - 1) * traffic + step_traffic) / N / W, 1)
    win_gbs = win_bytes / (t_ms / K / 1e3) / 1e9
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(t_ms / K, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": run_config(wl, world),
        "roofline": {"bound": "hbm", "kernel": "k_append (append-only decode step, phases 0..14)",
                     "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "peak_kind": f"{peak_kind} hbm_gbs (copy)",
                     "traffic": traffic, "traffic_note": traffic_note,
                     "alg_bytes_per_launch": round(app_bytes), "launch_ms": round(app_ms, 5)},
        "fold_step": {"kernel": "k_step (append + fold, phase 15)", "launch_ms": round(fold_ms, 5),
                      "alg_bytes_per_launch": round(fold_bytes),
                      "achieved_gbs": round(fold_bytes / (fold_ms / 1e3) / 1e9, 1),
                      "fold_cost_per_token_ms": round((fold_ms - app_ms) / W, 5),
                      "amortized_below_one_append": (fold_ms - app_ms) / W < app_ms},
        "window": {"alg_bytes": win_bytes, "achieved_gbs": round(win_gbs, 1), "frac": round(win_gbs / hbm, 4),
                   "alg_bytes_per_head_token": round(win_bytes / N / W, 1),
                   "ncu_dram_bytes_per_head_token": win_dram,
                   "int8_state_minimum_per_head_token": 128 * 128 + 128 * 128 // W,
                   "fp32_state_per_head_token": alg_bytes_fp32(wl.kda)},
        "gpu_launches": K * W,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_sweep:
        sweep = {}
        for wid in (2, 3):
            swl = wlm.WORKLOADS[wid]
            total, a_ms, f_ms = time_graphed(swl, args.sweep_steps, device)
            wb = swl.n_states * alg_bytes_window(swl.W, swl.C, swl.kda)
            gbs = wb / (total / args.sweep_steps / 1e3) / 1e9
            sweep[f"batch{swl.requests}"] = {
                "head_tokens_per_s": round(swl.n_states * swl.W * args.sweep_steps / (total / 1e3), 1),
                "append_step_us": round(a_ms * 1e3, 2), "fold_step_us": round(f_ms * 1e3, 2),
                "window_gbs": round(gbs, 1), "window_frac": round(gbs / hbm, 4), "note": "graph; L2 may hold it"}
        sweep[f"batch{wl.requests}"] = {
            "head_tokens_per_s": round(value / world, 1), "append_step_us": round(app_ms * 1e3, 2),
            "fold_step_us": round(fold_ms * 1e3, 2), "window_gbs": round(win_gbs, 1),
            "window_frac": round(win_gbs / hbm, 4)}
        result["batches"] = sweep
    if rank == 0 and not args.no_stagger:
        s_total, s_d, phases = time_staggered(wl, device)
        s_sorted = sorted(s_d)
        s_n = 50 * W
        result["staggered"] = {
            "note": f"{W} groups of {N // W} head-states, group g re-admitted from a zero state before token g "
                    "(lq_state_init_range), then "
                    "lq_decode_step with LQ_PHASE_ANY: each token appends every head-state, lists the windows it "
                    f"fills and folds them (1/{W} of the head-states); 50 timed windows, 2 launches per token; "
                    "max and p50 from 20 more windows with an event between tokens",
            "head_tokens_per_s": round(N * s_n / (s_total / 1e3), 1),
            "step_us_mean": round(1e3 * s_total / s_n, 2), "step_us_max": round(1e3 * s_sorted[-1], 2),
            "step_us_p50": round(1e3 * s_sorted[len(s_d) // 2], 2),
            "in_phase_step_us_max": round(1e3 * max(fold), 2),
            "in_phase_step_us_mean": round(1e3 * t_ms / K / W, 2),
            "head_states_per_phase_after": phases}
    if rank == 0 and not args.no_two:
        t_total, t_app, t_fold, n_tok = time_two_record(wl, device)
        result["two_record"] = {
            "note": f"two-record tokens (DeltaProduct with two steps, lq_decode_step2): {W // 2} tokens per "
                    f"{W}-record window, one kernel per token reads the boundary once; the last token of a window "
                    "adds the list fold; 50 timed windows",
            "head_tokens_per_s": round(N * n_tok / (t_total / 1e3), 1),
            "token_us_mean": round(1e3 * t_total / n_tok, 2),
            "append2_us": round(1e3 * statistics.mean(t_app), 2),
            "fold_token_us": round(1e3 * statistics.mean(t_fold), 2),
            "two_one_record_steps_us": round(2e3 * t_ms / K / W, 2)}
    if rank == 0 and not args.no_two:
        r_total, r_app, r_fold, n_tok = time_rwkv(device)
        result["rwkv7"] = {
            "note": "RWKV7 tokens (lq_decode_step_rwkv7: an erase record and a pure-write record, one kernel per "
                    f"token) on {N} head-states with per-key decay; {W // 2} tokens per {W}-record window, the "
                    "last one adds the list fold; 50 timed windows",
            "head_tokens_per_s": round(N * n_tok / (r_total / 1e3), 1),
            "token_us_mean": round(1e3 * r_total / n_tok, 2),
            "append_us": round(1e3 * statistics.mean(r_app), 2),
            "fold_token_us": round(1e3 * statistics.mean(r_fold), 2)}
    if rank == 0 and not args.no_kda:
        kwl = wlm.WORKLOADS[5]
        k_total, k_app, k_fold, _ = time_main(kwl, args, device, 1, 0, steps=20)
        kN, kW = kwl.n_states, kwl.W
        kb = kN * alg_bytes_window(kW, kwl.C, True)
        k_app_bytes = kN * statistics.mean(alg_bytes_append(p, kwl.C, True) for p in range(kW - 1))
        k_app_ms = statistics.mean(k_app)
        result["kda_config5"] = {
            "note": f"{kwl.name}: {kN} head-states with per-key decay, Student-t(3) values; 20 timed windows",
            "head_tokens_per_s": round(kN * kW * 20 / (k_total / 1e3), 1),
            "append_step_us": round(k_app_ms * 1e3, 2), "fold_step_us": round(statistics.mean(k_fold) * 1e3, 2),
            "alg_bytes_per_head_token": round(kb / kN / kW, 1),
            "window_gbs": round(kb / (k_total / 20 / 1e3) / 1e9, 1),
            "window_frac": round(kb / (k_total / 20 / 1e3) / 1e9 / hbm, 4),
            "append_gbs": round(k_app_bytes / (k_app_ms / 1e3) / 1e9, 1),
            "append_frac": round(k_app_bytes / (k_app_ms / 1e3) / 1e9 / hbm, 4)}
    for bits in (6, 4):
        if rank != 0 or args.no_bits4:
            break
        b_total, b_app, b_fold, _ = time_main(wl, args, device, 1, 0, bits=bits, steps=100)
        b_app_ms, b_fold_ms, b_win_ms = statistics.mean(b_app), statistics.mean(b_fold), b_total / 100
        bw = N * alg_bytes_window(W, wl.C, wl.kda, bits=bits)
        b_app_bytes = N * statistics.mean(alg_bytes_append(p, wl.C, wl.kda, bits=bits) for p in range(W - 1))
        packing = "two per byte" if bits == 4 else "four per three bytes: a nibble plane and a 2-bit plane"
        result[f"code_bits_{bits}"] = {
            "note": f"the same workload with {bits}-bit codes ({packing}); 100 timed windows",
            "head_tokens_per_s": round(N * W / (b_win_ms / 1e3), 1), "append_step_us": round(b_app_ms * 1e3, 2),
            "fold_step_us": round(b_fold_ms * 1e3, 2), "alg_bytes_per_head_token": round(bw / N / W, 1),
            "window_gbs": round(bw / (b_win_ms / 1e3) / 1e9, 1), "window_frac": round(bw / (b_win_ms / 1e3) / 1e9 / hbm, 4),
            "append_gbs": round(b_app_bytes / (b_app_ms / 1e3) / 1e9, 1),
            "append_frac": round(b_app_bytes / (b_app_ms / 1e3) / 1e9 / hbm, 4)}
    if rank == 0 and not args.no_fit:
        for name, sweeps, block, note in (
                ("comp_fit_8", 8, 0, "compensators as rank-one factors fitted one at a time by 8 power-iteration "
                                     "sweeps from the longest row (the other reading of Compensator Tokens)"),
                ("comp_block_4", 4, 1, "the same factors fitted together as a block by 4 sweeps of subspace "
                                       "iteration, each fold starting from the previous window's factors")):
            f_total, f_app, f_fold, _ = time_main(wl, args, device, 1, 0, steps=50, comp_fit=sweeps, comp_block=block)
            result[name] = {
                "note": note + "; 50 timed windows",
                "head_tokens_per_s": round(N * W / (f_total / 50 / 1e3), 1),
                "append_step_us": round(statistics.mean(f_app) * 1e3, 2),
                "fold_step_us": round(statistics.mean(f_fold) * 1e3, 2)}
    if rank == 0 and not args.no_fp32:
        f_ms = time_fp32(wl, device)
        fb = N * alg_bytes_fp32(wl.kda)
        int8_token_ms = t_ms / K / W
        result["fp32_baseline"] = {
            "kernel": "k_fp32_step (whole fp32 state, plain delta rule, one token per launch)",
            "launch_ms": round(f_ms, 5), "head_tokens_per_s": round(N / (f_ms / 1e3), 1),
            "alg_bytes_per_launch": fb, "achieved_gbs": round(fb / (f_ms / 1e3) / 1e9, 1),
            "frac": round(fb / (f_ms / 1e3) / 1e9 / hbm, 4),
            "int8_speedup_per_token": round(f_ms / int8_token_ms, 3),
            "note": "same head-states, initial states and tokens as the int8 path; speedup = fp32 ms per token / "
                    "int8 window ms / 16"}
    if rank == 0 and args.e2e_steps > 0:
        ms, h2d, d2h = time_e2e(wl, args.e2e_steps, device)
        result["e2e"] = {"value": round(N * W * args.e2e_steps / (ms / 1e3), 1), "unit": UNIT,
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                         "note": "per token: pinned host inputs -> device and the output -> host on two side "
                                 "streams, overlapping the lq_decode_step calls (a ring of 8 token slots)"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl)
    if rank == 0:
        # the summaries the metric names (batches 32/128/512, the fold step, the
        # window) and the baselines go last, where a truncated tail still shows them
        last = ("window", "fold_step", "batches", "e2e", "cpu_baseline", "gpu_launches", "clocks")
        ordered = {k: v for k, v in result.items() if k not in last}
        ordered.update((k, result[k]) for k in last if k in result)
        print(json.dumps(ordered), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


# ----------------------------------------------------------------------------- reference arm
def run_reference(args):
    """The oracle as the reference arm, on this machine's host cores (rank 0 only)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from quantized_linear_attention_gb300 import workload as wlm

    wl = wlm.WORKLOADS[args.workload]
    W = wl.W
    cores = os.cpu_count() or 1
    budget = float(os.environ.get("LQ_REFERENCE_BUDGET_S", "120"))
    m0 = min(wl.n_states, max(cores, 16))
    S0, _ = wlm.initial_state(wl, 0, m0)
    tk = wlm.tokens(wl, 0, W, 0, m0)
    st = oracle.OracleState(m0, W=W, C=wl.C, decay_per_key=wl.kda)
    st.init(S0)
    t0 = time.perf_counter()
    st.run(tk.q, tk.k, tk.v, tk.alpha, tk.beta, nthreads=cores)
    rate = m0 * W / (time.perf_counter() - t0)
    per_step_s = budget / max(args.steps + args.warmup, 1)
    M = int(min(wl.n_states, max(cores, rate * per_step_s / W)))
    S0, _ = wlm.initial_state(wl, 0, M)
    pool = wlm.tokens(wl, 0, 2 * W, 0, M)
    st = oracle.OracleState(M, W=W, C=wl.C, decay_per_key=wl.kda)
    st.init(S0)

    def step(i):
        sl = slice((i % 2) * W, (i % 2 + 1) * W)
        st.run(pool.q[sl], pool.k[sl], pool.v[sl], pool.alpha[sl], pool.beta[sl], nthreads=cores)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    value = M * W * args.steps / dt
    sample = f"{M} of {wl.n_states} head-states x {W} tokens per step (one window, fold included) of {wl.name}"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / max(args.steps, 1) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": run_config(wl, world),
        "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "host_cpu": f"{host_cpu_model()} ({os.uname().machine})", "sample": sample},
        "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400, help="timed windows (16 decode tokens each)")
    ap.add_argument("--warmup", type=int, default=5, help="untimed warm-up windows")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", type=int, default=4, help="workload id (4 = batch 512)")
    ap.add_argument("--sweep-steps", type=int, default=200)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fp32", action="store_true", help="skip the fp32-state baseline kernel")
    ap.add_argument("--no-bits4", action="store_true", help="skip the 6- and 4-bit-code runs of the same workload")
    ap.add_argument("--no-fit", action="store_true", help="skip the fitted-factor compensator run")
    ap.add_argument("--no-stagger", action="store_true", help="skip the mixed-window-phase run")
    ap.add_argument("--no-two", action="store_true", help="skip the two-record-token and RWKV7 runs")
    ap.add_argument("--no-kda", action="store_true", help="skip the per-key-decay (KDA) workload run")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
