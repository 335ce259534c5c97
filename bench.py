#!/usr/bin/env python
"""Benchmark of the SepLLM attention hot path on B300.

One timed step = sep_build_index + sep_attn_fwd + sep_attn_bwd on the
Pythia-160M-shaped training workload (B8 H12 L2048 d64, a=4, n=128,
separator probability 0.10), replayed from a CUDA graph with L2 flushed
(a 256 MiB write, then a 256 MiB read) between steps and device time taken from CUDA events.
Also measured, in sub-objects of the same JSON line: streaming decode on the
Llama-3-8B-shaped workload (64 sequences, c = 324, 2048 prompt tokens then
4096 decode steps; tokens/s against HBM bandwidth) and forward-only prefill
at L = 8192 and L = 65536.

FLOPs are counted over visited (unmasked) pairs only: 4 d per pair for the
forward, 10 d per pair for the backward, per q head.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 the script runs under torch.distributed.run, one rank per GPU;
every rank processes its own batch (weak scaling, no collective on the data
path) and rank 0 prints the line with the max time over ranks.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from separator_token_kv_sep_b300 import synth  # noqa: E402

METRIC = "Sep-Attention fwd+bwd TFLOP/s (visited pairs) & decode tok/s; % roofline"
# DRAM bytes per launch from one ncu capture of each kernel version at the
# bench's training workload; a kernel changed since its capture has no entry
# (its "traffic" is reported as null)
DRAM_TRAFFIC_BYTES = {"bwd_kv": 144.573952e6 + 20.909312e6, "fwd_attn": 81.934592e6 + 4.598016e6,
                      "bwd_dq": 118.828544e6 + 15.080448e6}
DECODE_DRAM_TRAFFIC_BYTES = 81.522944e6 + 1.996544e6
L2_FLUSH_BYTES = 256 << 20


def torch_amax(t):
    import torch
    return torch.amax(t)


class L2Flush:
    """Evicts L2 between timed steps: writes one 256 MiB buffer (twice the
    126 MB L2), then reads another 256 MiB buffer, so the lines left in L2
    are clean and the write-back of the flush's dirty lines happens here,
    not inside the next timed step."""

    def __init__(self, device):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device)

    def __call__(self):
        self.w.zero_()
        torch_amax(self.r)  # a plain read (int32 max: no widening copy)


L2_NOTE = "flushed between steps (256 MiB write, then a 256 MiB read)"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


# ---------------------------------------------------------------------------
# Work accounting (bookkeeping only; the computation itself runs in the
# library's kernels)
# ---------------------------------------------------------------------------

def visited_pairs_per_head(ids: np.ndarray, a: int, n: int) -> int:
    """Sum over the batch of the unmasked pairs of one head: row i sees the
    keep tokens before its window start W(i) plus the whole window [W(i), i]."""
    keep = np.isin(ids, synth.SEP_IDS) | (np.arange(ids.shape[1]) < a)[None, :]
    kp = np.concatenate([np.zeros((ids.shape[0], 1), np.int64), np.cumsum(keep, axis=1)], axis=1)
    i = np.arange(ids.shape[1])
    W = np.maximum(0, i - n + 1)
    return int((kp[:, W] + (i - W + 1)[None, :]).sum())


def visited_pairs_keep(keep: np.ndarray, n: int) -> int:
    """visited_pairs_per_head for an explicit keep mask [B, L]."""
    kp = np.concatenate([np.zeros((keep.shape[0], 1), np.int64), np.cumsum(keep, axis=1)], axis=1)
    i = np.arange(keep.shape[1])
    W = np.maximum(0, i - n + 1)
    return int((kp[:, W] + (i - W + 1)[None, :]).sum())


def gathered_band_pairs_per_head(ids: np.ndarray, a: int, n: int, bm: int):
    """Split of the visited pairs of one head (summed over the batch) between
    the two key sources of a 128-row query tile: keep tokens gathered from
    before the tile's first window start, and the dense band after it."""
    keep = np.isin(ids, synth.SEP_IDS) | (np.arange(ids.shape[1]) < a)[None, :]
    kp = np.concatenate([np.zeros((ids.shape[0], 1), np.int64), np.cumsum(keep, axis=1)], axis=1)
    L = ids.shape[1]
    i = np.arange(L)
    W0 = np.maximum(0, (i // bm) * bm - n + 1)
    gathered = int(kp[:, W0].sum())
    return gathered, visited_pairs_per_head(ids, a, n) - gathered


def decode_cache_lengths(sep: np.ndarray, a: int, s: int, w: int, c: int) -> np.ndarray:
    """Entries each sequence's cache holds after each step (new token
    included), from counts alone: tokens [a, cp) have been through
    compression, the separator block keeps the last <= s separators among
    them, and [max(a, cp), t] is the past + local window."""
    T, S = sep.shape
    csum = np.concatenate([np.zeros((1, S), np.int64), np.cumsum(sep, axis=0)], axis=0)
    cp = np.full(S, a, np.int64)
    out = np.zeros((T, S), np.int64)
    cols = np.arange(S)
    for t in range(T):
        if t >= a:
            n_sep = np.minimum(s, csum[cp, cols] - csum[a, cols])
            total = a + n_sep + (t - cp)
            cp = np.where(total == c, np.maximum(cp, t - w), cp)
            n_sep = np.minimum(s, csum[cp, cols] - csum[a, cols])
            out[t] = a + n_sep + (t + 1 - np.maximum(a, cp))
        else:
            out[t] = t + 1
    return out


# ---------------------------------------------------------------------------
# Clock sampling during the timed regions
# ---------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4)
                          if r[5 + k].lower().startswith("active")})
        loaded = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

def run_ours(args, rank, world, device):
    import torch
    from separator_token_kv_sep_b300 import api

    torch.cuda.set_device(device)
    peaks = load_peaks()
    flush = L2Flush(device)
    stream = torch.cuda.current_stream()

    # ---------------------------------------------------------- train step
    cfg = synth.PYTHIA_TRAIN_N128
    q_np, k_np, v_np, do_np, ids_np = synth.prefill_inputs(cfg, seed=shard_seed(cfg.seed, rank))
    bf = torch.bfloat16
    q = torch.from_numpy(q_np).to(device, bf)
    k = torch.from_numpy(k_np).to(device, bf)
    v = torch.from_numpy(v_np).to(device, bf)
    dout = torch.from_numpy(do_np).to(device, bf)
    ids = torch.from_numpy(ids_np).to(device)
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    pairs = visited_pairs_per_head(ids_np, cfg.a, cfg.n)
    fwd_flops = 4.0 * d * pairs * Hq
    bwd_flops = 10.0 * d * pairs * Hq
    idx_buf = torch.empty(api.sep_index_bytes(B, L), dtype=torch.uint8, device=device)
    ws_f = torch.empty(api.sep_attn_workspace_bytes(B, Hq, Hkv, L, d, api.SEP_BF16, False),
                       dtype=torch.uint8, device=device)
    ws_b = torch.empty(api.sep_attn_workspace_bytes(B, Hq, Hkv, L, d, api.SEP_BF16, True),
                       dtype=torch.uint8, device=device)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, L), dtype=torch.float32, device=device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    # step boundaries, and the per-kernel marks the library records through
    # sep_profile_events (fwd: gather | attention; bwd: prep | dK/dV | dQ
    # with the keep-row dK/dV writes)
    Ev = lambda: torch.cuda.Event(enable_timing=True, external=True)  # noqa: E731
    step_ev = [Ev(), Ev()]
    fwd_ev = [Ev() for _ in range(3)]
    bwd_ev = [Ev() for _ in range(4)]
    for e in step_ev + fwd_ev + bwd_ev:  # create the CUDA events outside the capture
        e.record()
    torch.cuda.synchronize()

    def train_step(mark=False):
        if mark:
            step_ev[0].record()
        api.sep_build_index(ids, synth.SEP_IDS, cfg.a, cfg.n, index_buf=idx_buf)
        if mark:
            api.sep_profile_events(fwd_ev)
        api.sep_attn_fwd(idx_buf, q, k, v, o=o, lse=lse, ws=ws_f)
        if mark:
            api.sep_profile_events(bwd_ev)
        api.sep_attn_bwd(idx_buf, q, k, v, o, lse, dout, dq=dq, dk=dk, dv=dv, ws=ws_b)
        if mark:
            api.sep_profile_events([])
            step_ev[1].record()

    for _ in range(2):
        train_step()
    torch.cuda.synchronize()
    assert api.sep_get_device_status() == 0
    # the timed graph holds the step's launches only; a second graph with the
    # per-kernel marks gives the breakdown (event nodes between the kernels
    # would lengthen the timed step)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        train_step()
    graph_m = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_m):
        train_step(mark=True)
    for _ in range(max(3, args.warmup)):
        flush()
        graph.replay()
        flush()
        graph_m.replay()
    torch.cuda.synchronize()

    kern_names = ["index", "fwd_gather", "fwd_attn", "bwd_prep", "bwd_kv", "bwd_dq"]
    marks = [step_ev[0], fwd_ev[0], fwd_ev[1], fwd_ev[2], bwd_ev[0], bwd_ev[1], bwd_ev[2],
             bwd_ev[3]]
    # index: step start -> fwd gather; fwd attn end -> bwd prep is launch glue
    spans = {"index": (0, 1), "fwd_gather": (1, 2), "fwd_attn": (2, 3), "bwd_prep": (4, 5),
             "bwd_kv": (5, 6), "bwd_dq": (6, 7)}
    sampler = ClockSampler(device.index if device.index is not None else 0)
    t_step = []
    t_kern = {n: [] for n in kern_names}
    with sampler:
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream()
        for _ in range(args.steps):
            flush()
            step_ev[0].record(stream)
            graph.replay()
            step_ev[1].record(stream)
            torch.cuda.synchronize()
            t_step.append(step_ev[0].elapsed_time(step_ev[1]))
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        total_ms = sum(t_step)
        total_ms = max_over_ranks(total_ms, world)
        t_marked = []
        for _ in range(args.steps):  # the breakdown, outside the timed steps
            flush()
            graph_m.replay()
            torch.cuda.synchronize()
            t_marked.append(step_ev[0].elapsed_time(step_ev[1]))
            for n in kern_names:
                a_, b_ = spans[n]
                t_kern[n].append(marks[a_].elapsed_time(marks[b_]))
        decode = run_decode(args, rank, device, flush, peaks) if args.only == "all" else None
        prefill = run_prefill(args, rank, device, flush, peaks) if args.only == "all" else None
        variants = run_variants(args, rank, device, flush, peaks) if args.only == "all" else None
        index_scaling = (run_index_scaling(args, rank, device, flush)
                         if args.only == "all" else None)
    assert api.sep_get_device_status() == 0
    clocks = sampler.summary()

    ms_per_step = total_ms / args.steps
    value = aggregate_value(fwd_flops + bwd_flops, world, args.steps, total_ms)
    mean = lambda xs: sum(xs) / len(xs)  # noqa: E731
    kern_ms = {n: mean(t_kern[n]) for n in kern_names}
    fwd_ms = kern_ms["fwd_gather"] + kern_ms["fwd_attn"]
    bwd_ms = sum(kern_ms[n] for n in ("bwd_prep", "bwd_kv", "bwd_dq"))
    fwd_tf = fwd_flops / (fwd_ms * 1e-3) / 1e12
    bwd_tf = bwd_flops / (bwd_ms * 1e-3) / 1e12
    # Algorithmic FLOPs of each tensor-core kernel over the visited pairs it
    # owns: attention forward 4d per pair; key-major dK/dV 8d per pair
    # (S and dP recomputed, dV, dK); query-major dQ 6d per pair (S, dP, dQ).
    kern_flops = {"fwd_attn": 4.0 * d * pairs * Hq, "bwd_kv": 8.0 * d * pairs * Hq,
                  "bwd_dq": 6.0 * d * pairs * Hq}
    dom = max(kern_flops, key=lambda n: kern_ms[n])
    dom_tf = kern_flops[dom] / (kern_ms[dom] * 1e-3) / 1e12
    kernels = {n: {"ms": round(kern_ms[n], 5)} for n in kern_names}
    for n, fl in kern_flops.items():
        kernels[n]["tflops"] = round(fl / (kern_ms[n] * 1e-3) / 1e12, 2)
        kernels[n]["gflop"] = round(fl / 1e9, 3)

    # ------------------------------------------------------------ e2e
    e2e = run_e2e(api, cfg, q_np, k_np, v_np, do_np, ids_np, device, args, fwd_flops + bwd_flops,
                  world) if args.only == "all" else None

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; separator ids 1..9 stand in for . , ? ! ; : space tab newline)",
        "config": {"workload": "pythia160m_train_step " + cfg.describe() +
                   " = sep_build_index + sep_attn_fwd + sep_attn_bwd (CUDA graph replay)",
                   "visited_pairs_per_head": pairs, "visited_over_causal":
                       round(pairs / (B * L * (L + 1) / 2), 4),
                   "l2": L2_NOTE, "parallelism": f"replicas x{world}"},
        "ms_per_step_with_marks": round(sum(t_marked) / len(t_marked), 5),
        "phases_ms": {"fwd": round(fwd_ms, 5), "bwd": round(bwd_ms, 5),
                      "fwd_tflops": round(fwd_tf, 2), "bwd_tflops": round(bwd_tf, 2)},
        "kernels": kernels,
        "roofline": {
            "bound": "tensor", "kernel": dom,
            "achieved": round(dom_tf, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": round(dom_tf / peaks["bf16_tflops"], 4),
            "frac_of_sustained": round(dom_tf / peaks["bf16_tflops_sustained"], 4)
            if peaks.get("bf16_tflops_sustained") else None,
            "peak_source": peaks["source"] + " (burst bf16; of measured)",
            "timing": "CUDA events recorded around the kernel inside a replay of the same "
                      "step captured with per-kernel event nodes",
            "traffic": DRAM_TRAFFIC_BYTES.get(dom),
            "traffic_unit": "bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum, "
                            "one ncu capture of this kernel at this workload)"},
        "e2e": e2e,
        "clocks": clocks,
        # index, keep gather, forward; prep, dK/dV, dQ (with the keep rows)
        "gpu_launches": 6 * args.steps,
        "decode": decode,
        "prefill": prefill,
        "mask_variants": variants,
        "index_scaling": index_scaling,
    }
    if rank == 0 and not args.no_cpu_baseline and args.only == "all":
        line["cpu_baseline"] = cpu_baseline_train(cfg, q_np, k_np, v_np, do_np, ids_np)
    return line


def shard_seed(base_seed: int, rank: int) -> int:
    """Each rank draws its own shard of the workload (independent problems:
    the data path needs no collective)."""
    return base_seed + rank


def aggregate_value(work_per_rank: float, world: int, steps: int, max_ms: float,
                    unit_scale: float = 1e12) -> float:
    """Whole-job throughput: the work every rank did over the slowest rank's
    time."""
    return work_per_rank * world * steps / (max_ms * 1e-3) / unit_scale


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_e2e(api, cfg, q_np, k_np, v_np, do_np, ids_np, device, args, flops, world):
    """The same step through the public API from pinned host buffers: H2D of
    the inputs, index + forward + backward, D2H of the gradients, every step.
    Steps are pipelined the way a training loop would run them: step j+1's
    inputs upload on one stream and step j-1's gradients download on another
    while step j computes, through two device slots ordered by events."""
    import torch
    bf = torch.bfloat16
    hq = torch.from_numpy(q_np).to(bf).pin_memory()
    hk = torch.from_numpy(k_np).to(bf).pin_memory()
    hv = torch.from_numpy(v_np).to(bf).pin_memory()
    hdo = torch.from_numpy(do_np).to(bf).pin_memory()
    hids = torch.from_numpy(ids_np).pin_memory()
    host_in = (hq, hk, hv, hdo, hids)
    dq_h = torch.empty_like(hq).pin_memory()
    dk_h = torch.empty_like(hk).pin_memory()
    dv_h = torch.empty_like(hv).pin_memory()
    host_out = (dq_h, dk_h, dv_h)
    h2d = sum(x.numel() * x.element_size() for x in host_in)
    d2h = sum(x.numel() * x.element_size() for x in host_out)
    B, Hq, L, d = hq.shape
    Hkv = hk.shape[1]
    dev_in = [tuple(torch.empty_like(x, device=device) for x in host_in) for _ in range(2)]
    dev_out = [tuple(torch.empty_like(x, device=device) for x in host_out) for _ in range(2)]
    idx_buf = torch.empty(api.sep_index_bytes(B, L), dtype=torch.uint8, device=device)
    ws_f = torch.empty(api.sep_attn_workspace_bytes(B, Hq, Hkv, L, d, api.SEP_BF16, False),
                       dtype=torch.uint8, device=device)
    ws_b = torch.empty(api.sep_attn_workspace_bytes(B, Hq, Hkv, L, d, api.SEP_BF16, True),
                       dtype=torch.uint8, device=device)
    o = torch.empty_like(dev_in[0][0])
    lse = torch.empty((B, Hq, L), dtype=torch.float32, device=device)
    s_comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    torch.cuda.synchronize()

    def upload(slot):
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_comp[slot])  # the step that last read this slot is done
            for dst, src in zip(dev_in[slot], host_in):
                dst.copy_(src, non_blocking=True)
            ev_in[slot].record(s_in)

    def compute(slot):
        q, k, v, dout, ids = dev_in[slot]
        dq, dk, dv = dev_out[slot]
        s_comp.wait_event(ev_in[slot])
        s_comp.wait_event(ev_out[slot])  # this slot's last gradients have left
        api.sep_build_index(ids, synth.SEP_IDS, cfg.a, cfg.n, index_buf=idx_buf)
        api.sep_attn_fwd(idx_buf, q, k, v, o=o, lse=lse, ws=ws_f)
        api.sep_attn_bwd(idx_buf, q, k, v, o, lse, dout, dq=dq, dk=dk, dv=dv, ws=ws_b)
        ev_comp[slot].record(s_comp)

    def download(slot):
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[slot])
            for dst, src in zip(host_out, dev_out[slot]):
                dst.copy_(src, non_blocking=True)
            ev_out[slot].record(s_out)

    def run(n):
        upload(0)
        for j in range(n):
            if j + 1 < n:
                upload((j + 1) % 2)
            compute(j % 2)
            download(j % 2)
        torch.cuda.synchronize()

    run(max(3, args.warmup))
    n = max(5, args.steps)
    t0 = time.perf_counter()
    run(n)
    dt = max_over_ranks(time.perf_counter() - t0, world)
    # the host link's own roofline: the step's uploads alone and its
    # downloads alone, each timed by CUDA events on its copy stream (best of 5)
    def link_gbs(copies, stream):
        best = float("inf")
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(5):
            with torch.cuda.stream(stream):
                e0.record(stream)
                for dst, src in copies:
                    dst.copy_(src, non_blocking=True)
                e1.record(stream)
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        nbytes = sum(src.numel() * src.element_size() for _, src in copies)
        return nbytes / (best * 1e-3) / 1e9
    h2d_gbs = link_gbs(list(zip(dev_in[0], host_in)), s_in)
    d2h_gbs = link_gbs(list(zip(host_out, dev_out[0])), s_out)
    link_ms = max(h2d / h2d_gbs, d2h / d2h_gbs) * 1e-6
    # the pipelined gradients equal a plain serial call's (dQ is deterministic)
    q, k, v, dout, ids = (x.to(device) for x in host_in)
    buf = api.sep_build_index(ids, synth.SEP_IDS, cfg.a, cfg.n)
    o2, lse2 = api.sep_attn_fwd(buf, q, k, v)
    dq2, _, _ = api.sep_attn_bwd(buf, q, k, v, o2, lse2, dout)
    torch.cuda.synchronize()
    assert torch.equal(dq2.cpu(), dq_h), "pipelined end-to-end gradients differ"
    return {"value": round(flops * world * n / dt / 1e12, 3), "unit": "TFLOP/s",
            "ms_per_step": round(dt / n * 1e3, 4), "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "link": {"h2d_gbs": round(h2d_gbs, 1), "d2h_gbs": round(d2h_gbs, 1),
                     "bound_ms_per_step": round(link_ms, 4),
                     "frac": round(link_ms / (dt / n * 1e3), 3),
                     "note": "pinned copies of one step's inputs (uploads) and gradients "
                             "(downloads), each direction alone; the bound is the slower "
                             "direction, as they overlap on separate streams"},
            "note": "public API, eager launches, pinned host buffers, wall clock; uploads, "
                    "compute and downloads of consecutive steps overlap on three streams"}


def run_decode(args, rank, device, flush, peaks):
    """Streaming decode: the prompt enters through one bulk prefill
    (untimed), then every decode step (cache update + attention over the
    cache) is timed by CUDA events with L2 flushed before it."""
    import torch
    from separator_token_kv_sep_b300 import api
    cfg = synth.STREAM_DECODE
    qp, kp, vp, ids_np = synth.stream_inputs(cfg, seed=shard_seed(cfg.seed, rank))
    P = qp.shape[0]
    bf = torch.bfloat16
    dq = torch.from_numpy(qp).to(device, bf)
    dk = torch.from_numpy(kp).to(device, bf)
    dv = torch.from_numpy(vp).to(device, bf)
    dids = torch.from_numpy(ids_np).to(device)
    out = torch.empty((cfg.S, cfg.Hq, cfg.d), dtype=bf, device=device)
    p = api.cache_params(cfg.S, cfg.Hkv, cfg.d, cfg.a, cfg.s, cfg.w, cfg.c, cfg.theta)
    buf = api.sep_cache_init(p, device=device)
    T = cfg.prompt + cfg.steps
    # the prompt enters in one bulk prefill (the state 2048 update-only steps
    # leave); it is not timed
    pidx = torch.arange(cfg.prompt, device=device) % P
    api.sep_cache_prefill(p, buf, dk[pidx].contiguous(), dv[pidx].contiguous(),
                          dids[:cfg.prompt].contiguous(), synth.SEP_IDS)
    torch.cuda.synchronize()
    n_dec = cfg.steps
    ev_a = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(n_dec)]
    ev_b = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(n_dec)]
    graph = torch.cuda.CUDAGraph()
    # capture the whole decode phase: flush, event, step, event per token
    with torch.cuda.graph(graph):
        for j in range(n_dec):
            t = cfg.prompt + j
            flush()
            ev_a[j].record()
            api.sep_cache_step(p, buf, dq[t % P], dk[t % P], dv[t % P], dids[t], synth.SEP_IDS,
                               out=out)
            ev_b[j].record()
    # the capture did not run anything: the cache is still at the end of the prompt
    graph.replay()
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in zip(ev_a, ev_b)]
    total_ms = sum(step_ms)
    assert api.sep_get_device_status() == 0
    sep = np.isin(ids_np, synth.SEP_IDS)
    lens = decode_cache_lengths(sep, cfg.a, cfg.s, cfg.w, cfg.c)[cfg.prompt:T]
    G = cfg.Hq // cfg.Hkv
    # K and V rows read once per kv head; q, out, new k/v and ids
    kv_bytes = lens.sum() * cfg.Hkv * cfg.d * 2 * 2
    io_bytes = n_dec * cfg.S * (2 * cfg.Hq * cfg.d * 2 + 2 * cfg.Hkv * cfg.d * 2 + 4)
    alg_bytes = float(kv_bytes + io_bytes)
    gbs = alg_bytes / (total_ms * 1e-3) / 1e9
    tok_s = cfg.S * n_dec / (total_ms * 1e-3)
    return {"workload": "llama3_8b_stream_decode " + cfg.describe(),
            "value": round(tok_s, 1), "unit": "tok/s", "ms_per_step": round(total_ms / n_dec, 5),
            "mean_cache_entries": round(float(lens.mean()), 2), "gqa_group": G,
            "l2": L2_NOTE + ", before every decode step",
            "roofline": {"bound": "hbm", "kernel": "cache_step_kernel (one launch per step)",
                         "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4),
                         "traffic": DECODE_DRAM_TRAFFIC_BYTES,
                         "algorithmic_bytes_per_step": round(alg_bytes / n_dec)},
            "gpu_launches": n_dec}


FIXLLM_DELTA = 10  # one kept token per 10 positions: the separator density 0.10 of the workload


def run_variants(args, rank, device, flush, peaks):
    """The training step of the same Pythia-shaped workload under the mask
    variants the pages set beside SepLLM: windows n = 64 and n = L (full
    causal, the layer-0 variant), StreamingLLM (no separators), the FixLLM
    control (every FIXLLM_DELTA-th token instead of the separators) and
    hybrid heads (half the kv groups on full causal attention).
    Each step is sep_build_index(_fixed) + sep_attn_fwd + sep_attn_bwd,
    replayed from a CUDA graph with L2 flushed before it."""
    import torch
    from separator_token_kv_sep_b300 import api
    cfg = synth.PYTHIA_TRAIN_N128
    q_np, k_np, v_np, do_np, ids_np = synth.prefill_inputs(cfg, seed=shard_seed(cfg.seed, rank))
    bf = torch.bfloat16
    q = torch.from_numpy(q_np).to(device, bf)
    k = torch.from_numpy(k_np).to(device, bf)
    v = torch.from_numpy(v_np).to(device, bf)
    dout = torch.from_numpy(do_np).to(device, bf)
    ids = torch.from_numpy(ids_np).to(device)
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    a = cfg.a
    pos = np.arange(L)
    sep_keep = np.isin(ids_np, synth.SEP_IDS) | (pos < a)[None, :]
    fix_keep = np.broadcast_to(((pos + 1) % FIXLLM_DELTA == 0) | (pos < a), (B, L))
    sink_keep = np.broadcast_to(pos < a, (B, L))
    # hybrid heads: the first half of the kv groups on full causal attention
    half_full = (1 << (Hkv // 2)) - 1
    variants = [("sep_n64", 64, sep_keep, "sep", 0), ("sep_full_layer_nL", L, sep_keep, "sep", 0),
                ("streamingllm_n128", 128, sink_keep, "none", 0),
                ("fixllm_n128_delta10", 128, fix_keep, "fix", 0),
                ("hybrid_half_full_sep_n128", 128, sep_keep, "sep", half_full)]
    idx_buf = torch.empty(api.sep_index_bytes(B, L), dtype=torch.uint8, device=device)
    ws_f = torch.empty(api.sep_attn_workspace_bytes(B, Hq, Hkv, L, d, api.SEP_BF16, False),
                       dtype=torch.uint8, device=device)
    ws_b = torch.empty(api.sep_attn_workspace_bytes(B, Hq, Hkv, L, d, api.SEP_BF16, True),
                       dtype=torch.uint8, device=device)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, L), dtype=torch.float32, device=device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    steps = max(3, min(args.steps, 20))
    out = {}
    for name, n, keep, kind, fg in variants:
        def step():
            if kind == "fix":
                api.sep_build_index_fixed(B, L, a, n, FIXLLM_DELTA, index_buf=idx_buf, device=device)
            else:
                api.sep_build_index(ids, synth.SEP_IDS if kind == "sep" else [], a, n,
                                    index_buf=idx_buf)
            if fg:
                api.sep_attn_fwd_hybrid(idx_buf, q, k, v, fg, o=o, lse=lse, ws=ws_f)
                api.sep_attn_bwd_hybrid(idx_buf, q, k, v, o, lse, dout, fg, dq=dq, dk=dk, dv=dv,
                                        ws=ws_b)
            else:
                api.sep_attn_fwd(idx_buf, q, k, v, o=o, lse=lse, ws=ws_f)
                api.sep_attn_bwd(idx_buf, q, k, v, o, lse, dout, dq=dq, dk=dk, dv=dv, ws=ws_b)
        step()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        times = []
        for it in range(steps + 3):
            flush()
            e0.record()
            graph.replay()
            e1.record()
            torch.cuda.synchronize()
            if it >= 3:
                times.append(e0.elapsed_time(e1))
        assert api.sep_get_device_status() == 0
        ms = sum(times) / len(times)
        # per head: full-attention groups visit every causal pair
        n_full = bin(fg).count("1") * (Hq // Hkv)
        causal = B * L * (L + 1) // 2
        pairs = visited_pairs_keep(keep, n)
        head_pairs = (Hq - n_full) * pairs + n_full * causal
        pairs = head_pairs / Hq
        flops = 14.0 * d * head_pairs
        out[name] = {"window_n": n, "full_kv_groups": bin(fg).count("1"), "ms": round(ms, 5),
                     "value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                     "visited_over_causal": round(pairs / (B * L * (L + 1) / 2), 4),
                     "frac_of_bf16_peak": round(flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)}
    out["packed_docs_n128"] = run_packed_variant(q, k, v, dout, ids_np, cfg, steps, device, flush,
                                                 peaks, rank)
    out["note"] = ("index + fwd + bwd of the Pythia-shaped workload (B8 H12 L2048 d64 bf16, a4) "
                   "per variant; FLOPs 14 d per visited pair; CUDA graph, L2 flushed before "
                   f"each step, {steps} timed steps")
    return out


def pack_lengths(total: int, lo: int, hi: int, seed: int):
    """Seeded document lengths, uniform in [lo, hi], the last one cut so they
    sum to total."""
    rng = np.random.default_rng(seed)
    out = []
    while sum(out) < total:
        out.append(int(min(rng.integers(lo, hi + 1), total - sum(out))))
    return out


def run_packed_variant(q, k, v, dout, ids_np, cfg, steps, device, flush, peaks, rank):
    """The same token budget (B8 x 2048 tokens, 12 heads, d64) as one pack of
    documents of seeded lengths in [64, 2048]: sep_build_index_varlen +
    sep_attn_fwd_varlen + sep_attn_bwd_varlen, each document masked on its
    own (its own sinks, window and separators)."""
    import torch
    from separator_token_kv_sep_b300 import api
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    total = B * L
    lengths = pack_lengths(total, 64, L, shard_seed(3001, rank))
    cu_np = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    max_len = int(max(lengths))
    nb = len(lengths)
    # per head, the batch rows' tokens one after another, cut at the
    # document boundaries instead of the row boundaries
    pq = q.permute(1, 0, 2, 3).reshape(Hq, total, d).contiguous()
    pk = k.permute(1, 0, 2, 3).reshape(Hkv, total, d).contiguous()
    pv = v.permute(1, 0, 2, 3).reshape(Hkv, total, d).contiguous()
    pdo = dout.permute(1, 0, 2, 3).reshape(Hq, total, d).contiguous()
    ids_flat = ids_np.reshape(-1)
    ids = torch.from_numpy(ids_flat).to(device)
    cu = torch.from_numpy(cu_np).to(device)
    idx_buf = torch.empty(api.sep_index_bytes(nb, max_len), dtype=torch.uint8, device=device)
    ws_f = torch.empty(api.sep_attn_workspace_bytes_varlen(nb, total, max_len, Hq, Hkv, d, False),
                       dtype=torch.uint8, device=device)
    ws_b = torch.empty(api.sep_attn_workspace_bytes_varlen(nb, total, max_len, Hq, Hkv, d, True),
                       dtype=torch.uint8, device=device)
    o = torch.empty_like(pq)
    lse = torch.empty((Hq, total), dtype=torch.float32, device=device)
    dq, dk, dv = torch.empty_like(pq), torch.empty_like(pk), torch.empty_like(pv)

    def step():
        api.sep_build_index_varlen(ids, cu, max_len, synth.SEP_IDS, cfg.a, cfg.n,
                                   index_buf=idx_buf)
        api.sep_attn_fwd_varlen(idx_buf, pq, pk, pv, nb, max_len, o=o, lse=lse, ws=ws_f)
        api.sep_attn_bwd_varlen(idx_buf, pq, pk, pv, o, lse, pdo, nb, max_len, dq=dq, dk=dk,
                                dv=dv, ws=ws_b)
    step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    times = []
    for it in range(steps + 3):
        flush()
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        if it >= 3:
            times.append(e0.elapsed_time(e1))
    assert api.sep_get_device_status() == 0
    ms = sum(times) / len(times)
    pairs = sum(visited_pairs_per_head(ids_flat[None, cu_np[b]:cu_np[b + 1]], cfg.a, cfg.n)
                for b in range(nb))
    flops = 14.0 * d * pairs * Hq
    causal = sum(x * (x + 1) // 2 for x in lengths)
    return {"window_n": cfg.n, "documents": nb, "max_len": max_len, "total_tokens": total,
            "ms": round(ms, 5), "value": round(flops / (ms * 1e-3) / 1e12, 2),
            "unit": "TFLOP/s", "visited_over_causal": round(pairs / causal, 4),
            "frac_of_bf16_peak": round(flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
            "note": "one pack of seeded document lengths in [64, 2048] (the last one cut): "
                    "sep_build_index_varlen + sep_attn_fwd_varlen + sep_attn_bwd_varlen"}


def run_index_scaling(args, rank, device, flush):
    """sep_build_index alone: the scaling run at B = 64, L = 65536 (16 MB of
    ids) and the long-prefill row B = 1, L = 65536; device time and
    algorithmic GB/s."""
    import torch
    from separator_token_kv_sep_b300 import api
    out = {}
    for B, L, a, n, p, seed in ((64, 65536, 4, 8192, 0.12, 2001), (1, 65536, 4, 8192, 0.12, 1005)):
        rng = np.random.default_rng(shard_seed(seed, rank))
        ids_np = synth.token_ids(rng, (B, L), p)
        ids = torch.from_numpy(ids_np).to(device)
        idx_buf = torch.empty(api.sep_index_bytes(B, L), dtype=torch.uint8, device=device)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        times = []
        for it in range(13):
            flush()
            e0.record()
            api.sep_build_index(ids, synth.SEP_IDS, a, n, index_buf=idx_buf)
            e1.record()
            torch.cuda.synchronize()
            if it >= 3:
                times.append(e0.elapsed_time(e1))
        assert api.sep_get_device_status() == 0
        ms = sum(times) / len(times)
        count = int((np.isin(ids_np, synth.SEP_IDS) | (np.arange(L) < a)[None, :]).sum())
        T = (L + 127) // 128
        alg = (4.0 * B * L + 4.0 * B * (L + 1) + 4.0 * count + 16.0 * B * T
               + 4.0 * B * ((L + 31) // 32))
        out[f"B{B}_L{L}"] = {"workload": f"sep_build_index B{B} L{L} a{a} n{n} p{p}",
                             "ms": round(ms, 5), "gbs": round(alg / (ms * 1e-3) / 1e9, 1),
                             "algorithmic_bytes": int(alg)}
    out["note"] = ("ids read + keep_prefix, keep_pos (valid entries), block records and keep "
                   "bits written; L2 flushed before each call; the call includes the memset "
                   "of the scan's scratch")
    return out


def run_prefill(args, rank, device, flush, peaks):
    """Forward-only prefill at L = 8192 and L = 65536 (index + forward)."""
    import torch
    from separator_token_kv_sep_b300 import api
    res = {}
    for cfg, reps in ((synth.LLAMA_PREFILL, 10), (synth.LONG_PREFILL, 3)):
        rng = np.random.Generator(np.random.PCG64(shard_seed(cfg.seed, rank)))
        ids_np = synth.token_ids(rng, (cfg.B, cfg.L), cfg.p)
        gen = torch.Generator(device=device)
        gen.manual_seed(shard_seed(cfg.seed, rank))
        bf = torch.bfloat16
        q = torch.randn((cfg.B, cfg.Hq, cfg.L, cfg.d), generator=gen, device=device).to(bf)
        k = torch.randn((cfg.B, cfg.Hkv, cfg.L, cfg.d), generator=gen, device=device).to(bf)
        v = torch.randn((cfg.B, cfg.Hkv, cfg.L, cfg.d), generator=gen, device=device).to(bf)
        ids = torch.from_numpy(ids_np).to(device)
        idx_buf = api.sep_build_index(ids, synth.SEP_IDS, cfg.a, cfg.n)
        o, lse = api.sep_attn_fwd(idx_buf, q, k, v)
        ws = torch.empty(api.sep_attn_workspace_bytes(cfg.B, cfg.Hq, cfg.Hkv, cfg.L, cfg.d,
                                                      api.SEP_BF16, False),
                         dtype=torch.uint8, device=device)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        times = []
        for it in range(reps + 2):
            flush()
            e0.record()
            api.sep_attn_fwd(idx_buf, q, k, v, o=o, lse=lse, ws=ws)
            e1.record()
            torch.cuda.synchronize()
            if it >= 2:
                times.append(e0.elapsed_time(e1))
        pairs = visited_pairs_per_head(ids_np, cfg.a, cfg.n)
        flops = 4.0 * cfg.d * pairs * cfg.Hq
        ms = sum(times) / len(times)
        tf = flops / (ms * 1e-3) / 1e12
        res[cfg.name] = {"workload": cfg.describe(), "ms": round(ms, 4),
                         "value": round(tf, 2), "unit": "TFLOP/s",
                         "visited_over_causal": round(pairs / (cfg.B * cfg.L * (cfg.L + 1) / 2), 4),
                         "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
                         "note": "sep_attn_fwd call (gather + attention kernel), events on the "
                                 "launching stream, L2 flushed before each call; inputs drawn "
                                 "on the device with torch's seeded generator"}
    return res


# ---------------------------------------------------------------------------
# CPU baselines (the float64 oracle, as it stands)
# ---------------------------------------------------------------------------

def _cores() -> int:
    return len(os.sched_getaffinity(0))


def cpu_baseline_train(cfg, q_np, k_np, v_np, do_np, ids_np, batches=(0,)):
    from oracle import sepllm as O
    bs = list(batches)
    t0 = time.perf_counter()
    O.attention_forward(q_np[bs], k_np[bs], v_np[bs], ids_np[bs], synth.SEP_IDS, cfg.a, cfg.n)
    O.attention_backward(q_np[bs], k_np[bs], v_np[bs], do_np[bs], ids_np[bs], synth.SEP_IDS,
                         cfg.a, cfg.n)
    dt = time.perf_counter() - t0
    pairs = visited_pairs_per_head(ids_np[bs], cfg.a, cfg.n)
    flops = 14.0 * cfg.d * pairs * cfg.Hq
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": _cores(),
            "kind": "oracle", "seconds": round(dt, 3),
            "sample": f"batch rows {bs} of the training workload ({len(bs)}/{cfg.B} of it), "
                      "float64 NumPy forward + backward with explicit masks"}


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is one batch row of the
    training workload (forward + backward, float64 NumPy)."""
    if rank != 0:
        return None
    cfg = synth.PYTHIA_TRAIN_N128
    q_np, k_np, v_np, do_np, ids_np = synth.prefill_inputs(cfg)
    from oracle import sepllm as O
    heads = [0, 1]

    def step(b):
        sl = slice(b, b + 1)
        qq, kk, vv, dd = (x[sl][:, heads] for x in (q_np, k_np, v_np, do_np))
        O.attention_forward(qq, kk, vv, ids_np[sl], synth.SEP_IDS, cfg.a, cfg.n)
        O.attention_backward(qq, kk, vv, dd, ids_np[sl], synth.SEP_IDS, cfg.a, cfg.n)

    for w in range(args.warmup):
        step(w % cfg.B)
    t0 = time.perf_counter()
    for s in range(args.steps):
        step(s % cfg.B)
    dt = time.perf_counter() - t0
    pairs = sum(visited_pairs_per_head(ids_np[s % cfg.B:s % cfg.B + 1], cfg.a, cfg.n)
                for s in range(args.steps))
    flops = 14.0 * cfg.d * pairs * len(heads)
    value = flops / dt / 1e12
    sample = (f"each step: one batch row, q heads {heads} of the training workload "
              f"(forward + backward, float64 NumPy)")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "pythia160m_train_step " + cfg.describe()},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": _cores(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["all", "train", "decode", "prefill", "index"],
                    default="all",
                    help="train: the training step alone (no e2e, decode or prefill legs); "
                         "decode / prefill / index: that leg alone (profiling runs)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus if args.gpus == 1 else 1)))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0
    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(device)
        dist.init_process_group("nccl", device_id=device)
    if args.only in ("decode", "prefill", "index"):
        torch.cuda.set_device(device)
        flush = L2Flush(device)
        if args.only == "decode":
            line = run_decode(args, rank, device, flush, load_peaks())
        elif args.only == "prefill":
            line = run_prefill(args, rank, device, flush, load_peaks())
        else:
            line = run_index_scaling(args, rank, device, flush)
    else:
        line = run_ours(args, rank, world, device)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
