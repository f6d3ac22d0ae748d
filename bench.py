#!/usr/bin/env python
"""Benchmark: useful attention TFLOP/s of blockwise ring attention on GB300.

One step = one pass of the whole hot path over one batch: the fused ring
forward (ra_ring_attention) and, when the library has it, the blockwise
backward (ra_ring_attention_bwd), on the long causal GQA workload
(b=1, S=262,144, h=32, n_kv=8, d=128, N=8 striped shards, bf16 inputs drawn
N(0,1) x 0.5).  Useful FLOPs: 2 b S^2 h d forward (causal), 2.5x that for the
backward.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
       python bench.py --block-steps     (ring-step timings only)
       python bench.py --ring            (under torchrun: the ring across the ranks)
Prints one JSON line (rank 0).  Under torchrun each rank runs its own replica
(weak scaling, no collective on the data path).
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "useful attention TFLOP/s fwd & bwd (causal, S=256K GQA) and % of BF16 tensor peak"
WORKLOAD = "causal256k"

# Per-launch DRAM traffic of the dominant kernel (dram__bytes_read.sum +
# dram__bytes_write.sum), valid only while the kernel source hash matches
# the one the capture was taken with.  Captured on the one-shard 32K case
# (5.19 GB) and scaled to this workload: the compulsory 2.3 GB with S (x 8),
# the rest with the causal step count (x 64).
TRAFFIC = {
    "bwd": {"bytes_per_launch": 204e9, "src_sha": "621eee2074e81eb6",
            "method": "ncu on the causal32k1 case (5.19 GB), scaled: 2.3 GB x 8 + 2.89 GB x 64"},
}


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # ten steps: the e2e pipeline's first uploads and last downloads are not
    # hidden (~0.4 s per run where pinned copies move ~27 GB/s), and fewer
    # steps would charge them to too little work
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the layout / causal-imbalance measurements")
    ap.add_argument("--block-steps", action="store_true",
                    help="only the ring-step (ra_block_step) timings at the workload's shard "
                         "size, as one JSON line (for profiling the block-step kernels)")
    ap.add_argument("--ring", action="store_true",
                    help="the real ring across the ranks: the workload's sequence split over "
                         "them, key/value blocks exchanged point to point (ring.py)")
    return ap.parse_args()


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: every rank contributes its own measurement and
    all of them receive the maximum (a no-op for one rank)."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(step_flops: float, steps: int, world: int, ms: float) -> float:
    """Whole-job useful TFLOP/s: every rank runs `steps` steps of its own
    replica; the job takes as long as the slowest rank."""
    return step_flops * steps * world / (ms / 1e3) / 1e12


def replica_seed(seed: int, rank: int) -> int:
    """Seed of rank `rank`'s replica inputs (independent batches per rank)."""
    return seed + 1000 * rank


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": pk["hbm_gbs"], "bf16": pk["bf16_tflops"],
                "bf16_sustained": pk.get("bf16_tflops_sustained", pk["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


def _src_sha(name):
    with open(os.path.join(ROOT, "long_context_exact_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- oracle arm
def _workload_config(w, layout: int, have_bwd: bool, world: int) -> dict:
    """The JSON line's `config` for a workload (both arms print the same)."""
    return {"workload": w.name, "b": w.b, "S": w.S, "h": w.h, "n_kv": w.n_kv, "d": w.d,
            "n_shards": w.n_shards,
            "layout": {0: "contiguous", 1: "striped", 2: "zigzag"}[layout],
            "causal": w.causal, "backward": have_bwd,
            "l2": "inputs larger than L2 (Q alone is "
                  f"{w.b * w.S * w.h * w.d * 2 / 1e9:.2f} GB); no flush",
            "parallelism": f"replica x{world}"}


def _workload_layout(w) -> int:
    from long_context_exact_gb300.inputs import STRIPED
    return STRIPED if STRIPED in w.layouts else w.layouts[0]


def _cpu_oracle_sample(w, fwd_rows: int, bwd_rows: int, seed: int, inputs=None):
    """Time the fp64 oracle on a bounded sample of the workload: forward on
    `fwd_rows` random query rows (all heads), backward on `bwd_rows`.
    `inputs` = (q, k, v, dO) from make_inputs, drawn here when not given.
    Returns (useful FLOPs done, forward seconds, seconds, threads, torch)."""
    import numpy as np
    import torch

    from long_context_exact_gb300 import accounting
    from long_context_exact_gb300.inputs import make_inputs
    from oracle import oracle

    oracle.build()
    if inputs is None:
        inputs = make_inputs(w.b, w.S, w.h, w.n_kv, w.d, w.seed, w.amplitude, with_dout=True)
    q, k, v, do = inputs
    rng = np.random.default_rng(seed)
    rows_f = np.sort(rng.choice(w.S, fwd_rows, replace=False))
    rows_b = np.sort(rng.choice(w.S, bwd_rows, replace=False))
    per_row_fwd = accounting.fwd_useful_flops(w.b, w.S, w.h, w.d, w.causal) / w.S
    t0 = time.perf_counter()
    oracle.attn_fwd_rows(q, k, v, w.causal, rows=rows_f)
    t1 = time.perf_counter()
    flops = per_row_fwd * fwd_rows
    if bwd_rows:
        oracle.attn_bwd_rows(q, k, v, do, w.causal, rows=rows_b)
        flops += 2.5 * per_row_fwd * bwd_rows
    t2 = time.perf_counter()
    threads = oracle.max_threads()
    return flops, (t1 - t0), (t2 - t0), threads, torch


def _cpu_oracle_single_thread_tiny():
    """The oracle on the tiny configuration (b1 h2 kv2 d64 S1024 N4,
    non-causal), every row, forward, on one thread: (seconds, TFLOP/s)."""
    from long_context_exact_gb300 import accounting
    from long_context_exact_gb300.inputs import WORKLOADS, workload_inputs
    from oracle import oracle

    w = WORKLOADS["tiny"]
    q, k, v = workload_inputs(w)[:3]
    n = oracle.max_threads()
    oracle.set_threads(1)
    try:
        t0 = time.perf_counter()
        oracle.attn_fwd_rows(q, k, v, w.causal)
        secs = time.perf_counter() - t0
    finally:
        oracle.set_threads(n)
    return secs, accounting.fwd_useful_flops(w.b, w.S, w.h, w.d, w.causal) / secs / 1e12


def run_reference(a, rank, world):
    if rank != 0:
        return
    from long_context_exact_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS[a.workload]
    fwd_rows, bwd_rows = 8, 2
    vals = []
    threads = 1
    # the workload's inputs once (drawing 256K rows per step would take longer
    # than the oracle's sample itself)
    inputs = make_inputs(w.b, w.S, w.h, w.n_kv, w.d, w.seed, w.amplitude, with_dout=True)
    for _ in range(a.warmup):
        _cpu_oracle_sample(w, fwd_rows, bwd_rows, seed=0, inputs=inputs)
    for s in range(a.steps):
        flops, _, secs, threads, _ = _cpu_oracle_sample(w, fwd_rows, bwd_rows, seed=s + 1,
                                                        inputs=inputs)
        vals.append((flops, secs))
    tot_f = sum(f for f, _ in vals)
    tot_s = sum(s for _, s in vals)
    value = tot_f / tot_s / 1e12
    sample = (f"fp64 oracle on {fwd_rows} forward + {bwd_rows} backward random query rows "
              f"(all {w.h} heads) of the {w.name} workload per step")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": tot_s / a.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _workload_config(w, _workload_layout(w), True, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------- extras
def _time_ms(fn, reps=2):
    import torch
    fn()
    torch.cuda.synchronize()
    best = None
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1)
        best = t if best is None else min(best, t)
    return best


def ring_imbalance(b, S, h, d, N, q, k, v, dev):
    """One ra_block_step per (query shard i, ring step s), timed with CUDA
    events, t(i, s); the makespan an N-device ring would see,
    T = sum_s max_i t(i, s), and its utilisation sum t / (N T), for the
    contiguous, striped and zig-zag placements."""
    import torch

    from long_context_exact_gb300 import binding as ra
    from long_context_exact_gb300.inputs import CONTIGUOUS, STRIPED, ZIGZAG

    rep = {}
    L = S // N
    for name, layout in (("contiguous", CONTIGUOUS), ("striped", STRIPED), ("zigzag", ZIGZAG)):
        _, _, tok = ra.position_map(layout, S, N, device=dev)
        t = [[0.0] * N for _ in range(N)]
        for i in range(N):
            qi = q.index_select(1, tok[i].long()).contiguous()
            st = ra.new_state(b, L, h, d, dev)
            for s_ in range(N):
                j = (i - s_) % N
                kj = k.index_select(1, tok[j].long()).contiguous()
                vj = v.index_select(1, tok[j].long()).contiguous()
                torch.cuda.synchronize()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                ra.block_step(qi, kj, vj, st, tok[i], tok[j], True)
                e1.record()
                torch.cuda.synchronize()
                t[i][s_] = e0.elapsed_time(e1)
                del kj, vj
            del qi, st
        total = sum(sum(r) for r in t)
        makespan = sum(max(t[i][s_] for i in range(N)) for s_ in range(N))
        rep["ring_" + name] = {
            "sum_ms": total, "makespan_ms": makespan, "utilisation": total / (N * makespan),
            "per_shard_ms": [sum(t[i]) for i in range(N)]}
    ra.stream_check()
    return rep


def imbalance_at(name, dev):
    """The ring imbalance picture at another workload's shape (its own
    seeded device inputs)."""
    import torch

    from long_context_exact_gb300.inputs import WORKLOADS

    w = WORKLOADS[name]
    gen = torch.Generator(device=dev).manual_seed(w.seed)

    def rnd(*shape):
        x = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32)
        return x.mul_(w.amplitude).to(torch.bfloat16)

    q, k, v = rnd(w.b, w.S, w.h, w.d), rnd(w.b, w.S, w.n_kv, w.d), rnd(w.b, w.S, w.n_kv, w.d)
    rep = ring_imbalance(w.b, w.S, w.h, w.d, w.n_shards, q, k, v, dev)
    rep["workload"] = w.name
    return {k_: ({kk: vv for kk, vv in v_.items() if kk != "per_shard_ms"}
                 if isinstance(v_, dict) else v_) for k_, v_ in rep.items()}


def layout_and_imbalance_report(w, q, k, v, dev):
    """Forward of the same shape non-causal, with contiguous shards and with
    zig-zag shards, and the causal load-balance picture of the third page's
    section 6 (and the first page's striped and zig-zag remedies): time one
    ra_block_step per (query shard i, ring step s), t(i, s), and form the
    makespan an N-device ring would see, T = sum_s max_i t(i, s), and its
    utilisation sum t / (N T)."""
    import torch

    from long_context_exact_gb300 import accounting
    from long_context_exact_gb300 import binding as ra
    from long_context_exact_gb300.inputs import CONTIGUOUS, STRIPED, ZIGZAG

    out = torch.empty((w.b, w.S, w.h, w.d), dtype=torch.float32, device=dev)
    lse = torch.empty((w.b, w.h, w.S), dtype=torch.float32, device=dev)
    rep = {}
    f_nc = accounting.fwd_useful_flops(w.b, w.S, w.h, w.d, False)
    f_c = accounting.fwd_useful_flops(w.b, w.S, w.h, w.d, True)
    for name, layout, causal, flops in (("noncausal", STRIPED, False, f_nc),
                                        ("causal_striped", STRIPED, True, f_c),
                                        ("causal_contiguous", CONTIGUOUS, True, f_c),
                                        ("causal_zigzag", ZIGZAG, True, f_c)):
        ms = _time_ms(lambda: ra.ring_attention(q, k, v, w.n_shards, layout, causal, out=out,
                                                lse=lse))
        rep[name + "_fwd_ms"] = ms
        rep[name + "_fwd_tflops"] = flops / (ms / 1e3) / 1e12
    rep["striped_causal_vs_noncausal_per_useful_flop"] = (
        rep["causal_striped_fwd_tflops"] / rep["noncausal_fwd_tflops"])
    del out, lse
    N = w.n_shards
    rep.update(ring_imbalance(w.b, w.S, w.h, w.d, N, q, k, v, dev))
    rep["model_utilisation_contiguous"] = {
        "(N+1)/2N": accounting.causal_utilisation_contiguous(N),
        "N/(2N-1)": accounting.causal_utilisation_contiguous(N, half_diagonal=True)}
    ra.stream_check()
    return rep


def exp2_roof_report(w, dev, clk):
    """The forward's second roof: the measured exp2 rate of the special-
    function units (ra_ex2_probe) turned into the useful TFLOP/s it allows.
    Every attended (query, key) element costs one exp2 and 4 d useful FLOPs
    forward; the backward recomputes one exp2 per element for 10 d FLOPs."""
    import torch

    from long_context_exact_gb300 import binding as ra

    iters = 2048
    sink, n = ra.ex2_probe(iters)
    best = _time_ms(lambda: ra.ex2_probe(iters, sink), reps=3)
    ra.stream_check()
    rate = n / (best / 1e3)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = (clk or {}).get("sm_mhz")
    return {"exp2_per_s": rate, "ms": best, "exp2_evaluated": n,
            "per_sm_per_clk": rate / sms / (mhz * 1e6) if mhz else None,
            "clock_note": "per-clock figure uses the median SM clock of the timed region",
            "fwd_roof_tflops": rate * 4 * w.d / 1e12,
            "bwd_roof_tflops": rate * 10 * w.d / 1e12}


def hbm_kernel_report(w, dev, peaks):
    """Achieved HBM bandwidth of the memory-bound kernels on one shard's rows
    (what a ring step of the block path finalizes or merges): ra_finalize
    reads and rewrites O and reads l, m, writing LSE; ra_merge reads two
    (O, LSE) pairs and writes one."""
    import torch

    from long_context_exact_gb300 import binding as ra

    L = w.S // w.n_shards
    gen = torch.Generator(device=dev).manual_seed(7)
    shape = (w.b, L, w.h, w.d)
    o_a = torch.randn(shape, generator=gen, device=dev)
    o_b = torch.randn(shape, generator=gen, device=dev)
    o_c = torch.randn(shape, generator=gen, device=dev)
    lse_a = torch.randn((w.b, w.h, L), generator=gen, device=dev)
    lse_b = torch.randn((w.b, w.h, L), generator=gen, device=dev)
    lse_c = torch.empty_like(lse_a)
    m = torch.randn((w.b, w.h, L), generator=gen, device=dev)
    l = 1.0 + torch.rand((w.b, w.h, L), generator=gen, device=dev)
    o_bytes = o_a.numel() * 4
    row_bytes = lse_a.numel() * 4
    out = {}
    fin_ms = _time_ms(lambda: ra.finalize((m, l, o_c), lse=lse_c), reps=3)
    mrg_ms = _time_ms(lambda: ra.merge(o_a, lse_a, o_b, lse_b, o=o_c, lse=lse_c), reps=3)
    ra.stream_check()
    for name, ms, nbytes in (("finalize", fin_ms, 2 * o_bytes + 3 * row_bytes),
                             ("merge", mrg_ms, 3 * o_bytes + 3 * row_bytes)):
        gbs = nbytes / (ms / 1e3) / 1e9
        out[name] = {"ms": ms, "bytes": nbytes, "gbs": gbs, "frac_of_hbm_peak": gbs / peaks["hbm_gbs"],
                     "rows": f"b={w.b} x L={L} x h={w.h}, d={w.d}"}
    del o_a, o_b, o_c
    return out


def prefill_report(w, q, k, v, dev):
    """Chunked prefill at the workload's length: the last Lq tokens of the
    sequence attend to all S keys (ra_chunked_prefill), with the automatic
    key split and with a single split."""
    import torch

    from long_context_exact_gb300 import binding as ra

    res = []
    kpos = torch.arange(w.S, dtype=torch.int32, device=dev)
    for Lq in (512, 4096):
        if Lq > w.S:
            continue
        qc = q[:, w.S - Lq:].contiguous()
        qpos = kpos[w.S - Lq:].contiguous()
        pairs = Lq * w.S - Lq * (Lq - 1) // 2          # visible (query, key) pairs per head
        flops = 4.0 * w.b * w.h * w.d * pairs
        for splits in (0, 1):
            ws = torch.empty(max(ra.prefill_workspace_size(Lq, w.S, splits, w.b, w.h, w.n_kv,
                                                           w.d), 16),
                             dtype=torch.uint8, device=dev)
            ms = _time_ms(lambda: ra.chunked_prefill(qc, k, v, qpos, kpos, True, n_splits=splits,
                                                     workspace=ws), reps=3)
            used = ws.numel() // (w.b * w.h * Lq * (2 + w.d) * 4)
            res.append({"Lq": Lq, "Lk": w.S, "n_splits": splits, "splits_used": int(used),
                        "ms": ms, "tflops": flops / (ms / 1e3) / 1e12})
            del ws
    ra.stream_check()
    return res


def block_step_report(w, q, k, v, dev):
    """One ring step through ra_block_step at the workload's shard size
    L = S / N, the per-device step of a ring across GPUs: a key block wholly
    before the queries (every tile seen in full), the diagonal block (equal
    positions), a striped step (query shard 1 against key shard 0 of N
    striped shards) and the non-causal step.  Useful FLOPs count the visible
    (query, key) pairs: 4 b h d per pair."""
    import torch

    from long_context_exact_gb300 import binding as ra

    N = w.n_shards
    L = w.S // N
    qb, kb, vb = (t[:, :L].contiguous() for t in (q, k, v))
    ar = torch.arange(L, dtype=torch.int32, device=dev)
    tri = L * (L + 1) // 2
    cases = (("off_diagonal", ar + L, ar, True, L * L), ("diagonal", ar, ar, True, tri),
             ("striped", ar * N + 1, ar * N, True, tri), ("noncausal", ar, ar, False, L * L))
    res = {"L": L, "b": w.b, "h": w.h, "n_kv": w.n_kv, "d": w.d}
    st = ra.new_state(w.b, L, w.h, w.d, dev)
    for name, qp, kp, causal, pairs in cases:
        ms = _time_ms(lambda: ra.block_step(qb, kb, vb, st, qp, kp, causal), reps=3)
        res[name] = {"ms": ms, "tflops": 4.0 * w.b * w.h * w.d * pairs / (ms / 1e3) / 1e12}
    del st, qb, kb, vb
    ra.stream_check()
    return res


def packed_report(w, q, k, v, do, layout, dev):
    """Packed documents in the workload's window (the third page's section 5,
    branch two: a kernel that skips the masked blocks): document lengths
    drawn log-uniformly in [1K, 64K] tokens (seeded), forward and backward
    with the block-diagonal causal mask.  Useful FLOPs count each document's
    own causal triangle: 2 b h d n^2 per document of n tokens forward, 2.5x
    that backward."""
    import numpy as np
    import torch

    from long_context_exact_gb300 import binding as ra
    from long_context_exact_gb300.inputs import packed_offsets

    cu_np = packed_offsets(w.S, w.seed, b=w.b)
    cu = torch.from_numpy(cu_np).to(dev)
    lens = (cu_np[:, 1:] - cu_np[:, :-1]).astype(np.float64)
    f_fwd = float(2.0 * w.h * w.d * (lens ** 2).sum())
    out = torch.empty((w.b, w.S, w.h, w.d), dtype=torch.float32, device=dev)
    lse = torch.empty((w.b, w.h, w.S), dtype=torch.float32, device=dev)
    fwd_ms = _time_ms(lambda: ra.ring_attention(q, k, v, w.n_shards, layout, True, out=out,
                                                lse=lse, cu_seqlens=cu), reps=2)
    bwd_ms = _time_ms(lambda: ra.ring_attention_bwd(q, k, v, out, lse, do, w.n_shards, layout,
                                                    True, cu_seqlens=cu), reps=2)
    ra.stream_check()
    return {"n_docs": int((lens > 0).sum()), "doc_len_min": int(lens[lens > 0].min()),
            "doc_len_max": int(lens.max()), "fwd_ms": fwd_ms,
            "fwd_tflops": f_fwd / (fwd_ms / 1e3) / 1e12, "bwd_ms": bwd_ms,
            "bwd_tflops": 2.5 * f_fwd / (bwd_ms / 1e3) / 1e12,
            "useful_fraction_of_unpacked_causal": f_fwd / (2.0 * w.b * w.S * w.S * w.h * w.d)}


# ---------------------------------------------------------------- our arm
def config_table_report(dev):
    """Throughput on each configuration of the pages' workload set, one
    GB300: the forward (and for the b = 2 configuration the backward, as
    2.5 x and as 2 x the forward's useful FLOPs), each timed as the best of
    two launches after one warm-up, inputs seeded on the device."""
    import torch

    from long_context_exact_gb300 import accounting
    from long_context_exact_gb300 import binding as ra
    from long_context_exact_gb300.inputs import CONTIGUOUS, STRIPED, WORKLOADS

    rep = {}
    for key in ("tiny", "noncausal32k", "causal64k", "causal256k", "bwd64k"):
        w = WORKLOADS[key]
        gen = torch.Generator(device=dev).manual_seed(w.seed)

        def rnd(*shape):
            x = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32)
            return x.mul_(w.amplitude).to(torch.bfloat16)

        q, k, v = rnd(w.b, w.S, w.h, w.d), rnd(w.b, w.S, w.n_kv, w.d), rnd(w.b, w.S, w.n_kv, w.d)
        out = torch.empty((w.b, w.S, w.h, w.d), dtype=torch.float32, device=dev)
        lse = torch.empty((w.b, w.h, w.S), dtype=torch.float32, device=dev)
        f_fwd = accounting.fwd_useful_flops(w.b, w.S, w.h, w.d, w.causal)
        for layout in w.layouts:
            name = {CONTIGUOUS: "contiguous", STRIPED: "striped"}.get(layout, "zigzag")
            ms = _time_ms(lambda: ra.ring_attention(q, k, v, w.n_shards, layout, w.causal,
                                                    out=out, lse=lse))
            row = {"workload": w.name, "fwd_ms": ms, "fwd_tflops": f_fwd / (ms / 1e3) / 1e12}
            if w.backward:
                do = rnd(w.b, w.S, w.h, w.d)
                dq = torch.empty_like(out)
                dk = torch.empty((w.b, w.S, w.n_kv, w.d), dtype=torch.float32, device=dev)
                dv = torch.empty_like(dk)
                ws = torch.empty(max(ra.bwd_workspace_size(w.S, w.n_shards, w.b, w.h, w.n_kv,
                                                           w.d), 16),
                                 dtype=torch.uint8, device=dev)
                bms = _time_ms(lambda: ra.ring_attention_bwd(q, k, v, out, lse, do, w.n_shards,
                                                             layout, w.causal, dq=dq, dk=dk,
                                                             dv=dv, workspace=ws))
                f_bwd = accounting.bwd_useful_flops(w.b, w.S, w.h, w.d, w.causal)
                row.update({"bwd_ms": bms, "bwd_tflops": f_bwd / (bms / 1e3) / 1e12,
                            "bwd_tflops_2x": 2.0 * f_fwd / (bms / 1e3) / 1e12,
                            "step_tflops": (f_fwd + f_bwd) / ((ms + bms) / 1e3) / 1e12})
                del do, dq, dk, dv, ws
            rep[f"{key}_{name}"] = row
        del q, k, v, out, lse
    ra.stream_check()
    return rep


def run_ours(a, rank, world, local_rank):
    import torch

    from long_context_exact_gb300 import accounting
    from long_context_exact_gb300 import binding as ra
    from long_context_exact_gb300 import build as lib_build
    from long_context_exact_gb300.inputs import STRIPED, WORKLOADS

    w = WORKLOADS[a.workload]
    layout = STRIPED if STRIPED in w.layouts else w.layouts[0]
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0:
        lib_build.build()
    if world > 1:
        torch.distributed.barrier()
    ra.load()

    gen = torch.Generator(device=dev).manual_seed(replica_seed(w.seed, rank))

    def rnd(*shape):
        x = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32)
        return x.mul_(w.amplitude).to(torch.bfloat16)

    q = rnd(w.b, w.S, w.h, w.d)
    k = rnd(w.b, w.S, w.n_kv, w.d)
    v = rnd(w.b, w.S, w.n_kv, w.d)
    do = rnd(w.b, w.S, w.h, w.d)
    out = torch.empty((w.b, w.S, w.h, w.d), dtype=torch.float32, device=dev)
    lse = torch.empty((w.b, w.h, w.S), dtype=torch.float32, device=dev)
    dq = torch.empty_like(out)
    dk = torch.empty((w.b, w.S, w.n_kv, w.d), dtype=torch.float32, device=dev)
    dv = torch.empty_like(dk)
    ws = torch.empty(max(ra.bwd_workspace_size(w.S, w.n_shards, w.b, w.h, w.n_kv, w.d), 16),
                     dtype=torch.uint8, device=dev)

    have_bwd = True
    try:
        ra.ring_attention(q, k, v, w.n_shards, layout, w.causal, out=out, lse=lse)
        ra.ring_attention_bwd(q, k, v, out, lse, do, w.n_shards, layout, w.causal, dq=dq, dk=dk,
                              dv=dv, workspace=ws)
    except ra.RAError as e:
        if e.status != ra.RA_ERR_UNSUPPORTED:
            raise
        have_bwd = False
    ra.stream_check()

    stream = torch.cuda.current_stream()
    ev = []

    def step(record: bool):
        e0 = torch.cuda.Event(enable_timing=True) if record else None
        e1 = torch.cuda.Event(enable_timing=True) if record else None
        e2 = torch.cuda.Event(enable_timing=True) if record else None
        if record:
            e0.record(stream)
        ra.ring_attention(q, k, v, w.n_shards, layout, w.causal, out=out, lse=lse)
        if record:
            e1.record(stream)
        if have_bwd:
            ra.ring_attention_bwd(q, k, v, out, lse, do, w.n_shards, layout, w.causal, dq=dq,
                                  dk=dk, dv=dv, workspace=ws)
        if record:
            e2.record(stream)
            ev.append((e0, e1, e2))

    for _ in range(a.warmup):
        step(False)
    ra.stream_check()

    clocks = ClockSampler(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    launches0 = ra.launch_count()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(a.steps):
        step(True)
    t_end.record(stream)
    torch.cuda.synchronize()
    launches = ra.launch_count() - launches0
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    ra.stream_check()
    elapsed_ms = t_start.elapsed_time(t_end)
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)

    f_fwd = accounting.fwd_useful_flops(w.b, w.S, w.h, w.d, w.causal)
    f_bwd = accounting.bwd_useful_flops(w.b, w.S, w.h, w.d, w.causal) if have_bwd else 0.0
    step_flops = f_fwd + f_bwd
    value = job_rate(step_flops, a.steps, world, elapsed_ms)
    fwd_ms = statistics.mean(e0.elapsed_time(e1) for e0, e1, _ in ev)
    bwd_ms = statistics.mean(e1.elapsed_time(e2) for _, e1, e2 in ev) if have_bwd else 0.0
    peaks = _peaks()

    # dominant kernel: the one with the most time per step
    if have_bwd and bwd_ms > fwd_ms:
        dom, dom_ms, dom_flops, dom_src = "bwd", bwd_ms, f_bwd, "ra_bwd.cu"
    else:
        dom, dom_ms, dom_flops, dom_src = "fwd", fwd_ms, f_fwd, "ra_fwd.cu"
    achieved = dom_flops / (dom_ms / 1e3) / 1e12
    tr = TRAFFIC.get(dom)
    traffic = tr["bytes_per_launch"] if tr and tr["src_sha"] == _src_sha(dom_src) else None
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_sustained"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_sustained"],
                "traffic": traffic, "kernel": dom,
                "traffic_note": tr["method"] if tr and traffic is not None else None,
                "peak_note": f"{peaks['source']} bf16 sustained; frac of burst "
                             f"{achieved / peaks['bf16']:.3f}"}

    # end to end through the C ABI's host-buffer pipeline (ra_pipeline_*):
    # every step copies its inputs up from pinned host memory and its results
    # back inside the timed region
    e2e = None
    if not a.no_e2e:
        host = {}
        for name, t in (("q", q), ("k", k), ("v", v)) + ((("do", do),) if have_bwd else ()):
            host[name] = ra.HostBuffer(t.shape, t.dtype)
            host[name].tensor.copy_(t.cpu())
        outs = [("out", out), ("lse", lse)] + ([("dq", dq), ("dk", dk), ("dv", dv)]
                                               if have_bwd else [])
        for name, t in outs:
            host[name] = ra.HostBuffer(t.shape, t.dtype)
        h2d = sum(host[n].nbytes for n in ("q", "k", "v", "do") if n in host)
        d2h = sum(host[n].nbytes for n, _ in outs)
        pl = ra.Pipeline(w.S, w.n_shards, layout, w.causal, w.b, w.h, w.n_kv, w.d,
                         backward=have_bwd)

        def e2e_run(n_steps):
            for _ in range(n_steps):
                pl.submit(host["q"], host["k"], host["v"], host.get("do"), host["out"],
                          host["lse"], host.get("dq"), host.get("dk"), host.get("dv"))
            pl.sync()

        e2e_run(2)
        if world > 1:
            torch.distributed.barrier()
        t0 = time.perf_counter()
        e2e_run(a.steps)
        e2e_ms = (time.perf_counter() - t0) * 1e3
        e2e_ms = max_over_ranks(e2e_ms, world, dev)
        pl.close()
        for hb in host.values():
            hb.free()
        e2e = {"value": job_rate(step_flops, a.steps, world, e2e_ms), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms / a.steps,
               "host_numa_node": ra.host_numa_node(),
               "api": "ra_pipeline_submit x steps, then ra_pipeline_sync (host wall clock)",
               "schedule": "two device buffer sets, copy streams up and down: step s+1's "
                           "inputs go up and step s's results come down while step s "
                           "computes; out, lse leave while the backward runs"}

    extras = None
    if rank == 0 and not a.no_extras:
        # Side measurements: one that fails records its error instead of the
        # whole line going missing.
        def extra(fn, *args):
            try:
                return fn(*args)
            except Exception as exc:  # noqa: BLE001 - reported in the JSON line
                return {"error": f"{type(exc).__name__}: {exc}"[:300]}

        extras = extra(layout_and_imbalance_report, w, q, k, v, dev)
        extras["configs"] = extra(config_table_report, dev)
        if w.S != 65536:
            extras["imbalance_causal64k"] = extra(imbalance_at, "causal64k", dev)
        extras["exp2_roof"] = extra(exp2_roof_report, w, dev, clk)
        extras["hbm_kernels"] = extra(hbm_kernel_report, w, dev, peaks)
        extras["chunked_prefill"] = extra(prefill_report, w, q, k, v, dev)
        extras["block_steps"] = extra(block_step_report, w, q, k, v, dev)
        if have_bwd:
            extras["packed_documents"] = extra(packed_report, w, q, k, v, do, layout, dev)

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        fwd_rows, bwd_rows = 64, 16   # ~10 s of oracle work on 16 host cores
        flops, _, secs, threads, _ = _cpu_oracle_sample(w, fwd_rows, bwd_rows, seed=123)
        st_secs, st_tflops = _cpu_oracle_single_thread_tiny()
        cpu = {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": threads,
               "host_cpus": os.cpu_count(), "kind": "oracle",
               "sample": f"fp64 oracle, {fwd_rows} forward + {bwd_rows} backward random query "
                         f"rows x {w.h} heads of this workload, {secs:.1f} s",
               "extrapolated_full_step_s": secs * step_flops / flops,
               "extrapolated_note": "measured seconds x (useful FLOPs of a whole forward + "
                                    "backward step / FLOPs of the sample); not measured",
               "single_thread_tiny": {"seconds": st_secs, "tflops": st_tflops,
                                      "workload": "tiny non-causal b1 h2 kv2 d64 S1024, "
                                                  "every row, forward"}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": elapsed_ms / a.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": _workload_config(w, layout, have_bwd, world),
            "pct_of_bf16_peak": 100.0 * value / world / peaks["bf16_sustained"],
            "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
            "fwd_tflops": f_fwd / (fwd_ms / 1e3) / 1e12,
            "bwd_tflops": (f_bwd / (bwd_ms / 1e3) / 1e12) if have_bwd else None,
            "bwd_tflops_2x": (2.0 * f_fwd / (bwd_ms / 1e3) / 1e12) if have_bwd else None,
            "bwd_flops_convention": "bwd_tflops counts 2.5 x the forward's useful FLOPs (five "
                                    "GEMMs with the recomputed QK^T); bwd_tflops_2x counts 2 x "
                                    "(the pages' 'roughly twice')",
            "clocks": clk, "e2e": e2e, "gpu_launches": launches, "roofline": roofline,
            "cpu_baseline": cpu,
            "extras": extras,
        }
        print(json.dumps(line), flush=True)


def run_ring(a, rank, world, local_rank):
    """One sequence of the workload split over the ranks of a real ring:
    rank r holds shard r (the workload's placement) of Q, K, V and dO; a step
    is the ring forward and backward of ring.py, key/value blocks (and the
    backward's dK, dV) moving to the next rank over point-to-point sends
    while each rank computes with the library's block calls.  The total work
    is fixed as the ranks grow (strong scaling); `value` is the useful
    TFLOP/s of the whole sequence."""
    import torch

    from long_context_exact_gb300 import accounting, ring
    from long_context_exact_gb300 import binding as ra
    from long_context_exact_gb300 import build as lib_build
    from long_context_exact_gb300.inputs import STRIPED, WORKLOADS

    w = WORKLOADS[a.workload]
    layout = STRIPED if STRIPED in w.layouts else w.layouts[0]
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0:
        lib_build.build()
    if world > 1:
        torch.distributed.barrier()
    ra.load()
    if w.S % world != 0:
        raise SystemExit(f"S={w.S} is not a multiple of the {world} ranks")
    _, _, tok = ra.position_map(layout, w.S, world, device=dev)
    pos = tok[rank].contiguous()
    L = w.S // world
    gen = torch.Generator(device=dev).manual_seed(replica_seed(w.seed, rank))

    def rnd(*shape):
        x = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32)
        return x.mul_(w.amplitude).to(torch.bfloat16)

    q, k, v, do = rnd(w.b, L, w.h, w.d), rnd(w.b, L, w.n_kv, w.d), rnd(w.b, L, w.n_kv, w.d), \
        rnd(w.b, L, w.h, w.d)

    def step():
        out, lse = ring.ring_attention_fwd(q, k, v, pos, pos, w.causal)
        ring.ring_attention_bwd(q, k, v, out, lse, do, pos, pos, w.causal)

    for _ in range(a.warmup):
        step()
    ra.stream_check()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clk_sampler = ClockSampler(local_rank)
    clk_sampler.start()
    launches0 = ra.launch_count()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(a.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clk_sampler.stop()
    launches = ra.launch_count() - launches0
    ra.stream_check()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    flops = accounting.fwd_useful_flops(w.b, w.S, w.h, w.d, w.causal) + \
        accounting.bwd_useful_flops(w.b, w.S, w.h, w.d, w.causal)
    value = flops * a.steps / (ms / 1e3) / 1e12
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms / a.steps,
            "higher_is_better": True, "scaling": "strong", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic", "mode": "ring",
            "config": {"workload": w.name, "b": w.b, "S": w.S, "h": w.h, "n_kv": w.n_kv,
                       "d": w.d, "ring_ranks": world, "rows_per_rank": L,
                       "layout": {0: "contiguous", 1: "striped", 2: "zigzag"}[layout],
                       "causal": w.causal, "parallelism": f"ring x{world}",
                       "l2": "inputs larger than L2; no flush"},
            "pct_of_bf16_peak": 100.0 * value / world / _peaks()["bf16_sustained"],
            "clocks": clk, "gpu_launches": launches, "e2e": None, "roofline": None,
            "cpu_baseline": None,
            "note": "per step: ring forward (N block steps + finalize) and backward (N block "
                    "backward steps) with the key/value exchange over torch.distributed "
                    "point-to-point; e2e and roofline are reported by the default mode"}
        print(json.dumps(line), flush=True)


def run_block_steps(a):
    """The ring-step timings of block_step_report alone, on seeded device
    inputs of one shard's shape (the workload's seed and amplitude)."""
    import torch

    from long_context_exact_gb300 import binding as ra
    from long_context_exact_gb300.inputs import WORKLOADS

    ra.load()
    dev = torch.device("cuda", 0)
    w = WORKLOADS[a.workload]
    gen = torch.Generator(device=dev).manual_seed(w.seed)

    def rnd(*shape):
        x = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32)
        return x.mul_(w.amplitude).to(torch.bfloat16)

    L = w.S // w.n_shards
    q, k, v = rnd(w.b, L, w.h, w.d), rnd(w.b, L, w.n_kv, w.d), rnd(w.b, L, w.n_kv, w.d)
    rep = block_step_report(w, q, k, v, dev)
    print(json.dumps({"mode": "block_steps", "workload": w.name, "block_steps": rep}), flush=True)


def main():
    a = _args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if a.impl == "reference":
        run_reference(a, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        if a.block_steps:
            run_block_steps(a)
        elif a.ring:
            run_ring(a, rank, world, local_rank)
        else:
            run_ours(a, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
