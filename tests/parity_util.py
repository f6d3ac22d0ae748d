"""Helpers shared by the GPU parity tests: which rows and keys take the
library's plain-bf16 path, error measures over them, the oracle's gradient
computed on several cores, and inputs whose attention is sharply peaked.

Test infrastructure only (it calls the oracle; the product never imports it).

Precision rule of the library (stated in ra.h): a query tile whose earliest
row sees fewer than 512 keys sends P (and dS) to the tensor cores as a bf16
pair hi + lo; every other tile rounds them once to bf16.  On the ring a row
at position t sees t + 1 keys under the causal rule and all S otherwise, so
for full-size workloads nearly all of the work is on the plain path and the
parity tests check it separately, relative to the size of the reference.
"""

from __future__ import annotations

import os
import threading

import numpy as np

SPLIT_KEYS = 512    # the library's hi + lo threshold (keys seen by a tile's earliest row)
TILE = 128          # query rows per tile

# Measured errors per test, written out at the end of the session when
# RA_PARITY_REPORT names a file (tests/conftest.py).
RECORDS: dict = {}


def record(prefix: str = "", **errs) -> None:
    """Keep the measured errors of the running test under its node id."""
    name = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    RECORDS.setdefault(name, {}).update({prefix + k: float(v) for k, v in errs.items()})


def plain_rows(orc, layout: int, S: int, N: int, causal: bool) -> np.ndarray:
    """Boolean [S] over token positions: True where the token's query tile
    takes the plain bf16 path."""
    if not causal:
        return np.full(S, S >= SPLIT_KEYS)
    _, _, tok = orc.position_map(layout, S, N)
    L = S // N
    out = np.zeros(S, dtype=bool)
    for i in range(N):
        for a0 in range(0, L, TILE):
            rows = tok[i, a0:min(L, a0 + TILE)]
            out[rows] = int(tok[i, a0]) + 1 >= SPLIT_KEYS
    return out


def plain_only_keys(orc, layout: int, S: int, N: int, causal: bool) -> np.ndarray:
    """Boolean [S] over key positions: True where every query that sees the
    key is on the plain path, so the key's dK and dV come from plain steps
    only.  A causal key j is seen by the queries t >= j."""
    pr = plain_rows(orc, layout, S, N, causal)
    if not causal:
        return pr.copy() if pr.all() else np.zeros(S, dtype=bool)
    split_tokens = np.nonzero(~pr)[0]
    last_split = int(split_tokens.max()) if split_tokens.size else -1
    return np.arange(S) > last_split


def max_abs(a, r) -> float:
    return float(np.abs(np.asarray(a) - np.asarray(r)).max()) if np.size(r) else 0.0


def rel_to_max(a, r) -> tuple[float, float]:
    """(max |a - r| / max |r|, max |r|) -- the error relative to the size of
    the reference, so that a tiny reference cannot hide a wrong result."""
    r = np.asarray(r)
    if r.size == 0:
        return 0.0, 0.0
    ref = float(np.abs(r).max())
    err = float(np.abs(np.asarray(a) - r).max())
    return (err / ref if ref > 0 else (0.0 if err == 0 else np.inf)), ref


def bwd_oracle_parallel(orc, q, k, v, dout, causal: bool, rows=None, scale=None,
                        cu_seqlens=None, workers: int | None = None):
    """The oracle's analytic gradient with dO kept on ``rows`` (all rows by
    default), computed as a sum over disjoint row subsets run concurrently.

    Gradients are linear in dO: the gradient for dO restricted to a set of
    rows is the sum of the gradients for dO restricted to the parts of any
    partition of it.  dq rows come from the part that holds them; dk and dv
    are the fp64 sums of the parts'.  Each part is one unchanged oracle call
    (the oracle parallelises over (batch, KV head) only), run on its own
    thread (ctypes releases the interpreter lock) with as many OpenMP
    threads as there are (batch, KV head) tasks."""
    b, S = q.shape[0], q.shape[1]
    n_kv = k.shape[2]
    rows = np.arange(S, dtype=np.int64) if rows is None else np.asarray(rows, np.int64)
    cores = os.cpu_count() or 1
    tasks = max(1, b * n_kv)
    if workers is None:
        workers = max(1, cores // tasks)
    workers = max(1, min(workers, rows.size))
    # interleaved parts: under the causal rule a row's cost grows with its position
    parts = [rows[w::workers] for w in range(workers)]
    results = [None] * workers
    errors = []

    def run(w):
        try:
            orc.set_threads(min(tasks, cores))
            results[w] = orc.attn_bwd_rows(q, k, v, dout, causal, scale=scale, rows=parts[w],
                                           cu_seqlens=cu_seqlens)
        except BaseException as e:   # re-raised on the calling thread
            errors.append(e)

    threads = [threading.Thread(target=run, args=(w,)) for w in range(workers)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    if errors:
        raise errors[0]
    h, d = q.shape[2], q.shape[3]
    dq = np.empty((b, rows.size, h, d))
    pos = {int(t): n for n, t in enumerate(rows)}
    dk = np.zeros((b, S, n_kv, d))
    dv = np.zeros((b, S, n_kv, d))
    for w in range(workers):
        pq, pk, pv = results[w]
        dq[:, [pos[int(t)] for t in parts[w]]] = pq
        dk += pk
        dv += pv
    return dq, dk, dv


def peak_targets(orc, layout: int, S: int, N: int, causal: bool) -> np.ndarray:
    """For every query token t, the key the peaked inputs align with it: in
    the last shard of t's ring order (shard (i - s) mod N for s = N-1 down to
    0) that holds a key t may see, the key at t's own local row, or when that
    row is not visible one counted down from the latest visible row by how
    far t's row lies beyond it.  At s = 0 the shard is
    t's own, where t sees itself, so every token gets a target (itself when
    no other shard holds a visible key).  Returns int64 [S] key positions."""
    shard, local, tok = orc.position_map(layout, S, N)
    L = S // N
    target = np.full(S, -1, dtype=np.int64)
    t_all = np.arange(S)
    for s in range(N - 1, -1, -1):
        todo = target < 0
        if not todo.any():
            break
        t = t_all[todo]
        i = shard[t].astype(np.int64)
        p = (i - s) % N
        if causal:
            # positions increase with the local row in every layout
            last = np.empty(t.shape, dtype=np.int64)
            for pp in np.unique(p):
                sel = p == pp
                last[sel] = np.searchsorted(tok[pp], t[sel], side="right") - 1
        else:
            last = np.full(t.shape, L - 1, dtype=np.int64)
        lo = local[t].astype(np.int64)
        ok = last >= 0
        # t's own local row when visible, else counted down from the latest
        # visible row (so that targets stay spread over the visible rows)
        row = np.where(lo <= last, lo, last - np.mod(lo - last - 1, np.maximum(last + 1, 1)))
        target[t[ok]] = tok[p[ok], row[ok]]
    return target


def peaked_inputs(orc, b: int, S: int, h: int, n_kv: int, d: int, N: int, layout: int,
                  causal: bool, seed: int, alpha=(0.6, 1.6), with_dout: bool = False):
    """Q, K, V (and dO) i.i.d. N(0,1) as make_inputs draws them, then, for
    every key that is some query's target (``peak_targets``), K replaced per
    KV head kh by alpha * (sum of the targeting queries' rows of query head
    kh * g + t mod g) / sqrt(their count), alpha drawn per key uniformly from
    the given range (seeded), rounded to bf16.

    A query aligned with its own key scores about alpha * sqrt(d) above zero
    (11 to 18 natural-log units at d = 128 for a single query per key), far
    above its other scores, so its row max jumps when the ring reaches that
    key late in its order -- by more than 8 log2 units in most rows."""
    import torch

    from long_context_exact_gb300.inputs import make_inputs
    t_in = make_inputs(b, S, h, n_kv, d, seed, with_dout=with_dout)
    q, k = t_in[0], t_in[1].clone()
    g = h // n_kv
    target = peak_targets(orc, layout, S, N, causal)
    rng = np.random.default_rng(seed + 3000)
    a_key = rng.uniform(alpha[0], alpha[1], size=S)
    qf = q.float()
    kf = k.float()
    tq = np.nonzero(target >= 0)[0]
    keys = target[tq]
    counts = np.bincount(keys, minlength=S).astype(np.float64)
    acc = torch.zeros((b, S, n_kv, d), dtype=torch.float32)
    for kh in range(n_kv):
        hsel = torch.from_numpy(kh * g + (tq % g))
        rows_q = qf[:, torch.from_numpy(tq), :, :]                    # [b, T, h, d]
        pick = rows_q[:, torch.arange(tq.size), hsel, :]              # [b, T, d]
        acc[:, :, kh, :].index_add_(1, torch.from_numpy(keys), pick)
    used = counts > 0
    scale_k = np.zeros(S)
    scale_k[used] = a_key[used] / np.sqrt(counts[used])
    sk = torch.from_numpy(scale_k).float()[None, :, None, None]
    mask = torch.from_numpy(used)[None, :, None, None]
    kf = torch.where(mask, acc * sk, kf)
    k = kf.to(torch.bfloat16)
    return (q, k) + tuple(t_in[2:])
