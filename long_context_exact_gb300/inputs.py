"""Seeded synthetic inputs for blockwise ring attention.

This module only draws random numbers and picks sample rows; it holds none of
the method's arithmetic.  Both the CUDA path's tests and the oracle consume the
same tensors from here.

Recipe: ``torch.Generator('cpu').manual_seed(seed)``; draw float32 ``randn`` in
the order Q, K, V, dO, each shaped [b, S, heads, d] in natural token order;
multiply by the workload's amplitude (0.5 is exact in bf16); round to bf16
(round-to-nearest-even).  The workloads below have the shapes of the long
causal GQA example the third page works through (S = 262,144, h = 32,
n_kv = 8, d = 128), plus smaller cases.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

CONTIGUOUS = 0
STRIPED = 1
ZIGZAG = 2


@dataclass(frozen=True)
class Workload:
    name: str
    b: int
    S: int
    h: int
    n_kv: int
    d: int
    n_shards: int
    causal: bool
    layouts: tuple
    seed: int
    amplitude: float = 1.0
    rows_per_head: int | None = None   # None = every row
    backward: bool = False

    @property
    def L(self) -> int:
        return self.S // self.n_shards


WORKLOADS = {
    "tiny": Workload("tiny non-causal b1 h2 kv2 d64 S1024 N4", 1, 1024, 2, 2, 64, 4,
                     False, (CONTIGUOUS,), 0),
    "noncausal32k": Workload("non-causal GQA b1 h32 kv8 d128 S32768 N8", 1, 32768, 32, 8,
                             128, 8, False, (CONTIGUOUS,), 1, rows_per_head=256),
    "causal64k": Workload("causal GQA b1 h32 kv8 d128 S65536 N8", 1, 65536, 32, 8, 128, 8,
                          True, (CONTIGUOUS, STRIPED), 2, rows_per_head=512),
    "causal256k": Workload("long causal GQA b1 h32 kv8 d128 S262144 N8 striped", 1, 262144,
                           32, 8, 128, 8, True, (STRIPED,), 3, amplitude=0.5,
                           rows_per_head=256),
    # profiling-size cases: inputs still larger than L2, ~2 GB on the device;
    # with one shard of 32K rows the backward runs the same one-shard units
    # as the 256K workload (shards of 32K rows)
    "causal32k": Workload("causal GQA fwd+bwd b1 h32 kv8 d128 S32768 N8 striped", 1, 32768, 32,
                          8, 128, 8, True, (STRIPED,), 5, rows_per_head=128, backward=True),
    "causal32k1": Workload("causal GQA fwd+bwd b1 h32 kv8 d128 S32768 N1", 1, 32768, 32, 8, 128,
                           1, True, (STRIPED,), 5, rows_per_head=128, backward=True),
    # packed documents (log-uniform lengths 1K..64K) in one causal window
    "packed64k": Workload("packed causal GQA b1 h32 kv8 d128 S65536 N8 striped", 1, 65536, 32,
                          8, 128, 8, True, (STRIPED,), 6, rows_per_head=256),
    "bwd64k": Workload("causal GQA fwd+bwd b2 h32 kv8 d128 S65536 N16 striped", 2, 65536,
                       32, 8, 128, 16, True, (STRIPED,), 4, rows_per_head=128,
                       backward=True),
}


def make_inputs(b: int, S: int, h: int, n_kv: int, d: int, seed: int,
                amplitude: float = 1.0, with_dout: bool = False):
    """Q [b,S,h,d], K/V [b,S,n_kv,d] (and dO [b,S,h,d]) as bf16 CPU tensors."""
    gen = torch.Generator("cpu").manual_seed(seed)
    out = []
    for heads in (h, n_kv, n_kv) + ((h,) if with_dout else ()):
        x = torch.randn((b, S, heads, d), generator=gen, dtype=torch.float32)
        if amplitude != 1.0:
            x.mul_(amplitude)
        out.append(x.to(torch.bfloat16))
    return tuple(out)


def workload_inputs(w: Workload):
    return make_inputs(w.b, w.S, w.h, w.n_kv, w.d, w.seed, w.amplitude, w.backward)


def packed_offsets(S: int, seed: int, min_len: int = 1024, max_len: int = 65536,
                   b: int = 1) -> np.ndarray:
    """Document offsets [b, n_docs + 1] (int32) of a packed window of S
    tokens: document lengths drawn log-uniformly in [min_len, max_len]
    (seeded numpy Generator), the last one cut at S; every batch row gets its
    own draw and rows are padded with empty documents to a common count."""
    rng = np.random.default_rng(seed + 2000)
    rows = []
    for _ in range(b):
        offs = [0]
        while offs[-1] < S:
            n = int(np.exp(rng.uniform(np.log(min_len), np.log(max_len))))
            offs.append(min(S, offs[-1] + max(1, n)))
        rows.append(offs)
    n = max(len(r) for r in rows)
    return np.array([r + [S] * (n - len(r)) for r in rows], dtype=np.int32)


def sample_rows(S: int, n_shards: int, count: int | None, seed: int) -> np.ndarray:
    """Sorted token positions to check: a seeded uniform sample without
    replacement, plus rows 0, 1, L-1, L, S-1 and the first and last token of
    every shard under both placements.  ``count=None`` returns every row."""
    if count is None or count >= S:
        return np.arange(S, dtype=np.int64)
    L = S // n_shards
    rng = np.random.default_rng(seed + 1000)
    picked = set(int(x) for x in rng.choice(S, size=count, replace=False))
    forced = {0, 1, L - 1, L, S - 1}
    for p in range(n_shards):
        forced |= {p * L, p * L + L - 1, p, (L - 1) * n_shards + p}
    picked |= {t for t in forced if 0 <= t < S}
    return np.array(sorted(picked), dtype=np.int64)
