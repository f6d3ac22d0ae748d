"""FLOP and byte accounting for reporting (host logic, no arithmetic of the
method itself).

- Useful forward FLOPs: 4 b S^2 h d non-causal (two GEMMs, 2 FLOPs per
  multiply-add), half of that, 2 b S^2 h d, causal -- the third page's
  section 2, first invariant.
- Useful backward FLOPs: 2.5 x forward (five GEMMs per tile, counting the
  recomputation of Q K^T); the fourth page's "roughly twice" figure is
  reported next to it.
- Causal load-balance model of the third page's section 6: contiguous shards
  give device i work proportional to i + 1 and utilisation (N + 1) / 2N, or
  N / (2N - 1) with the diagonal block counted as half.
- Per-device received bytes (second invariant): (N - 1)/N * b S 2 n_kv d p;
  per-step arithmetic intensity I_step = (h / n_kv) S / N.
"""

from __future__ import annotations


def fwd_useful_flops(b: int, S: int, h: int, d: int, causal: bool) -> float:
    f = 4.0 * b * float(S) * float(S) * h * d
    return f / 2 if causal else f


def bwd_useful_flops(b: int, S: int, h: int, d: int, causal: bool) -> float:
    return 2.5 * fwd_useful_flops(b, S, h, d, causal)


def causal_utilisation_contiguous(N: int, half_diagonal: bool = False) -> float:
    return N / (2 * N - 1) if half_diagonal else (N + 1) / (2 * N)


def ring_step_flops(b: int, S: int, N: int, h: int, d: int) -> float:
    """FLOPs of one (query shard, KV shard) pair, non-causal: 4 b L^2 h d."""
    L = S / N
    return 4.0 * b * L * L * h * d


def ring_step_kv_bytes(b: int, S: int, N: int, n_kv: int, d: int, p: int = 2) -> float:
    """Bytes of one K/V shard: b L 2 n_kv d p."""
    return b * (S / N) * 2 * n_kv * d * p


def received_bytes(b: int, S: int, N: int, n_kv: int, d: int, p: int = 2) -> float:
    return (N - 1) / N * b * S * 2 * n_kv * d * p


def step_intensity(S: int, N: int, h: int, n_kv: int) -> float:
    return (h / n_kv) * S / N


def fwd_algorithmic_bytes(b: int, S: int, h: int, n_kv: int, d: int) -> float:
    """Compulsory HBM bytes of one forward: read Q, K, V (bf16), write O (fp32)
    and LSE (fp32)."""
    return b * S * (h * d * 2 + 2 * n_kv * d * 2 + h * d * 4 + h * 4)
