"""Python face of the fp64 CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: the product path never imports this module.  Only
the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.  It shares no code with the CUDA library.

Inputs are bfloat16 tensors (widened exactly to float64) or float64 arrays;
every result is a float64 numpy array.  Function-level docstrings name the passage of the
pages each routine restates; the C file holds the arithmetic.

Parity status: every routine here is pinned by a ``-m "not gpu"`` test against
something other than itself (brute-force matrices, library routines, closed
forms, invariants, finite differences, or values printed on the pages).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_SRC = os.path.join(_HERE, "oracle.c")
_lock = threading.Lock()
_lib = None

CONTIGUOUS = 0
STRIPED = 1
ZIGZAG = 2


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` with gcc (-O2, OpenMP, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.orc_position_map.argtypes = [i32, i64, i32, P, P, P]
            lib.orc_position_map.restype = i32
            lib.orc_ring_order.argtypes = [i32, P]
            lib.orc_ring_order.restype = None
            lib.orc_attn_fwd_rows.argtypes = [P, P, P, i32, i64, i32, i32, i32,
                                              i32, dbl, P, i64, P, P, P, P]
            lib.orc_attn_fwd_rows.restype = None
            lib.orc_attn_bwd_rows.argtypes = [P, P, P, P, i32, i64, i32, i32,
                                              i32, i32, dbl, P, i64, P, P, P, P, P]
            lib.orc_attn_bwd_rows.restype = None
            lib.orc_block_update.argtypes = [P, P, P, P, P, i32, i64, i64, i32,
                                             i32, i32, i32, dbl, P, P, P]
            lib.orc_block_update.restype = None
            lib.orc_finalize.argtypes = [P, P, P, i32, i64, i32, i32, P, P]
            lib.orc_finalize.restype = None
            lib.orc_merge.argtypes = [P, P, P, P, i32, i64, i32, i32, P, P]
            lib.orc_merge.restype = None
            lib.orc_max_threads.argtypes = []
            lib.orc_max_threads.restype = i32
            lib.orc_set_threads.argtypes = [i32]
            lib.orc_set_threads.restype = None
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Exact float64 copy of a bf16/float tensor or array (C-contiguous)."""
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(x, dtype=np.float64)
    import torch
    return np.ascontiguousarray(x.detach().cpu().to(torch.float64).numpy())


def _gather_rows(x, rows: np.ndarray) -> np.ndarray:
    """x[:, rows] widened to float64 without widening the whole tensor."""
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(x[:, rows], dtype=np.float64)
    import torch
    idx = torch.from_numpy(np.ascontiguousarray(rows, np.int64))
    return _f64(x.detach().cpu().index_select(1, idx))


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def default_scale(d: int) -> float:
    """1/sqrt(d), the scale of the attention definition on the first page."""
    return 1.0 / float(np.sqrt(d))


# --------------------------------------------------------------------------
def position_map(layout: int, S: int, N: int):
    """Token placement (contiguous / striped / zig-zag), third page section 6
    and the first page's "Striped Attention" and "Zig-Zag Ring Attention".
    Returns (shard_of[S], local_of[S], token_of[N, S//N]) as int32."""
    lib = _load()
    shard = np.empty(S, np.int32)
    local = np.empty(S, np.int32)
    tok = np.empty(S, np.int32)
    rc = lib.orc_position_map(layout, S, N, _ptr(shard), _ptr(local), _ptr(tok))
    if rc != 0:
        raise ValueError("invalid position map arguments")
    return shard, local, tok.reshape(N, S // N if N else 0)


def ring_order(N: int) -> np.ndarray:
    """order[i, s] = KV shard visited by query shard i at ring step s,
    (i - s) mod N (fourth page, "The Ring Communication Protocol")."""
    lib = _load()
    out = np.empty(N * N, np.int32)
    lib.orc_ring_order(N, _ptr(out))
    return out.reshape(N, N)


def max_threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return int(_load().orc_max_threads())


def set_threads(n: int) -> None:
    """Set the OpenMP thread count of later oracle calls (timing only)."""
    _load().orc_set_threads(int(n))


def doc_bounds(cu_seqlens, S: int):
    """Per-token document bounds from packed-document offsets.
    cu_seqlens [b, n_docs + 1] (non-decreasing, from 0 to S): token t of
    batch row bb belongs to the document [cu[d], cu[d+1]) containing it.
    Returns (doc_start, doc_end) as int64 [b, S]."""
    cu = np.asarray(cu_seqlens, np.int64)
    if cu.ndim == 1:
        cu = cu[None]
    starts = np.empty((cu.shape[0], S), np.int64)
    ends = np.empty((cu.shape[0], S), np.int64)
    for bb in range(cu.shape[0]):
        assert cu[bb, 0] == 0 and cu[bb, -1] == S and np.all(np.diff(cu[bb]) >= 0)
        lens = np.diff(cu[bb])
        starts[bb] = np.repeat(cu[bb, :-1], lens)
        ends[bb] = np.repeat(cu[bb, 1:], lens)
    return starts, ends


def _docs(cu_seqlens, b: int, S: int):
    if cu_seqlens is None:
        return None, None, None, None
    ds, de = doc_bounds(cu_seqlens, S)
    if ds.shape[0] == 1 and b > 1:
        ds, de = np.repeat(ds, b, axis=0), np.repeat(de, b, axis=0)
    ds, de = np.ascontiguousarray(ds), np.ascontiguousarray(de)
    return ds, de, _ptr(ds), _ptr(de)


def attn_fwd_rows(q, k, v, causal: bool, scale: float | None = None, rows=None,
                  cu_seqlens=None):
    """Direct definition softmax(scale*QK^T)V with the causal rule and GQA
    sharing, on the listed query rows (natural token order).  With
    cu_seqlens (packed documents) a token sees only keys of its document.

    q [b,S,h,d], k/v [b,S,n_kv,d] (bf16 tensors or float arrays).
    Returns out [b,R,h,d], lse [b,h,R] as float64."""
    lib = _load()
    b, S, h, d = q.shape
    n_kv = k.shape[2]
    assert h % n_kv == 0
    if scale is None:
        scale = default_scale(d)
    rows = np.arange(S, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    R = rows.shape[0]
    qr, kd, vd = _gather_rows(q, rows), _f64(k), _f64(v)
    out = np.empty((b, R, h, d), np.float64)
    lse = np.empty((b, h, R), np.float64)
    ds, de, pds, pde = _docs(cu_seqlens, b, S)
    lib.orc_attn_fwd_rows(_ptr(qr), _ptr(kd), _ptr(vd), b, S, h, n_kv, d,
                          int(bool(causal)), float(scale), _ptr(rows), R,
                          _ptr(out), _ptr(lse), pds, pde)
    return out, lse


def attn_bwd_rows(q, k, v, dout, causal: bool, scale: float | None = None, rows=None,
                  cu_seqlens=None):
    """Analytic gradient of the direct definition with dO restricted to the
    listed rows.  Returns dq_rows [b,R,h,d], dk [b,S,n_kv,d], dv [b,S,n_kv,d]."""
    lib = _load()
    b, S, h, d = q.shape
    n_kv = k.shape[2]
    if scale is None:
        scale = default_scale(d)
    rows = np.arange(S, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    R = rows.shape[0]
    qr, gr = _gather_rows(q, rows), _gather_rows(dout, rows)
    kd, vd = _f64(k), _f64(v)
    dq = np.empty((b, R, h, d), np.float64)
    dk = np.empty((b, S, n_kv, d), np.float64)
    dv = np.empty((b, S, n_kv, d), np.float64)
    ds, de, pds, pde = _docs(cu_seqlens, b, S)
    lib.orc_attn_bwd_rows(_ptr(qr), _ptr(kd), _ptr(vd), _ptr(gr), b, S, h, n_kv,
                          d, int(bool(causal)), float(scale), _ptr(rows), R,
                          _ptr(dq), _ptr(dk), _ptr(dv), pds, pde)
    return dq, dk, dv


def new_state(b: int, Lq: int, h: int, d: int):
    """Initial online-softmax state: m = -inf, l = 0, O = 0."""
    return (np.full((b, h, Lq), -np.inf), np.zeros((b, h, Lq)),
            np.zeros((b, Lq, h, d)))


def block_update(q, k, v, q_pos, k_pos, causal: bool, scale: float, state):
    """One online-softmax update of (m, l, O) in place with one K/V block.
    q [b,Lq,h,d], k/v [b,Lk,n_kv,d]; q_pos [Lq], k_pos [Lk] token positions."""
    lib = _load()
    qd, kd, vd = _f64(q), _f64(k), _f64(v)
    b, Lq, h, d = qd.shape
    Lk, n_kv = kd.shape[1], kd.shape[2]
    qp = np.ascontiguousarray(q_pos, np.int32)
    kp = np.ascontiguousarray(k_pos, np.int32)
    m, l, o = state
    for a in (m, l, o):
        assert a.dtype == np.float64 and a.flags.c_contiguous
    lib.orc_block_update(_ptr(qd), _ptr(kd), _ptr(vd), _ptr(qp), _ptr(kp), b,
                         Lq, Lk, h, n_kv, d, int(bool(causal)), float(scale),
                         _ptr(m), _ptr(l), _ptr(o))
    return state


def finalize(state):
    """O* = O / l, LSE = m + ln l.  Returns (out [b,Lq,h,d], lse [b,h,Lq])."""
    lib = _load()
    m, l, o = state
    b, Lq, h, d = o.shape
    out = np.empty_like(o)
    lse = np.empty_like(m)
    lib.orc_finalize(_ptr(o), _ptr(l), _ptr(m), b, Lq, h, d, _ptr(out), _ptr(lse))
    return out, lse


def merge(o_a, lse_a, o_b, lse_b):
    """Rescale-merge of two normalised partial results over disjoint keys."""
    lib = _load()
    arrs = [np.ascontiguousarray(x, np.float64) for x in (o_a, lse_a, o_b, lse_b)]
    b, Lq, h, d = arrs[0].shape
    o = np.empty_like(arrs[0])
    lse = np.empty_like(arrs[1])
    lib.orc_merge(_ptr(arrs[0]), _ptr(arrs[1]), _ptr(arrs[2]), _ptr(arrs[3]),
                  b, Lq, h, d, _ptr(o), _ptr(lse))
    return o, lse


def ring_blockwise_forward(q, k, v, n_shards: int, layout: int, causal: bool,
                           scale: float | None = None, order=None):
    """The pages' ring schedule on one machine: query shard i keeps its rows and
    meets KV shard (i - s) mod N at step s (or order[i, s] if given), updating
    (m, l, O) with ``block_update``; then ``finalize``.

    Returns (out [b,S,h,d], lse [b,h,S]) in natural token order."""
    qd, kd, vd = _f64(q), _f64(k), _f64(v)
    b, S, h, d = qd.shape
    if scale is None:
        scale = default_scale(d)
    _, _, token_of = position_map(layout, S, n_shards)
    order = ring_order(n_shards) if order is None else np.asarray(order)
    out = np.empty((b, S, h, d))
    lse = np.empty((b, h, S))
    for i in range(n_shards):
        qt = token_of[i]
        state = new_state(b, qt.shape[0], h, d)
        qi = np.ascontiguousarray(qd[:, qt])
        for s in range(n_shards):
            kt = token_of[int(order[i, s])]
            block_update(qi, np.ascontiguousarray(kd[:, kt]),
                         np.ascontiguousarray(vd[:, kt]), qt, kt, causal, scale,
                         state)
        o_i, lse_i = finalize(state)
        out[:, qt] = o_i
        lse[:, :, qt] = lse_i
    return out, lse
