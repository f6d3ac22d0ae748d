"""ctypes binding of the C ABI in ``include/ra.h`` (argument marshalling only).

Every call passes ``tensor.data_ptr()`` and the current CUDA stream to the
library; all arithmetic runs in the library's kernels.  There is no fallback:
if the shared library is missing or cannot load, calls raise ``RAError``.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

from .inputs import CONTIGUOUS, STRIPED, ZIGZAG  # noqa: F401  (re-exported layout ids)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libra.so")

RA_OK = 0
RA_ERR_INVALID_ARG = 1
RA_ERR_UNSUPPORTED = 2
RA_ERR_CUDA = 3
RA_ERR_DEVICE_TIMEOUT = 4
RA_ERR_WORKSPACE = 5

_STATUS_NAMES = {0: "RA_OK", 1: "RA_ERR_INVALID_ARG", 2: "RA_ERR_UNSUPPORTED", 3: "RA_ERR_CUDA",
                 4: "RA_ERR_DEVICE_TIMEOUT", 5: "RA_ERR_WORKSPACE"}


class RAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int), ("h", ctypes.c_int), ("n_kv", ctypes.c_int),
                ("d", ctypes.c_int)]


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load the C-ABI library (once) and declare every entry point."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise RAError(RA_ERR_CUDA, f"library not built: {path} (run __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        P, I, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        sig = {
            "ra_block_step": [P, P, P, P, P, P, P, P, I64, I64, Dims, I, F, P],
            "ra_finalize": [P, P, P, P, I64, Dims, P],
            "ra_merge": [P, P, P, P, P, P, I64, Dims, P],
            "ra_ring_attention": [P, P, P, P, P, I64, I, I, I, F, Dims, P],
            "ra_ring_attention_packed": [P, P, P, P, P, I64, I, I, I, F, Dims, P, I, P],
            "ra_ring_attention_packed_bwd": [P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, I64,
                                             I, I, I, F, Dims, P, I, P],
            "ra_ring_attention_bwd": [P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, I64, I, I, I,
                                      F, Dims, P],
            "ra_block_step_bwd": [P, P, P, P, P, P, P, P, P, P, P, I64, I64, Dims, I, F, P,
                                  ctypes.c_size_t, P],
            "ra_position_map": [I, I64, I, P, P, P, P],
            "ra_ring_order": [I, P, P],
            "ra_stream_check": [P],
            "ra_selftest_wait_timeout": [ctypes.c_longlong, P],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = I
        lib.ra_ring_attention_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, P, I64, I, I, I, F,
                                                      Dims, P]
        lib.ra_ring_attention_bwd_noalloc.restype = I
        lib.ra_prefill_workspace_size.argtypes = [I64, I64, I, Dims]
        lib.ra_prefill_workspace_size.restype = ctypes.c_size_t
        lib.ra_chunked_prefill.argtypes = [P, P, P, P, P, P, P, I64, I64, I, Dims, I, F, P,
                                           ctypes.c_size_t, P]
        lib.ra_chunked_prefill.restype = I
        lib.ra_bwd_workspace_size.argtypes = [I64, I, Dims]
        lib.ra_bwd_workspace_size.restype = ctypes.c_size_t
        lib.ra_block_bwd_workspace_size.argtypes = [I64, Dims]
        lib.ra_block_bwd_workspace_size.restype = ctypes.c_size_t
        lib.ra_last_error.argtypes = []
        lib.ra_last_error.restype = ctypes.c_char_p
        lib.ra_version.argtypes = []
        lib.ra_version.restype = I
        lib.ra_ex2_probe.argtypes = [I64, P, I64, P]
        lib.ra_ex2_probe.restype = I
        lib.ra_ex2_probe_threads.argtypes = []
        lib.ra_ex2_probe_threads.restype = I64
        lib.ra_launch_count.argtypes = []
        lib.ra_launch_count.restype = ctypes.c_uint64
        lib.ra_host_alloc.argtypes = [ctypes.c_size_t, ctypes.POINTER(P)]
        lib.ra_host_alloc.restype = I
        lib.ra_host_free.argtypes = [P]
        lib.ra_host_free.restype = I
        lib.ra_host_numa_node.argtypes = []
        lib.ra_host_numa_node.restype = I
        lib.ra_pipeline_create.argtypes = [I64, I, I, I, F, Dims, I, ctypes.POINTER(P)]
        lib.ra_pipeline_create.restype = I
        lib.ra_pipeline_submit.argtypes = [P, P, P, P, P, P, P, P, P, P]
        lib.ra_pipeline_submit.restype = I
        lib.ra_pipeline_sync.argtypes = [P]
        lib.ra_pipeline_sync.restype = I
        lib.ra_pipeline_destroy.argtypes = [P]
        lib.ra_pipeline_destroy.restype = I
        _lib = lib
        return lib


def _check(status: int):
    if status != RA_OK:
        msg = load().ra_last_error().decode(errors="replace")
        raise RAError(status, msg)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dims(b, h, n_kv, d) -> Dims:
    return Dims(int(b), int(h), int(n_kv), int(d))


def _need(t, dtype, name):
    if t.dtype != dtype:
        raise RAError(RA_ERR_INVALID_ARG, f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise RAError(RA_ERR_INVALID_ARG, f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise RAError(RA_ERR_INVALID_ARG, f"{name} must be contiguous")


def _bits(t):
    return t.view(torch.int16)


# ---------------------------------------------------------------- forward
def _docs(cu_seqlens, b):
    """(pointer, n_docs) of packed-document offsets as int32 [b, n_docs + 1]."""
    if cu_seqlens is None:
        return None, 0, None
    _need(cu_seqlens, torch.int32, "cu_seqlens")
    cu = cu_seqlens if cu_seqlens.dim() == 2 else cu_seqlens.unsqueeze(0).expand(b, -1)
    cu = cu.contiguous()
    if cu.shape[0] != b:
        raise RAError(RA_ERR_INVALID_ARG, "cu_seqlens needs one row per batch row")
    return _ptr(cu), cu.shape[1] - 1, cu


def ring_attention(q, k, v, n_shards: int, layout: int = STRIPED, causal: bool = True,
                   scale: float = 0.0, out=None, lse=None, stream=None, cu_seqlens=None):
    """Exact attention over N virtual shards in ring order (one fused launch).
    q [b,S,h,d], k/v [b,S,n_kv,d] bf16 CUDA tensors in natural token order.
    cu_seqlens (int32 [b, n_docs+1] or [n_docs+1]): packed documents.
    Returns (out [b,S,h,d] float32, lse [b,h,S] float32)."""
    lib = load()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    b, S, h, d = q.shape
    n_kv = k.shape[2]
    if out is None:
        out = torch.empty((b, S, h, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((b, h, S), dtype=torch.float32, device=q.device)
    _need(out, torch.float32, "out")
    _need(lse, torch.float32, "lse")
    cu_p, n_docs, _keep = _docs(cu_seqlens, b)
    if cu_p is None:
        _check(lib.ra_ring_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), S,
                                     int(n_shards), int(layout), int(bool(causal)), float(scale),
                                     _dims(b, h, n_kv, d), _stream(stream)))
    else:
        _check(lib.ra_ring_attention_packed(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), S,
                                            int(n_shards), int(layout), int(bool(causal)),
                                            float(scale), _dims(b, h, n_kv, d), cu_p, n_docs,
                                            _stream(stream)))
    return out, lse


def new_state(b: int, Lq: int, h: int, d: int, device):
    """Fresh online-softmax state (m = -inf, l = 0, o = 0) on the device."""
    m = torch.full((b, h, Lq), float("-inf"), dtype=torch.float32, device=device)
    l = torch.zeros((b, h, Lq), dtype=torch.float32, device=device)
    o = torch.zeros((b, Lq, h, d), dtype=torch.float32, device=device)
    return m, l, o


def block_step(q, k, v, state, q_pos=None, k_pos=None, causal: bool = False,
               scale: float = 0.0, stream=None):
    """Fold one K/V block into (m, l, o) in place (one ring step)."""
    lib = load()
    m, l, o = state
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    for t, n in ((m, "m"), (l, "l"), (o, "o")):
        _need(t, torch.float32, n)
    if causal:
        _need(q_pos, torch.int32, "q_pos")
        _need(k_pos, torch.int32, "k_pos")
    b, Lq, h, d = q.shape
    Lk, n_kv = k.shape[1], k.shape[2]
    _check(lib.ra_block_step(_ptr(q), _ptr(k), _ptr(v), _ptr(m), _ptr(l), _ptr(o),
                             _ptr(q_pos) if causal else None, _ptr(k_pos) if causal else None,
                             Lq, Lk, _dims(b, h, n_kv, d), int(bool(causal)), float(scale),
                             _stream(stream)))
    return state


def finalize(state, lse=None, stream=None):
    """o <- o / l in place; returns (o, lse) with lse = m + ln l."""
    lib = load()
    m, l, o = state
    b, Lq, h, d = o.shape
    if lse is None:
        lse = torch.empty_like(m)
    _check(lib.ra_finalize(_ptr(o), _ptr(l), _ptr(m), _ptr(lse), Lq, _dims(b, h, 1, d),
                           _stream(stream)))
    return o, lse


def merge(o_a, lse_a, o_b, lse_b, o=None, lse=None, stream=None):
    """Rescale-merge of two normalised partial results over disjoint keys."""
    lib = load()
    b, Lq, h, d = o_a.shape
    o = torch.empty_like(o_a) if o is None else o
    lse = torch.empty_like(lse_a) if lse is None else lse
    for t, n in ((o_a, "o_a"), (lse_a, "lse_a"), (o_b, "o_b"), (lse_b, "lse_b"), (o, "o"),
                 (lse, "lse")):
        _need(t, torch.float32, n)
    _check(lib.ra_merge(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), _ptr(o), _ptr(lse), Lq,
                        _dims(b, h, 1, d), _stream(stream)))
    return o, lse


# ---------------------------------------------------------------- backward
def prefill_workspace_size(Lq: int, Lk: int, n_splits: int, b: int, h: int, n_kv: int,
                           d: int) -> int:
    return int(load().ra_prefill_workspace_size(Lq, Lk, n_splits, _dims(b, h, n_kv, d)))


def chunked_prefill(q, k, v, q_pos=None, k_pos=None, causal: bool = True, scale: float = 0.0,
                    n_splits: int = 0, out=None, lse=None, workspace=None, stream=None):
    """Lq new queries against Lk resident keys with the keys split over
    concurrent block steps; returns (out [b,Lq,h,d] float, lse [b,h,Lq])."""
    lib = load()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    b, Lq, h, d = q.shape
    Lk, n_kv = k.shape[1], k.shape[2]
    out = torch.empty((b, Lq, h, d), dtype=torch.float32, device=q.device) if out is None else out
    lse = torch.empty((b, h, Lq), dtype=torch.float32, device=q.device) if lse is None else lse
    if workspace is None:
        nbytes = prefill_workspace_size(Lq, Lk, n_splits, b, h, n_kv, d)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    for t, n in ((q_pos, "q_pos"), (k_pos, "k_pos")):
        if t is not None:
            _need(t, torch.int32, n)
    _check(lib.ra_chunked_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                  _ptr(q_pos) if q_pos is not None else None,
                                  _ptr(k_pos) if k_pos is not None else None, Lq, Lk, n_splits,
                                  _dims(b, h, n_kv, d), 1 if causal else 0, scale,
                                  _ptr(workspace), workspace.numel(), _stream(stream)))
    return out, lse


def bwd_workspace_size(S: int, n_shards: int, b: int, h: int, n_kv: int, d: int) -> int:
    return int(load().ra_bwd_workspace_size(S, int(n_shards), _dims(b, h, n_kv, d)))


def ring_attention_bwd(q, k, v, out, lse, dout, n_shards: int, layout: int = STRIPED,
                       causal: bool = True, scale: float = 0.0, dq=None, dk=None, dv=None,
                       workspace=None, stream=None, cu_seqlens=None):
    """Gradients (dq, dk, dv) as float32, recomputing P from the saved LSE."""
    lib = load()
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (dout, "dout")):
        _need(t, torch.bfloat16, n)
    for t, n in ((out, "out"), (lse, "lse")):
        _need(t, torch.float32, n)
    b, S, h, d = q.shape
    n_kv = k.shape[2]
    dq = torch.empty((b, S, h, d), dtype=torch.float32, device=q.device) if dq is None else dq
    dk = torch.empty((b, S, n_kv, d), dtype=torch.float32, device=q.device) if dk is None else dk
    dv = torch.empty((b, S, n_kv, d), dtype=torch.float32, device=q.device) if dv is None else dv
    ws_bytes = bwd_workspace_size(S, n_shards, b, h, n_kv, d)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    cu_p, n_docs, _keep = _docs(cu_seqlens, b)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
            _ptr(dv), _ptr(workspace), workspace.numel() * workspace.element_size(), S,
            int(n_shards), int(layout), int(bool(causal)), float(scale), _dims(b, h, n_kv, d))
    if cu_p is None:
        _check(lib.ra_ring_attention_bwd(*args, _stream(stream)))
    else:
        _check(lib.ra_ring_attention_packed_bwd(*args, cu_p, n_docs, _stream(stream)))
    return dq, dk, dv


def block_bwd_workspace_size(Lq: int, b: int, h: int, n_kv: int, d: int) -> int:
    return int(load().ra_block_bwd_workspace_size(Lq, _dims(b, h, n_kv, d)))


def block_step_bwd(q, k, v, out, lse, dout, grads, q_pos=None, k_pos=None,
                   causal: bool = False, scale: float = 0.0, workspace=None, stream=None):
    """One ring step of the backward: ADD the contribution of the key/value
    block (k, v) to grads = (dq [b,Lq,h,d], dk, dv [b,Lk,n_kv,d]) float32,
    given the query rows' whole-sequence out / lse.  Returns grads."""
    lib = load()
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (dout, "dout")):
        _need(t, torch.bfloat16, n)
    dq, dk, dv = grads
    for t, n in ((out, "out"), (lse, "lse"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        _need(t, torch.float32, n)
    if causal:
        _need(q_pos, torch.int32, "q_pos")
        _need(k_pos, torch.int32, "k_pos")
    b, Lq, h, d = q.shape
    Lk, n_kv = k.shape[1], k.shape[2]
    ws_bytes = block_bwd_workspace_size(Lq, b, h, n_kv, d)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    _check(lib.ra_block_step_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
        _ptr(dv), _ptr(q_pos) if causal else None, _ptr(k_pos) if causal else None, Lq, Lk,
        _dims(b, h, n_kv, d), int(bool(causal)), float(scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return grads


def ring_attention_bwd_noalloc(q, k, v, out, lse, dout, n_shards: int, layout: int = STRIPED,
                               causal: bool = True, scale: float = 0.0, dq=None, dk=None,
                               dv=None, stream=None):
    """The backward with the library's fixed scratch array instead of a
    workspace (for callers that cannot allocate device memory at this point;
    see ra_ring_attention_bwd_noalloc in include/ra.h)."""
    lib = load()
    b, S, h, d = q.shape
    n_kv = k.shape[2]
    dq = torch.empty((b, S, h, d), dtype=torch.float32, device=q.device) if dq is None else dq
    dk = torch.empty((b, S, n_kv, d), dtype=torch.float32, device=q.device) if dk is None else dk
    dv = torch.empty((b, S, n_kv, d), dtype=torch.float32, device=q.device) if dv is None else dv
    _check(lib.ra_ring_attention_bwd_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
        _ptr(dv), S, int(n_shards), int(layout), int(bool(causal)), float(scale),
        _dims(b, h, n_kv, d), _stream(stream)))
    return dq, dk, dv


# ---------------------------------------------------------------- maps, checks
def position_map(layout: int, S: int, n_shards: int, device="cuda", stream=None):
    """(shard_of[S], local_of[S], token_of[N, L]) int32 computed on the device."""
    lib = load()
    shard = torch.empty(S, dtype=torch.int32, device=device)
    local = torch.empty(S, dtype=torch.int32, device=device)
    tok = torch.empty(S, dtype=torch.int32, device=device)
    _check(lib.ra_position_map(int(layout), S, int(n_shards), _ptr(shard), _ptr(local), _ptr(tok),
                               _stream(stream)))
    return shard, local, tok.view(n_shards, S // n_shards)


def ring_order(n_shards: int, device="cuda", stream=None):
    lib = load()
    order = torch.empty(n_shards * n_shards, dtype=torch.int32, device=device)
    _check(lib.ra_ring_order(int(n_shards), _ptr(order), _stream(stream)))
    return order.view(n_shards, n_shards)


def stream_check(stream=None):
    """Synchronise the stream and raise if a device wait timed out."""
    _check(load().ra_stream_check(_stream(stream)))


def launch_count() -> int:
    """Kernels the library has launched in this process."""
    return int(load().ra_launch_count())


def ex2_probe(iters: int, sink=None, stream=None):
    """Launch the exp2-rate probe; returns (sink tensor, exp2 evaluated).
    The caller brackets the call with CUDA events."""
    lib = load()
    n = int(lib.ra_ex2_probe_threads())
    if sink is None:
        sink = torch.empty(n, dtype=torch.float32, device="cuda")
    _check(lib.ra_ex2_probe(iters, _ptr(sink), sink.numel(), _stream(stream)))
    return sink, 8 * iters * n


def selftest_wait_timeout(budget_cycles: int, stream=None):
    _check(load().ra_selftest_wait_timeout(int(budget_cycles), _stream(stream)))


# ------------------------------------------------------------------ host buffers
class HostBuffer:
    """Pinned host memory from ``ra_host_alloc`` (on the NUMA node nearest the
    current GPU), viewed as a CPU tensor ``.tensor`` of the given shape and
    dtype.  The memory is freed by ``free()`` or when this object is
    collected; keep the object alive while ``.tensor`` (or a view) is used."""

    def __init__(self, shape, dtype):
        lib = load()
        shape = tuple(int(x) for x in shape)
        nbytes = torch.Size(shape).numel() * torch.empty((), dtype=dtype).element_size()
        ptr = ctypes.c_void_p()
        _check(lib.ra_host_alloc(nbytes, ctypes.byref(ptr)))
        self._ptr = ptr.value
        self.nbytes = nbytes
        if nbytes == 0:
            self.tensor = torch.empty(shape, dtype=dtype)
        else:
            raw = (ctypes.c_uint8 * nbytes).from_address(self._ptr)
            self.tensor = torch.frombuffer(raw, dtype=torch.uint8).view(dtype).view(shape)

    def data_ptr(self) -> int:
        return self._ptr or 0

    def free(self):
        if getattr(self, "_ptr", None):
            self.tensor = None
            _check(load().ra_host_free(ctypes.c_void_p(self._ptr)))
            self._ptr = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def host_numa_node() -> int:
    return int(load().ra_host_numa_node())


class Pipeline:
    """``ra_pipeline``: ring-attention steps on host buffers, each step's
    copies overlapped with its neighbours' compute (two device buffer sets,
    three streams).  ``submit`` takes CPU tensors (or ``HostBuffer``s) and
    returns at once; ``sync`` waits for every submitted step."""

    def __init__(self, S: int, n_shards: int, layout: int, causal: bool, b: int, h: int,
                 n_kv: int, d: int, backward: bool = True, scale: float = 0.0):
        lib = load()
        handle = ctypes.c_void_p()
        _check(lib.ra_pipeline_create(S, n_shards, layout, int(bool(causal)), scale,
                                      _dims(b, h, n_kv, d), int(bool(backward)),
                                      ctypes.byref(handle)))
        self._h = handle.value
        self.backward = backward
        rows = b * S
        # bytes each host buffer must hold: inputs bf16, results fp32
        self._need = {"q": rows * h * d * 2, "k": rows * n_kv * d * 2, "v": rows * n_kv * d * 2,
                      "dout": rows * h * d * 2, "out": rows * h * d * 4, "lse": rows * h * 4,
                      "dq": rows * h * d * 4, "dk": rows * n_kv * d * 4, "dv": rows * n_kv * d * 4}

    def _hp(self, name, x):
        if x is None:
            return None
        if isinstance(x, HostBuffer):
            nbytes, ptr = x.nbytes, x.data_ptr()
        else:
            if x.is_cuda or not x.is_contiguous():
                raise RAError(RA_ERR_INVALID_ARG, "pipeline buffers are contiguous host tensors")
            nbytes, ptr = x.numel() * x.element_size(), x.data_ptr()
        if nbytes < self._need[name]:
            raise RAError(RA_ERR_INVALID_ARG,
                          f"{name}: {nbytes} bytes given, {self._need[name]} needed")
        return ctypes.c_void_p(ptr)

    def submit(self, q, k, v, dout=None, out=None, lse=None, dq=None, dk=None, dv=None):
        hp = self._hp
        _check(load().ra_pipeline_submit(ctypes.c_void_p(self._h), hp("q", q), hp("k", k),
                                         hp("v", v), hp("dout", dout), hp("out", out),
                                         hp("lse", lse), hp("dq", dq), hp("dk", dk),
                                         hp("dv", dv)))

    def sync(self):
        _check(load().ra_pipeline_sync(ctypes.c_void_p(self._h)))

    def close(self):
        if getattr(self, "_h", None):
            load().ra_pipeline_destroy(ctypes.c_void_p(self._h))
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
