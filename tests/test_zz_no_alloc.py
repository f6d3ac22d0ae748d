"""The allocation-free backward, ra_ring_attention_bwd_noalloc.

It exists for callers that cannot allocate device memory where they run the
backward (inside a CUDA-graph capture, in plug-ins handed tensors by a host
framework that owns the allocator).  It must give what the workspace-taking
ra_ring_attention_bwd gives, call after call, with its scratch in the
library's fixed device array.  This file is collected last on purpose."""

import ctypes

import numpy as np
import pytest
import torch

from long_context_exact_gb300 import binding as ra
from long_context_exact_gb300.inputs import CONTIGUOUS, STRIPED, make_inputs

pytestmark = pytest.mark.gpu

G_TOL = 1e-2   # the parity tolerance of the backward tests


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_exact_gb300 import build as b
    b.build()
    return ra.load()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_backward_matches_workspace_backward_twice(lib):
    cases = [(1, 2048, 8, 2, 128, 4, STRIPED, True), (2, 1536, 4, 1, 128, 3, CONTIGUOUS, True)]
    for (b, S, h, n_kv, d, N, layout, causal) in cases:   # two calls in a row
        q, k, v, do = (t.cuda() for t in make_inputs(b, S, h, n_kv, d, seed=S + b,
                                                      with_dout=True))
        out, lse = ra.ring_attention(q, k, v, N, layout, causal)
        ref = ra.ring_attention_bwd(q, k, v, out, lse, do, N, layout, causal)
        dq = torch.full((b, S, h, d), float("nan"), device="cuda")
        dk = torch.full((b, S, n_kv, d), float("nan"), device="cuda")
        dv = torch.full((b, S, n_kv, d), float("nan"), device="cuda")
        # a known last error first: a successful call must leave it as it was
        assert lib.ra_ring_order(0, None, None) != ra.RA_OK
        marker = lib.ra_last_error()
        st = lib.ra_ring_attention_bwd_noalloc(
            _p(q), _p(k), _p(v), _p(out), _p(lse), _p(do), _p(dq), _p(dk), _p(dv), S, N,
            layout, int(causal), 0.0, ra.Dims(b, h, n_kv, d),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == ra.RA_OK, lib.ra_last_error()
        assert lib.ra_last_error() == marker
        ra.stream_check()
        for got, want in zip((dq, dk, dv), ref):
            err = (got - want).abs().max().item()
            assert np.isfinite(err) and err <= G_TOL, err


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    b, h, n_kv, d = 1, 32, 8, 128
    S = 1 << 20          # needs 2 * 32 * 2^20 * 4 bytes = 256 MiB of scratch
    fake = ctypes.c_void_p(0x10000)
    st = lib.ra_ring_attention_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                           S, 8, STRIPED, 1, 0.0, ra.Dims(b, h, n_kv, d), None)
    assert st == ra.RA_ERR_WORKSPACE
    assert b"allocation-free" in lib.ra_last_error()


def test_forward_and_noalloc_backward_replay_as_a_cuda_graph(lib):
    """A whole step (ring forward, allocation-free backward) captured once as
    a CUDA graph and replayed on new inputs copied into the same buffers
    gives the eager results: no call in the path allocates or synchronises."""
    b, S, h, n_kv, d, N, layout = 1, 2048, 8, 2, 128, 4, STRIPED
    first = [t.cuda() for t in make_inputs(b, S, h, n_kv, d, seed=21, with_dout=True)]
    second = [t.cuda() for t in make_inputs(b, S, h, n_kv, d, seed=22, with_dout=True)]
    q, k, v, do = (t.clone() for t in first)
    out = torch.empty((b, S, h, d), dtype=torch.float32, device="cuda")
    lse = torch.empty((b, h, S), dtype=torch.float32, device="cuda")
    dq = torch.empty((b, S, h, d), dtype=torch.float32, device="cuda")
    dk = torch.empty((b, S, n_kv, d), dtype=torch.float32, device="cuda")
    dv = torch.empty_like(dk)

    def step():
        ra.ring_attention(q, k, v, N, layout, True, out=out, lse=lse)
        ra.ring_attention_bwd_noalloc(q, k, v, out, lse, do, N, layout, True, dq=dq, dk=dk, dv=dv)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                      # warm-up outside the capture (scratch address lookup)
    torch.cuda.current_stream().wait_stream(side)
    ra.stream_check()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for inputs in (second, first):
        for dst, src in zip((q, k, v, do), inputs):
            dst.copy_(src)
        for t in (out, lse, dq, dk, dv):
            t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        ra.stream_check()
        e_out, e_lse = ra.ring_attention(*inputs[:3], N, layout, True)
        e_grads = ra.ring_attention_bwd(*inputs[:3], e_out, e_lse, inputs[3], N, layout, True)
        assert torch.equal(out, e_out) and torch.equal(lse, e_lse)
        # dq, dk, dv are sums of fp32 partials added in arrival order: equal
        # to the eager run up to fp32 rounding relative to their size
        for got, want in zip((dq, dk, dv), e_grads):
            assert float((got - want).abs().max()) <= 1e-5 * float(want.abs().max())
