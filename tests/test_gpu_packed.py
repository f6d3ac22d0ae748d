"""GPU parity of packed documents (block-diagonal mask with causal rule)
against the fp64 oracle, forward and backward, through the C ABI.

Tolerances as the unpacked tests: max-abs 1e-2 on O, dQ, dK, dV and 1e-3 on
the LSE."""

import numpy as np
import pytest
import torch

from long_context_exact_gb300 import binding as ra
from long_context_exact_gb300.inputs import (CONTIGUOUS, STRIPED, WORKLOADS, ZIGZAG, make_inputs,
                                             packed_offsets, sample_rows, workload_inputs)

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
LSE_TOL = 1e-3
G_TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_exact_gb300 import build as b
    b.build()
    ra.load()


def _cu(offsets):
    return torch.tensor(np.asarray(offsets, np.int32)).cuda()


CASES = [
    # b, S, h, n_kv, d, N, layout, causal, offsets (per batch row)
    (1, 1024, 4, 2, 128, 4, STRIPED, True, [[0, 100, 356, 357, 1024]]),   # one-token document
    (1, 1024, 4, 2, 128, 4, CONTIGUOUS, True, [[0, 256, 512, 1024]]),     # tile-aligned bounds
    (2, 2048, 8, 2, 128, 8, STRIPED, True, None),                          # drawn, b = 2
    (1, 2048, 8, 2, 128, 4, ZIGZAG, True, None),
    (1, 1536, 6, 2, 64, 3, CONTIGUOUS, False, [[0, 700, 700, 1536]]),     # non-causal, empty doc
    (1, 1024, 4, 4, 64, 2, STRIPED, False, None),
    (1, 600, 4, 2, 128, 3, CONTIGUOUS, True, [[0, 1, 599, 600]]),         # ragged shards
    (1, 512, 4, 2, 128, 1, CONTIGUOUS, True, [[0, 512]]),                 # one document
]


def _offsets(b, S, offsets, seed):
    if offsets is not None:
        return np.asarray(offsets, np.int32)
    return packed_offsets(S, seed, min_len=64, max_len=S // 2, b=b)


@pytest.mark.parametrize("b,S,h,n_kv,d,N,layout,causal,offsets", CASES)
def test_packed_forward_matches_oracle(orc, b, S, h, n_kv, d, N, layout, causal, offsets):
    cu = _offsets(b, S, offsets, seed=S + N)
    q, k, v = make_inputs(b, S, h, n_kv, d, seed=S + 3 * N + d)
    ref_o, ref_l = orc.attn_fwd_rows(q, k, v, causal, cu_seqlens=cu)
    out, lse = ra.ring_attention(q.cuda(), k.cuda(), v.cuda(), N, layout, causal,
                                 cu_seqlens=_cu(cu))
    ra.stream_check()
    o = out.double().cpu().numpy()
    l = lse.double().cpu().numpy()
    assert np.abs(o - ref_o).max() <= O_TOL
    assert np.all(np.isfinite(l))                  # every token sees itself or its document
    assert np.abs(l - ref_l).max() <= LSE_TOL


@pytest.mark.parametrize("b,S,h,n_kv,d,N,layout,causal,offsets", CASES)
def test_packed_backward_matches_oracle(orc, b, S, h, n_kv, d, N, layout, causal, offsets):
    cu = _offsets(b, S, offsets, seed=S + N)
    q, k, v, do = make_inputs(b, S, h, n_kv, d, seed=S + 5 * N + d, with_dout=True)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    cut = _cu(cu)
    out, lse = ra.ring_attention(qd, kd, vd, N, layout, causal, cu_seqlens=cut)
    dq, dk, dv = ra.ring_attention_bwd(qd, kd, vd, out, lse, dod, N, layout, causal, cu_seqlens=cut)
    ra.stream_check()
    rq, rk, rv = orc.attn_bwd_rows(q, k, v, do, causal, cu_seqlens=cu)
    errs = [float(np.abs(a.double().cpu().numpy() - r).max()) for a, r in ((dq, rq), (dk, rk), (dv, rv))]
    assert max(errs) <= G_TOL, errs


def test_packed_single_document_equals_unpacked():
    q, k, v = (t.cuda() for t in make_inputs(1, 2048, 8, 2, 128, seed=9))
    o1, l1 = ra.ring_attention(q, k, v, 8, STRIPED, True)
    o2, l2 = ra.ring_attention(q, k, v, 8, STRIPED, True, cu_seqlens=_cu([[0, 2048]]))
    ra.stream_check()
    assert (o1 - o2).abs().max().item() <= 1e-6 and (l1 - l2).abs().max().item() <= 1e-6


def test_workload_packed_64k(orc):
    w = WORKLOADS["packed64k"]
    q, k, v = workload_inputs(w)[:3]
    cu = packed_offsets(w.S, w.seed)
    rows = sample_rows(w.S, w.n_shards, w.rows_per_head, w.seed)
    # plus the first tokens of every document (the rows with the fewest keys)
    rows = np.unique(np.concatenate([rows, cu[0, :-1], np.minimum(cu[0, :-1] + 1, w.S - 1)]))
    ref_o, ref_l = orc.attn_fwd_rows(q, k, v, True, rows=rows, cu_seqlens=cu)
    out, lse = ra.ring_attention(q.cuda(), k.cuda(), v.cuda(), w.n_shards, STRIPED, True,
                                 cu_seqlens=_cu(cu))
    ra.stream_check()
    o = out.double().cpu().numpy()[:, rows]
    l = lse.double().cpu().numpy()[:, :, rows]
    assert np.abs(o - ref_o).max() <= O_TOL
    assert np.abs(l - ref_l).max() <= LSE_TOL
