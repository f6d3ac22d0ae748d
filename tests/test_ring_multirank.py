"""The multi-process ring (long_context_exact_gb300/ring.py) on the host:
2 and 4 gloo ranks exchange real key/value blocks (and, in the backward, the
travelling dK / dV accumulators) with point-to-point sends, as NCCL ranks on
GPUs would.  The per-step compute is the fp64 oracle (its blockwise update
and finalize) and, for the backward, a plain numpy restatement of one block's
gradient contribution written here; the sums over the ring must equal the
oracle's direct definition and its analytic gradient.  Each rank records the
positions of the key/value block it holds at each step: they must be those
of block (r - s) mod N, bit for bit."""

import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleOps:
    """Ring-step compute on the host in fp64: the oracle's block update and
    finalize; the backward block contribution restated with numpy."""

    def __init__(self, orc):
        self.orc = orc
        self.held = []       # (step, positions of the key/value block held)

    def new_state(self, b, Lq, h, d, device):
        return self.orc.new_state(b, Lq, h, d)

    def block_step(self, q, k, v, state, q_pos, k_pos, causal, scale):
        self.held.append(k_pos.numpy().copy())
        self.orc.block_update(q.numpy(), k.numpy(), v.numpy(), q_pos.numpy(), k_pos.numpy(),
                              causal, scale, state)

    def finalize(self, state):
        return self.orc.finalize(state)

    def block_step_bwd(self, q, k, v, out, lse, dout, grads, q_pos, k_pos, causal, scale):
        """Contribution of one key/value block to the gradients, P from the
        query rows' whole-sequence LSE: dS = P (dO V^T - rowsum(dO O))."""
        self.held.append(k_pos.numpy().copy())
        q, k, v, dout, out, lse = (t.numpy() for t in (q, k, v, dout, out, lse))
        dq, dk, dv = (t.numpy() for t in grads)     # views: added to in place
        b, Lq, h, d = q.shape
        g = h // k.shape[2]
        vis = (k_pos.numpy()[None, :] <= q_pos.numpy()[:, None]) if causal else \
            np.ones((Lq, k.shape[1]), dtype=bool)
        for bb in range(b):
            for hq in range(h):
                kh = hq // g
                s = scale * q[bb, :, hq] @ k[bb, :, kh].T
                p = np.where(vis, np.exp(s - lse[bb, hq][:, None]), 0.0)
                dsum = (dout[bb, :, hq] * out[bb, :, hq]).sum(-1)
                ds = p * (dout[bb, :, hq] @ v[bb, :, kh].T - dsum[:, None])
                dq[bb, :, hq] += scale * ds @ k[bb, :, kh]
                dk[bb, :, kh] += scale * ds.T @ q[bb, :, hq]
                dv[bb, :, kh] += p.T @ dout[bb, :, hq]


def _rank_main(rank, world, port, case, out):
    from long_context_exact_gb300 import ring
    from long_context_exact_gb300.inputs import make_inputs
    from oracle import oracle as orc
    b, S, h, n_kv, d, layout, causal = case
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        q, k, v, do = (t.double() for t in make_inputs(b, S, h, n_kv, d, seed=S + world,
                                                       with_dout=True))
        _, _, tok = orc.position_map(layout, S, world)
        mine = torch.from_numpy(tok[rank].astype(np.int64))
        pos = torch.from_numpy(tok[rank].astype(np.int32))
        qi, ki, vi, doi = (t[:, mine].contiguous() for t in (q, k, v, do))
        scale = 1.0 / np.sqrt(d)
        ops = OracleOps(orc)
        keep = [t.clone() for t in (qi, ki, vi, pos)]
        o_i, l_i = ring.ring_attention_fwd(qi, ki, vi, pos, pos, causal, scale, ops=ops)
        # the caller's blocks are untouched by the exchanges
        assert all(torch.equal(a, b_) for a, b_ in zip(keep, (qi, ki, vi, pos)))
        fwd_held = ops.held
        ops.held = []
        dq, dk, dv = ring.ring_attention_bwd(qi, ki, vi, torch.from_numpy(o_i),
                                             torch.from_numpy(l_i), doi, pos, pos, causal,
                                             scale, ops=ops, grad_dtype=torch.float64)
        assert all(torch.equal(a, b_) for a, b_ in zip(keep, (qi, ki, vi, pos)))
        out[rank] = dict(o=o_i, lse=l_i, dq=dq.numpy(), dk=dk.numpy(), dv=dv.numpy(),
                         fwd_held=fwd_held, bwd_held=ops.held)
        dist.barrier()
    finally:
        dist.destroy_process_group()


CASES = [
    # world, (b, S, h, n_kv, d, layout, causal)
    (2, (1, 256, 4, 2, 16, 1, True)),
    (2, (2, 256, 4, 1, 16, 0, True)),
    (4, (1, 256, 4, 2, 16, 2, True)),
    (4, (1, 128, 2, 2, 8, 1, False)),
    (3, (1, 192, 6, 2, 8, 1, True)),     # odd ring, g = 3
    (3, (1, 192, 6, 2, 8, 2, True)),     # zig-zag over three ranks
]


@pytest.mark.parametrize("world,case", CASES)
def test_ring_over_gloo_ranks(orc, world, case):
    b, S, h, n_kv, d, layout, causal = case
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        res = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), case, res), nprocs=world,
                           join=True, start_method="spawn")
        res = dict(res)
    assert set(res) == set(range(world))
    from long_context_exact_gb300.inputs import make_inputs
    q, k, v, do = make_inputs(b, S, h, n_kv, d, seed=S + world, with_dout=True)
    ref_o, ref_l = orc.attn_fwd_rows(q, k, v, causal)
    rq, rk, rv = orc.attn_bwd_rows(q, k, v, do, causal)
    _, _, tok = orc.position_map(layout, S, world)
    order = orc.ring_order(world)
    for r in range(world):
        t = tok[r]
        got = res[r]
        # the schedule: at step s rank r holds block (r - s) mod N
        for name in ("fwd_held", "bwd_held"):
            held = got[name]
            assert len(held) == world
            for s_ in range(world):
                assert np.array_equal(held[s_], tok[order[r, s_]]), (name, r, s_)
        np.testing.assert_allclose(got["o"], ref_o[:, t], atol=1e-12, rtol=0)
        fin = np.isfinite(ref_l[:, :, t])
        np.testing.assert_allclose(got["lse"][fin], ref_l[:, :, t][fin], atol=1e-12, rtol=0)
        np.testing.assert_allclose(got["dq"], rq[:, t], atol=1e-10, rtol=0)
        # the accumulators that arrived home are this rank's own block's
        np.testing.assert_allclose(got["dk"], rk[:, t], atol=1e-10, rtol=0)
        np.testing.assert_allclose(got["dv"], rv[:, t], atol=1e-10, rtol=0)


def test_single_rank_ring_is_one_block_step(orc):
    """World size 1: no exchange, one step over the rank's own block."""
    from long_context_exact_gb300 import ring
    from long_context_exact_gb300.inputs import make_inputs
    port = _free_port()
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=0,
                            world_size=1)
    try:
        q, k, v, do = (t.double() for t in make_inputs(1, 64, 2, 1, 8, seed=3, with_dout=True))
        pos = torch.arange(64, dtype=torch.int32)
        ops = OracleOps(orc)
        o, l = ring.ring_attention_fwd(q, k, v, pos, pos, True, 1 / np.sqrt(8), ops=ops)
        ref_o, ref_l = orc.attn_fwd_rows(q, k, v, True, scale=1 / np.sqrt(8))
        np.testing.assert_allclose(o, ref_o, atol=1e-12, rtol=0)
        dq, dk, dv = ring.ring_attention_bwd(q, k, v, torch.from_numpy(o), torch.from_numpy(l),
                                             do, pos, pos, True, 1 / np.sqrt(8), ops=ops,
                                             grad_dtype=torch.float64)
        rq, rk, rv = orc.attn_bwd_rows(q, k, v, do, True, scale=1 / np.sqrt(8))
        for a, r_ in ((dq, rq), (dk, rk), (dv, rv)):
            np.testing.assert_allclose(a.numpy(), r_, atol=1e-10, rtol=0)
    finally:
        dist.destroy_process_group()
