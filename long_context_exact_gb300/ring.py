"""Ring attention across processes, one per GPU: the pages' ring protocol
with real key/value exchange between devices.

Rank r of a ring of N ranks holds one query block and one key/value block of
the sequence (any placement: contiguous, striped or zig-zag shards, given by
the token positions of its rows).  At ring step s it holds the key/value
block of rank (r - s) mod N, folds it into the online-softmax state of its
query rows with one block step, and meanwhile sends that block on to rank
r + 1 and receives the next one from rank r - 1 into a second buffer ("The
Ring Attention Protocol and Overlapped Communication" on the first page; the
summary's "The Ring Communication Protocol: Overlapping Transfer with
Computation").  After N steps it finalizes: out = O / l, lse = m + ln l.

The backward ("The Backward Pass and Gradient Exchange"; "The Backward Pass:
Symmetric Ring Operation"): dQ of a query block stays with its rank; the
key/value block travels with its gradient accumulators dK, dV, each rank
adding the contribution of its query rows, and after a full cycle the
accumulators arrive back at the block's own rank.  The key/value send of a
step overlaps that step's compute; the accumulators move after it.

Transport is torch.distributed point-to-point (NCCL between GPUs; gloo on
the host for tests).  No kernel or library is ever given another rank's
memory: every block is copied into local buffers first.  The per-step
compute is the library's ra_block_step / ra_finalize / ra_block_step_bwd
(``CudaBlockOps``); a test may pass its own ``ops`` object with the same
four methods to check the exchange schedule on the host.
"""

from __future__ import annotations

import torch
import torch.distributed as dist


class CudaBlockOps:
    """The library's block calls: the compute of every ring step."""

    def new_state(self, b, Lq, h, d, device):
        from . import binding
        return binding.new_state(b, Lq, h, d, device)

    def block_step(self, q, k, v, state, q_pos, k_pos, causal, scale):
        from . import binding
        binding.block_step(q, k, v, state, q_pos, k_pos, causal, scale)

    def finalize(self, state):
        from . import binding
        return binding.finalize(state)

    def block_step_bwd(self, q, k, v, out, lse, dout, grads, q_pos, k_pos, causal, scale):
        from . import binding
        binding.block_step_bwd(q, k, v, out, lse, dout, grads, q_pos, k_pos, causal, scale)


class RingGroup:
    """The ranks of a process group as a ring: each rank sends to the next
    and receives from the previous one."""

    def __init__(self, group=None):
        self.group = group
        if group is None and not dist.is_initialized():   # one process: a ring of one
            self.rank, self.size, self.next, self.prev = 0, 1, 0, 0
            return
        self.rank = dist.get_rank(group)
        self.size = dist.get_world_size(group)
        ranks = list(range(dist.get_world_size())) if group is None else \
            dist.get_process_group_ranks(group)
        self.next = ranks[(self.rank + 1) % self.size]
        self.prev = ranks[(self.rank - 1) % self.size]

    def exchange(self, send, recv):
        """Start sending `send` to the next rank and receiving `recv` from the
        previous one; returns the requests to wait on."""
        if self.size == 1:
            return []
        ops = [dist.P2POp(dist.isend, t, self.next, self.group) for t in send]
        ops += [dist.P2POp(dist.irecv, t, self.prev, self.group) for t in recv]
        return dist.batch_isend_irecv(ops)


def _wait(reqs):
    for r in reqs:
        r.wait()


def ring_attention_fwd(q, k, v, q_pos, k_pos, causal: bool = True, scale: float = 0.0,
                       group=None, ops=None):
    """This rank's query rows against every key/value block of the ring.

    q [b, Lq, h, d] and k, v [b, Lk, n_kv, d] are this rank's blocks (every
    rank's blocks have the same shapes); q_pos [Lq], k_pos [Lk] int32 are the
    token positions of their rows, increasing.  Returns (out [b, Lq, h, d],
    lse [b, h, Lq]) over the whole sequence."""
    ring = RingGroup(group)
    ops = ops or CudaBlockOps()
    b, Lq, h, d = q.shape
    state = ops.new_state(b, Lq, h, d, q.device)
    # private copies: later steps receive into both buffers, and the
    # caller's k, v, k_pos (perhaps q_pos itself) must stay as they are
    cur = [k.clone(), v.clone(), k_pos.clone()]
    nxt = [torch.empty_like(t) for t in cur]
    for s in range(ring.size):
        # block (r - s) mod N is here; (r - s - 1) mod N is on its way
        reqs = ring.exchange(cur, nxt) if s < ring.size - 1 else []
        ops.block_step(q, cur[0], cur[1], state, q_pos, cur[2], causal, scale)
        _wait(reqs)
        if reqs:
            cur, nxt = nxt, cur
    return ops.finalize(state)


def ring_attention_bwd(q, k, v, out, lse, dout, q_pos, k_pos, causal: bool = True,
                       scale: float = 0.0, group=None, ops=None, grad_dtype=torch.float32):
    """Gradients of this rank's blocks: dq [b, Lq, h, d] of its query rows and
    dk, dv [b, Lk, n_kv, d] of its key/value rows (float32: the library's
    accumulators), from the query rows' whole-sequence out and lse
    (ring_attention_fwd)."""
    ring = RingGroup(group)
    ops = ops or CudaBlockOps()
    b, Lq, h, d = q.shape
    dq = torch.zeros((b, Lq, h, d), dtype=grad_dtype, device=q.device)
    cur_kv = [k.clone(), v.clone(), k_pos.clone()]   # private: received into later
    nxt_kv = [torch.empty_like(t) for t in cur_kv]
    cur_g = [torch.zeros(k.shape, dtype=grad_dtype, device=k.device) for _ in range(2)]
    nxt_g = [torch.empty_like(t) for t in cur_g]
    for s in range(ring.size):
        reqs = ring.exchange(cur_kv, nxt_kv) if s < ring.size - 1 else []
        ops.block_step_bwd(q, cur_kv[0], cur_kv[1], out, lse, dout, (dq, cur_g[0], cur_g[1]),
                           q_pos, cur_kv[2], causal, scale)
        # the accumulators move on after the step that added to them; the
        # last move brings every block's home
        reqs_g = ring.exchange(cur_g, nxt_g)
        _wait(reqs)
        _wait(reqs_g)
        if reqs:
            cur_kv, nxt_kv = nxt_kv, cur_kv
        if reqs_g:
            cur_g, nxt_g = nxt_g, cur_g
    return dq, cur_g[0], cur_g[1]
