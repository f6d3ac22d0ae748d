"""Pins for the fp64 CPU oracle: each test checks it against something other
than itself -- brute-force full matrices built with library softmax, PyTorch's
own attention routine and autograd, closed forms, invariants the pages state,
finite differences, and the worked examples printed on the pages.

A plausible slip anywhere in the oracle (a dropped rescale, a wrong sign or
index, a transposed operand, the wrong GQA head, an off-by-one causal rule)
fails at least one of these.
"""

import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

from long_context_exact_gb300.inputs import make_inputs, sample_rows

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _brute(q, k, v, causal, scale):
    """Full S x S score matrix per (batch, head) with scipy's softmax."""
    qd = q.to(torch.float64).numpy()
    kd = k.to(torch.float64).numpy()
    vd = v.to(torch.float64).numpy()
    b, S, h, d = qd.shape
    g = h // kd.shape[2]
    kx = np.repeat(kd, g, axis=2)   # query head hq reads kv head hq // g
    vx = np.repeat(vd, g, axis=2)
    sc = np.einsum("bqhd,bkhd->bhqk", qd, kx) * scale
    if causal:
        sc = np.where(np.tril(np.ones((S, S), bool))[None, None], sc, -np.inf)
    lse = logsumexp(sc, axis=-1)
    p = softmax(sc, axis=-1)
    out = np.einsum("bhqk,bkhd->bqhd", p, vx)
    return out, lse, p


CASES = [
    # b, S, h, n_kv, d, causal
    (1, 64, 2, 2, 16, False),
    (2, 96, 4, 2, 16, True),
    (1, 128, 8, 2, 32, True),
    (2, 80, 6, 3, 8, False),
    (1, 256, 2, 1, 64, True),
]


@pytest.mark.parametrize("b,S,h,n_kv,d,causal", CASES)
def test_direct_definition_matches_brute_force(orc, b, S, h, n_kv, d, causal):
    q, k, v = make_inputs(b, S, h, n_kv, d, seed=7)
    scale = 1.0 / np.sqrt(d)
    out, lse = orc.attn_fwd_rows(q, k, v, causal, scale)
    ref_out, ref_lse, _ = _brute(q, k, v, causal, scale)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_direct_definition_matches_torch_sdpa(orc, causal):
    b, S, h, n_kv, d = 2, 128, 8, 2, 32
    q, k, v = make_inputs(b, S, h, n_kv, d, seed=11)
    out, _ = orc.attn_fwd_rows(q, k, v, causal)
    tq, tk, tv = (x.to(torch.float64).transpose(1, 2) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(h // n_kv, 1), tv.repeat_interleave(h // n_kv, 1),
        is_causal=causal).transpose(1, 2).numpy()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_sampled_rows_equal_full_rows(orc):
    b, S, h, n_kv, d = 1, 256, 4, 2, 16
    q, k, v = make_inputs(b, S, h, n_kv, d, seed=3)
    rows = sample_rows(S, 4, 20, seed=3)
    full_o, full_l = orc.attn_fwd_rows(q, k, v, True)
    o, l = orc.attn_fwd_rows(q, k, v, True, rows=rows)
    np.testing.assert_array_equal(o, full_o[:, rows])
    np.testing.assert_array_equal(l, full_l[:, :, rows])


# ---------------------------------------------------------------- closed forms
def test_zero_queries_give_uniform_weights(orc):
    b, S, h, n_kv, d = 1, 200, 4, 2, 16
    _, k, v = make_inputs(b, S, h, n_kv, d, seed=5)
    q = torch.zeros((b, S, h, d), dtype=torch.bfloat16)
    vd = v.to(torch.float64).numpy()
    for causal in (False, True):
        out, lse = orc.attn_fwd_rows(q, k, v, causal)
        counts = np.arange(1, S + 1) if causal else np.full(S, S)
        np.testing.assert_allclose(lse[0], np.log(counts)[None, :].repeat(h, 0), atol=1e-13)
        for hq in range(h):
            kh = hq // (h // n_kv)
            csum = np.cumsum(vd[0, :, kh], axis=0)
            exp = csum / counts[:, None] if causal else np.repeat(csum[-1:] / S, S, 0)
            np.testing.assert_allclose(out[0, :, hq], exp, atol=1e-12)


def test_constant_values_pass_through(orc):
    b, S, h, n_kv, d = 2, 64, 4, 4, 8
    q, k, _ = make_inputs(b, S, h, n_kv, d, seed=9)
    v = torch.full((b, S, n_kv, d), 0.75, dtype=torch.bfloat16)
    for causal in (False, True):
        out, _ = orc.attn_fwd_rows(q, k, v, causal)
        np.testing.assert_allclose(out, 0.75, atol=1e-13)


def test_causal_first_row_and_single_token(orc):
    b, S, h, n_kv, d = 1, 32, 2, 1, 16
    q, k, v = make_inputs(b, S, h, n_kv, d, seed=4)
    scale = 0.3
    out, lse = orc.attn_fwd_rows(q, k, v, True, scale)
    qd, kd, vd = (x.to(torch.float64).numpy() for x in (q, k, v))
    for hq in range(h):
        np.testing.assert_allclose(out[0, 0, hq], vd[0, 0, 0], atol=1e-14)
        np.testing.assert_allclose(lse[0, hq, 0], scale * qd[0, 0, hq] @ kd[0, 0, 0], atol=1e-13)
    o1, l1 = orc.attn_fwd_rows(q[:, :1], k[:, :1], v[:, :1], False, scale)
    np.testing.assert_allclose(o1[0, 0, 0], vd[0, 0, 0], atol=1e-14)


def test_weights_are_a_distribution(orc):
    """With V = identity the output row is the weight row P_t: it is >= 0,
    sums to 1, and is 0 on keys after t when causal."""
    S = d = 64
    q, k, _ = make_inputs(1, S, 2, 1, d, seed=2)
    v = torch.eye(S, dtype=torch.bfloat16).reshape(1, S, 1, d)
    for causal in (False, True):
        out, _ = orc.attn_fwd_rows(q, k, v, causal)
        p = out[0]
        assert (p >= 0).all()
        np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-13)
        if causal:
            upper = np.triu(np.ones((S, S), bool), 1)
            for hq in range(2):
                assert np.all(p[:, hq][upper] == 0.0)


# ---------------------------------------------------------------- invariants
def test_noncausal_key_permutation_invariance(orc):
    q, k, v = make_inputs(2, 150, 4, 2, 16, seed=12)
    perm = torch.from_numpy(np.random.default_rng(0).permutation(150))
    o1, l1 = orc.attn_fwd_rows(q, k, v, False)
    o2, l2 = orc.attn_fwd_rows(q, k[:, perm], v[:, perm], False)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


@pytest.mark.parametrize("layout", [0, 1, 2])
@pytest.mark.parametrize("N", [1, 2, 4, 8])
@pytest.mark.parametrize("causal", [False, True])
def test_blockwise_ring_recurrence_is_exact(orc, layout, N, causal):
    """The online-softmax recurrence over shards in ring order reproduces the
    direct definition (first page: the recurrence gives the identical result)."""
    q, k, v = make_inputs(1, 128, 4, 2, 16, seed=21)
    o_ref, l_ref = orc.attn_fwd_rows(q, k, v, causal)
    o, l = orc.ring_blockwise_forward(q, k, v, N, layout, causal)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(l, l_ref, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_any_shard_visit_order_gives_same_result(orc, causal):
    """Fourth page: blocks may be combined in any order."""
    N = 4
    q, k, v = make_inputs(1, 128, 2, 1, 16, seed=8)
    o_ref, l_ref = orc.ring_blockwise_forward(q, k, v, N, 1, causal)
    rng = np.random.default_rng(1)
    order = np.stack([rng.permutation(N) for _ in range(N)])
    o, l = orc.ring_blockwise_forward(q, k, v, N, 1, causal, order=order)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(l, l_ref, atol=1e-12)


def test_contiguous_and_striped_agree(orc):
    q, k, v = make_inputs(1, 256, 4, 2, 16, seed=13)
    oc, lc = orc.ring_blockwise_forward(q, k, v, 8, 0, True)
    os_, ls_ = orc.ring_blockwise_forward(q, k, v, 8, 1, True)
    np.testing.assert_allclose(oc, os_, atol=1e-12)
    np.testing.assert_allclose(lc, ls_, atol=1e-12)


def test_block_update_keeps_rows_with_no_visible_key(orc):
    q, k, v = make_inputs(1, 8, 1, 1, 4, seed=1)
    state = orc.new_state(1, 8, 1, 4)
    # keys at positions 100.. are after every query position 0..7
    orc.block_update(q, k, v, np.arange(8), np.arange(100, 108), True, 0.5, state)
    m, l, o = state
    assert np.all(m == -np.inf) and np.all(l == 0) and np.all(o == 0)
    out, lse = orc.finalize(state)
    assert np.all(out == 0) and np.all(lse == -np.inf)


def test_merge_of_disjoint_key_sets(orc):
    """Merging results over two disjoint key sets equals one pass over all
    keys (second page's rescale-merge)."""
    b, S, h, n_kv, d = 1, 96, 4, 2, 16
    q, k, v = make_inputs(b, S, h, n_kv, d, seed=17)
    scale = 1.0 / np.sqrt(d)
    pos = np.arange(S)
    sel = np.random.default_rng(2).permutation(S)
    a_idx, b_idx = np.sort(sel[:40]), np.sort(sel[40:])
    parts = []
    for idx in (a_idx, b_idx):
        st = orc.new_state(b, S, h, d)
        ti = torch.from_numpy(idx)
        orc.block_update(q, k[:, ti], v[:, ti], pos, pos[idx], True, scale, st)
        parts.append(orc.finalize(st))
    o, lse = orc.merge(parts[0][0], parts[0][1], parts[1][0], parts[1][1])
    o_ref, l_ref = orc.attn_fwd_rows(q, k, v, True, scale)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(lse, l_ref, atol=1e-12)
    # a side with no keys (lse = -inf) leaves the other untouched
    empty_o = np.zeros_like(o)
    empty_l = np.full_like(lse, -np.inf)
    o2, l2 = orc.merge(o, lse, empty_o, empty_l)
    np.testing.assert_array_equal(o2, o)
    np.testing.assert_array_equal(l2, lse)
    o3, l3 = orc.merge(empty_o, empty_l, empty_o, empty_l)
    assert np.all(o3 == 0) and np.all(l3 == -np.inf)


# ---------------------------------------------------------------- page examples
def test_position_map_matches_printed_example(orc):
    rows = {}
    with open(os.path.join(GOLDEN, "position_map_8tok_4dev.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                name, *toks = line.split()
                rows[name] = np.array([int(t) for t in toks], np.int32).reshape(4, 2)
    for layout, name in ((0, "contiguous"), (1, "striped")):
        shard, local, tok = orc.position_map(layout, 8, 4)
        np.testing.assert_array_equal(tok, rows[name])
        np.testing.assert_array_equal(tok[shard, local], np.arange(8))


def test_position_map_zigzag_matches_page_rule(orc):
    with open(os.path.join(GOLDEN, "position_map_zigzag.txt")) as f:
        cases = [line.split() for line in f if line.strip() and not line.startswith("#")]
    assert cases
    for S, N, *toks in cases:
        S, N = int(S), int(N)
        shard, local, tok = orc.position_map(2, S, N)
        np.testing.assert_array_equal(tok, np.array([int(t) for t in toks], np.int32).reshape(N, -1))
        np.testing.assert_array_equal(tok[shard, local], np.arange(S))


def test_position_map_zigzag_balances_causal_work(orc):
    # The page: zig-zag gives every device the same number of causal
    # (query, key) pairs, N/2 full-block equivalents.  Under the inclusive
    # rule a query at position t sees t + 1 keys; summed over the two
    # half-blocks of C = L/2 tokens of device p this is N L^2 / 2 + L / 2 for
    # every p (the L/2 is the diagonal's half of the elements).
    for S, N in ((64, 4), (4096, 8), (1 << 14, 16)):
        _, _, tok = orc.position_map(2, S, N)
        L = S // N
        work = (tok.astype(np.int64) + 1).sum(axis=1)
        assert np.all(work == N * L * L // 2 + L // 2), (S, N, work)
        _, _, tok_c = orc.position_map(0, S, N)
        assert len(set((tok_c.astype(np.int64) + 1).sum(axis=1).tolist())) == N  # contiguous is not


def test_position_map_zigzag_rejects_odd_half_blocks(orc):
    with pytest.raises(ValueError):
        orc.position_map(2, 12, 4)   # 12 tokens cannot form 8 equal half-blocks


@pytest.mark.parametrize("layout", [0, 1, 2])
def test_position_map_round_trip(orc, layout):
    S, N = 4096, 16
    shard, local, tok = orc.position_map(layout, S, N)
    np.testing.assert_array_equal(tok[shard, local], np.arange(S))
    assert sorted(tok.ravel().tolist()) == list(range(S))


def test_ring_order_matches_printed_rule(orc):
    table = np.loadtxt(os.path.join(GOLDEN, "ring_index.txt"), dtype=np.int32)
    np.testing.assert_array_equal(orc.ring_order(4), table)
    o = orc.ring_order(8)
    assert all(sorted(r) == list(range(8)) for r in o)   # every block once
    assert all(o[i, 0] == i for i in range(8))           # own block first


# ---------------------------------------------------------------- gradients
def _torch_grads(q, k, v, dout, causal, scale):
    g = q.shape[2] // k.shape[2]
    tq, tk, tv = (x.to(torch.float64).transpose(1, 2).requires_grad_(True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(g, 1), tv.repeat_interleave(g, 1), is_causal=causal, scale=scale)
    o.backward(dout.to(torch.float64).transpose(1, 2))
    return tuple(x.grad.transpose(1, 2).numpy() for x in (tq, tk, tv))


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_matches_torch_autograd(orc, causal):
    b, S, h, n_kv, d = 2, 64, 4, 2, 16
    q, k, v, do = make_inputs(b, S, h, n_kv, d, seed=31, with_dout=True)
    scale = 1.0 / np.sqrt(d)
    dq, dk, dv = orc.attn_bwd_rows(q, k, v, do, causal, scale)
    rq, rk, rv = _torch_grads(q, k, v, do, causal, scale)
    np.testing.assert_allclose(dq, rq, atol=1e-12)
    np.testing.assert_allclose(dk, rk, atol=1e-12)
    np.testing.assert_allclose(dv, rv, atol=1e-12)


def test_gradient_of_row_subset_equals_masked_upstream(orc):
    b, S, h, n_kv, d = 1, 96, 4, 1, 16
    q, k, v, do = make_inputs(b, S, h, n_kv, d, seed=33, with_dout=True)
    scale = 1.0 / np.sqrt(d)
    rows = sample_rows(S, 4, 10, seed=33)
    dq, dk, dv = orc.attn_bwd_rows(q, k, v, do, True, scale, rows=rows)
    mask = torch.zeros(S, dtype=torch.bool)
    mask[torch.from_numpy(rows)] = True
    do_m = torch.where(mask[None, :, None, None], do, torch.zeros_like(do))
    rq, rk, rv = _torch_grads(q, k, v, do_m, True, scale)
    np.testing.assert_allclose(dq, rq[:, rows], atol=1e-12)
    np.testing.assert_allclose(dk, rk, atol=1e-12)
    np.testing.assert_allclose(dv, rv, atol=1e-12)


def test_gradient_finite_differences(orc):
    """Central differences of L = sum(dO * O) in fp64 match the analytic
    gradient."""
    b, S, h, n_kv, d = 1, 24, 2, 1, 8
    q, k, v, do = make_inputs(b, S, h, n_kv, d, seed=41, with_dout=True)
    scale = 0.4
    qd, kd, vd, gd = (x.to(torch.float64).numpy() for x in (q, k, v, do))

    def loss(qq, kk, vv):
        o, _ = orc.attn_fwd_rows(qq, kk, vv, True, scale)
        return float((o * gd).sum())

    dq, dk, dv = orc.attn_bwd_rows(q, k, v, do, True, scale)
    rng = np.random.default_rng(0)
    eps = 1e-6
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        for _ in range(12):
            arrs = [qd.copy(), kd.copy(), vd.copy()]
            idx = tuple(rng.integers(0, s) for s in arrs[which].shape)
            arrs[which][idx] += eps
            lp = loss(*arrs)
            arrs[which][idx] -= 2 * eps
            lm = loss(*arrs)
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(grad[idx])), (which, idx, fd, grad[idx])


def test_gradient_sum_invariants(orc):
    """sum_j dK_j = 0 (softmax rows sum to 1, so sum_j dS_tj = 0) and
    sum_j dV_j = sum over the group's query heads and all rows of dO."""
    b, S, h, n_kv, d = 2, 128, 8, 2, 16
    q, k, v, do = make_inputs(b, S, h, n_kv, d, seed=43, with_dout=True)
    _, dk, dv = orc.attn_bwd_rows(q, k, v, do, True)
    np.testing.assert_allclose(dk.sum(1), 0.0, atol=1e-11)
    gd = do.to(torch.float64).numpy().reshape(b, S, n_kv, h // n_kv, d)
    np.testing.assert_allclose(dv.sum(1), gd.sum(axis=(1, 3)), atol=1e-11)


# ---------------------------------------------------------------- packed documents
# The third page's section 5: documents packed end to end into one window, a
# block-diagonal mask keeping every document to itself.
PACKS = [
    # S, cu_seqlens per batch row
    (96, [[0, 17, 40, 40, 96], [0, 96, 96, 96, 96]]),   # an empty document; one spanning all
    (64, [[0, 1, 2, 3, 64], [0, 30, 31, 63, 64]]),      # one-token documents
]


def _per_document(q, k, v, do, cu, causal, fn):
    """Run fn on every document slice of every batch row separately."""
    res = []
    for bb, offs in enumerate(cu):
        parts = []
        for s0, s1 in zip(offs[:-1], offs[1:]):
            if s1 > s0:
                sl = slice(s0, s1)
                args = [x[bb:bb + 1, sl] for x in (q, k, v)] + ([do[bb:bb + 1, sl]] if do is not None else [])
                parts.append(((s0, s1), fn(*args, causal)))
        res.append(parts)
    return res


@pytest.mark.parametrize("S,cu", PACKS)
@pytest.mark.parametrize("causal", [True, False])
def test_packed_forward_equals_independent_documents(orc, S, cu, causal):
    q, k, v = make_inputs(2, S, 4, 2, 16, seed=S)
    o, l = orc.attn_fwd_rows(q, k, v, causal, cu_seqlens=cu)
    for bb, parts in enumerate(_per_document(q, k, v, None, cu, causal, orc.attn_fwd_rows)):
        for (s0, s1), (od, ld) in parts:
            np.testing.assert_array_equal(o[bb, s0:s1], od[0])
            np.testing.assert_array_equal(l[bb, :, s0:s1], ld[0])


@pytest.mark.parametrize("S,cu", PACKS)
@pytest.mark.parametrize("causal", [True, False])
def test_packed_backward_equals_independent_documents(orc, S, cu, causal):
    q, k, v, do = make_inputs(2, S, 4, 2, 16, seed=S + 1, with_dout=True)
    dq, dk, dv = orc.attn_bwd_rows(q, k, v, do, causal, cu_seqlens=cu)
    for bb, parts in enumerate(_per_document(q, k, v, do, cu, causal, orc.attn_bwd_rows)):
        for (s0, s1), (dqd, dkd, dvd) in parts:
            np.testing.assert_array_equal(dq[bb, s0:s1], dqd[0])
            np.testing.assert_array_equal(dk[bb, s0:s1], dkd[0])
            np.testing.assert_array_equal(dv[bb, s0:s1], dvd[0])


def test_packed_mask_matches_brute_force(orc):
    """An explicit S x S mask from document ids (same document, and key <=
    query) with scipy's softmax, against the oracle's interval rule."""
    S, cu = 40, [0, 7, 19, 40]
    q, k, v = make_inputs(1, S, 2, 1, 8, seed=3)
    doc = np.repeat(np.arange(3), np.diff(cu))
    mask = (doc[:, None] == doc[None, :]) & (np.arange(S)[None, :] <= np.arange(S)[:, None])
    qd, kd, vd = (x.double().numpy() for x in (q, k, v))
    o, l = orc.attn_fwd_rows(q, k, v, True, cu_seqlens=[cu])
    for hq in range(2):
        s = qd[0, :, hq] @ kd[0, :, 0].T / np.sqrt(8)
        s = np.where(mask, s, -np.inf)
        np.testing.assert_allclose(l[0, hq], logsumexp(s, axis=1), atol=1e-12)
        np.testing.assert_allclose(o[0, :, hq], softmax(s, axis=1) @ vd[0, :, 0], atol=1e-12)


def test_single_document_is_the_unpacked_definition(orc):
    q, k, v = make_inputs(1, 50, 2, 2, 8, seed=4)
    for causal in (True, False):
        o1, l1 = orc.attn_fwd_rows(q, k, v, causal)
        o2, l2 = orc.attn_fwd_rows(q, k, v, causal, cu_seqlens=[[0, 50]])
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(l1, l2)
