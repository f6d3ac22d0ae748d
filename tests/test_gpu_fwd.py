"""GPU parity of the forward path against the fp64 oracle, through the C ABI.

Tolerances: max-abs 1e-2 on O and 1e-3 on LSE (bf16 inputs, fp32
accumulation); integer maps bit-exact.  Small cases compare every element;
the long workloads compare sampled query rows the oracle computes one by one.
"""

import numpy as np
import pytest
import torch

from long_context_exact_gb300 import binding as ra
from long_context_exact_gb300.inputs import (CONTIGUOUS, STRIPED, WORKLOADS, ZIGZAG,
                                             make_inputs, sample_rows, workload_inputs)
from parity_util import peaked_inputs, plain_rows, record, rel_to_max

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
LSE_TOL = 1e-3
REL_TOL = 1e-2   # error relative to max|ref| on the plain-bf16-path rows


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_exact_gb300 import build as b
    b.build()
    ra.load()


def _dev(*ts):
    return [t.cuda() for t in ts]


def _nan_out(b, S, h, d, device="cuda"):
    """Output buffers filled with NaN, so a row the kernel never writes fails."""
    return (torch.full((b, S, h, d), float("nan"), dtype=torch.float32, device=device),
            torch.full((b, h, S), float("nan"), dtype=torch.float32, device=device))


def _ring(q, k, v, N, layout, causal, scale=0.0):
    b, S, h, d = q.shape
    out, lse = _nan_out(b, S, h, d, q.device)
    return ra.ring_attention(q, k, v, N, layout, causal, scale=scale, out=out, lse=lse)


def _rel_plain(o, ref_o, plain, what, tag=""):
    """On the rows that take the plain bf16 path: max|gpu - ref| / max|ref|
    <= REL_TOL, so that a small reference cannot hide a wrong result."""
    if not plain.any():
        return 0.0
    rel, ref = rel_to_max(o[:, plain], ref_o[:, plain])
    record(tag, o_plain_rel=rel)
    assert rel <= REL_TOL, f"{what}: plain-path rows max-abs error / max|ref| {rel:.3e} (max|ref| {ref:.3e})"
    return rel


def _cmp(out, lse, ref_out, ref_lse, rows=None, tag=""):
    """Every output written (no NaN left in the NaN-filled buffers), then the
    spec max-abs bounds on O and LSE over the checked rows."""
    assert not bool(torch.isnan(out).any()) and not bool(torch.isnan(lse).any()), \
        "unwritten (NaN) outputs"
    if rows is not None:
        idx = torch.from_numpy(np.asarray(rows, dtype=np.int64)).to(out.device)
        out = out.index_select(1, idx)
        lse = lse.index_select(2, idx)
    o = out.double().cpu().numpy()
    l = lse.double().cpu().numpy()
    err_o = np.abs(o - ref_out).max()
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(l), fin)
    err_l = np.abs(l[fin] - ref_lse[fin]).max() if fin.any() else 0.0
    record(tag, o_max_abs=err_o, lse_max_abs=err_l)
    assert err_o <= O_TOL, f"O max-abs {err_o}"
    assert err_l <= LSE_TOL, f"LSE max-abs {err_l}"
    return err_o, err_l


# ------------------------------------------------------------------ maps
@pytest.mark.parametrize("layout", [CONTIGUOUS, STRIPED, ZIGZAG])
@pytest.mark.parametrize("S,N", [(8, 4), (1024, 4), (65536, 8), (65536, 16), (3 * 200, 3)])
def test_position_map_bit_exact(orc, layout, S, N):
    shard, local, tok = ra.position_map(layout, S, N)
    r_shard, r_local, r_tok = orc.position_map(layout, S, N)
    assert np.array_equal(shard.cpu().numpy(), r_shard)
    assert np.array_equal(local.cpu().numpy(), r_local)
    assert np.array_equal(tok.cpu().numpy(), r_tok)


@pytest.mark.parametrize("N", [1, 2, 4, 8, 16, 37])
def test_ring_order_bit_exact(orc, N):
    assert np.array_equal(ra.ring_order(N).cpu().numpy(), orc.ring_order(N))


# ------------------------------------------------------------------ ring attention
SMALL = [
    # b, S, h, n_kv, d, N, layout, causal
    (1, 1024, 2, 2, 64, 4, CONTIGUOUS, False),     # the tiny workload (g = 1, d = 64)
    (1, 1024, 8, 2, 128, 4, CONTIGUOUS, False),
    (1, 1024, 8, 2, 128, 4, CONTIGUOUS, True),
    (1, 1024, 8, 2, 128, 4, STRIPED, True),
    (2, 2048, 8, 2, 128, 8, STRIPED, True),
    (1, 768, 4, 4, 64, 2, STRIPED, True),          # g = 1 causal
    (1, 600, 8, 2, 128, 3, CONTIGUOUS, True),      # ragged: L = 200
    (1, 600, 8, 2, 128, 3, STRIPED, True),
    (1, 600, 6, 2, 64, 3, STRIPED, False),         # g = 3 (odd), ragged, non-causal
    (1, 300, 4, 1, 128, 1, CONTIGUOUS, True),      # N = 1, ragged single shard
    (1, 64, 8, 2, 128, 1, STRIPED, True),          # shorter than one tile
    (1, 1, 2, 1, 64, 1, CONTIGUOUS, True),         # a single token
    (1, 1024, 8, 2, 128, 4, ZIGZAG, True),         # zig-zag: half-blocks of one tile
    (2, 2048, 8, 2, 128, 8, ZIGZAG, True),
    (1, 2048, 4, 4, 64, 2, ZIGZAG, True),          # g = 1, d = 64, four-tile half-blocks
    (1, 1536, 6, 2, 64, 2, ZIGZAG, False),         # g = 3 (odd), non-causal
    (1, 256, 4, 1, 128, 1, ZIGZAG, True),          # N = 1: one shard, two half-blocks
]


@pytest.mark.parametrize("b,S,h,n_kv,d,N,layout,causal", SMALL)
def test_ring_attention_matches_oracle(orc, b, S, h, n_kv, d, N, layout, causal):
    q, k, v = make_inputs(b, S, h, n_kv, d, seed=S + h + d + N)
    ref_o, ref_l = orc.attn_fwd_rows(q, k, v, causal)
    out, lse = _ring(*_dev(q, k, v), N, layout, causal)
    ra.stream_check()
    _cmp(out, lse, ref_o, ref_l)


def test_layouts_agree_and_results_are_deterministic():
    q, k, v = _dev(*make_inputs(1, 4096, 8, 2, 128, seed=5))
    oc, lc = _ring(q, k, v, 8, CONTIGUOUS, True)
    os_, ls_ = _ring(q, k, v, 8, STRIPED, True)
    oz, lz = _ring(q, k, v, 8, ZIGZAG, True)
    ra.stream_check()
    # each path is within O_TOL of the exact result; P is rounded to bf16 on
    # all, in different accumulation orders
    for o_, l_ in ((os_, ls_), (oz, lz)):
        assert (oc - o_).abs().max().item() < O_TOL
        assert (lc - l_).abs().max().item() < 1e-4
    o2, l2 = _ring(q, k, v, 8, STRIPED, True)
    assert torch.equal(o2, os_) and torch.equal(l2, ls_)


def test_custom_scale(orc):
    q, k, v = make_inputs(1, 512, 4, 2, 128, seed=77)
    ref_o, ref_l = orc.attn_fwd_rows(q, k, v, True, scale=0.05)
    out, lse = _ring(*_dev(q, k, v), 4, STRIPED, True, scale=0.05)
    _cmp(out, lse, ref_o, ref_l)


# ------------------------------------------------------------------ block step
@pytest.mark.parametrize("Lq,Lk,causal,g,d", [
    (256, 256, False, 4, 128), (200, 333, True, 4, 128), (128, 512, True, 1, 64),
    (384, 130, True, 2, 128), (64, 1000, False, 3, 64),
])
def test_block_step_matches_oracle_update(orc, Lq, Lk, causal, g, d):
    n_kv = 2
    h = g * n_kv
    q, _, _ = make_inputs(1, Lq, h, n_kv, d, seed=Lq)
    _, k, v = make_inputs(1, Lk, h, n_kv, d, seed=Lk + 1)
    rng = np.random.default_rng(Lq + Lk)
    q_pos = np.sort(rng.choice(4 * (Lq + Lk), Lq, replace=False)).astype(np.int32)
    k_pos = np.sort(rng.choice(4 * (Lq + Lk), Lk, replace=False)).astype(np.int32)
    scale = 1.0 / np.sqrt(d)
    # a non-trivial starting state from a first block
    q0, k0, v0 = make_inputs(1, 192, h, n_kv, d, seed=3)
    k0 = k0[:, :192]
    v0 = v0[:, :192]
    k0_pos = np.sort(rng.choice(4 * (Lq + Lk), 192, replace=False)).astype(np.int32)
    st_ref = orc.new_state(1, Lq, h, d)
    orc.block_update(q, k0, v0, q_pos, k0_pos, causal, scale, st_ref)
    orc.block_update(q, k, v, q_pos, k_pos, causal, scale, st_ref)

    qd, kd, vd, k0d, v0d = _dev(q, k, v, k0.contiguous(), v0.contiguous())
    qp, kp, k0p = (torch.from_numpy(a).cuda() for a in (q_pos, k_pos, k0_pos))
    st = ra.new_state(1, Lq, h, d, "cuda")
    ra.block_step(qd, k0d, v0d, st, qp, k0p, causal)
    ra.block_step(qd, kd, vd, st, qp, kp, causal)
    ra.stream_check()
    m, l, o = (t.double().cpu().numpy() for t in st)
    rm, rl, ro = st_ref
    fin = np.isfinite(rm)
    assert np.array_equal(np.isfinite(m), fin)
    # the state itself: m is the exact running max, l and O relative to it
    assert np.abs(m[fin] - rm[fin]).max() <= 1e-4
    rel_l = np.abs(l[fin] - rl[fin]) / rl[fin]
    assert rel_l.max() <= 1e-3
    # normalised results
    out, lse = ra.finalize(st, lse=torch.full_like(st[0], float("nan")))
    r_out, r_lse = orc.finalize(st_ref)
    _cmp(out, lse, r_out, r_lse)


def _block_steps_vs_oracle(orc, q, blocks, q_pos, causal=True, k_pos_offset=0):
    """Fold the key/value blocks [(k, v, k_pos), ...] into one state with
    ra_block_step and with the oracle's update; compare the finalized rows.
    k_pos_offset > 0 hands the library k_pos at that many int32 past a
    16-byte boundary (the position scans then load one int at a time)."""
    b, Lq, h, d = q.shape
    scale = 1.0 / np.sqrt(d)
    st_ref = orc.new_state(b, Lq, h, d)
    st = ra.new_state(b, Lq, h, d, "cuda")
    qd = _dev(q)[0]
    qp = torch.from_numpy(q_pos).cuda()
    for k, v, k_pos in blocks:
        orc.block_update(q, k, v, q_pos, k_pos, causal, scale, st_ref)
        kd, vd = _dev(k, v)
        kp = torch.zeros(len(k_pos) + k_pos_offset, dtype=torch.int32, device="cuda")
        kp[k_pos_offset:] = torch.from_numpy(k_pos).cuda()
        kp = kp[k_pos_offset:]
        assert kp.data_ptr() % 16 == 4 * k_pos_offset
        ra.block_step(qd, kd, vd, st, qp, kp, causal)
    ra.stream_check()
    out, lse = ra.finalize(st, lse=torch.full_like(st[0], float("nan")))
    r_out, r_lse = orc.finalize(st_ref)
    _cmp(out, lse, r_out, r_lse)


@pytest.mark.parametrize("sort_keys,k_pos_offset", [(True, 0), (False, 0), (True, 1)])
def test_block_step_irregular_positions(orc, sort_keys, k_pos_offset):
    """A causal block step over >= 16K keys runs, per query tile, the leading
    key tiles every row sees in full without the mask and the rest with it;
    with positions neither contiguous nor (for the keys) sorted that split
    point differs from tile to tile, and the result must not depend on it.
    With sorted keys the three query tiles see 24, 71 and 116 leading tiles
    in full: the first stays in the masked launch (a short prefix), the
    others split; the last key tile is ragged (20,000 keys)."""
    Lq, Lk, h, n_kv, d = 384, 20000, 4, 2, 128
    rng = np.random.default_rng(27 + sort_keys)
    q, _, _ = make_inputs(1, Lq, h, n_kv, d, seed=28)
    _, k, v = make_inputs(1, Lk, h, n_kv, d, seed=29)
    q_pos = np.sort(rng.choice(np.arange(4000, 26000), Lq, replace=False)).astype(np.int32)
    k_pos = rng.choice(26000, Lk, replace=False).astype(np.int32)
    if sort_keys:
        k_pos = np.sort(k_pos)
    _block_steps_vs_oracle(orc, q, [(k, v, k_pos)], q_pos, k_pos_offset=k_pos_offset)


@pytest.mark.parametrize("b,Lk", [(1, 16512), (2, 16512), (1, 16400)])
def test_block_step_key_block_wholly_before_or_after(orc, b, Lk):
    """Ring steps off the diagonal: a key block wholly before the queries
    (every tile seen in full: the masked launch has nothing left) and one
    wholly after them (the unmasked launch has nothing: the state stays as
    it was, bit for bit).  129 key tiles: the two-launch path; with 16,400
    keys the last tile is ragged and is the first launch's position-masked
    tile after the 128 complete ones."""
    Lq, h, n_kv, d = 256, 4, 2, 64
    q, _, _ = make_inputs(b, Lq, h, n_kv, d, seed=31)
    _, k, v = make_inputs(b, Lk, h, n_kv, d, seed=32)
    _, k2, v2 = make_inputs(b, Lk, h, n_kv, d, seed=33)
    q_pos = np.arange(40000, 40000 + Lq, dtype=np.int32)
    before = np.arange(0, 2 * Lk, 2, dtype=np.int32)           # all < 40000
    after = np.arange(50000, 50000 + Lk, dtype=np.int32)       # all > every query
    _block_steps_vs_oracle(orc, q, [(k, v, before)], q_pos)
    st = ra.new_state(b, Lq, h, d, "cuda")
    qd, kd, vd, k2d, v2d = _dev(q, k, v, k2, v2)
    qp = torch.from_numpy(q_pos).cuda()
    n0 = ra.launch_count()
    ra.block_step(qd, kd, vd, st, qp, torch.from_numpy(before).cuda(), True)
    assert ra.launch_count() - n0 == 2       # unmasked launch, then masked
    saved = [t.clone() for t in st]
    ra.block_step(qd, k2d, v2d, st, qp, torch.from_numpy(after).cuda(), True)
    ra.stream_check()
    for a, b_ in zip(st, saved):
        assert torch.equal(a, b_)


# ------------------------------------------------------------------ peaked attention
# Inputs from parity_util.peaked_inputs: every query has one key aligned with
# it, placed in the last shard of its ring order that holds a key it sees, so
# its row max jumps late in the walk, in most rows by more than 8 log2 units
# after the exponent shift was set.  That drives, on purpose, the rescale of
# O and l by 2^(old shift - new shift) and (once every row of a warp has a
# shift, when P is formed before the tile's max is known) the forming of a
# tile's P again against the new shift.  At S = 2048 every tile takes the
# hi + lo path; at S >= 8192 most take the plain bf16 path.
PEAKED = [
    # S, h, n_kv, d, N, layout, causal
    (2048, 8, 2, 128, 4, STRIPED, True),
    (2048, 8, 2, 128, 4, CONTIGUOUS, True),
    (2048, 8, 2, 128, 4, ZIGZAG, True),
    (2048, 8, 2, 128, 4, CONTIGUOUS, False),
    (16384, 8, 2, 128, 4, STRIPED, True),
    (16384, 8, 2, 128, 4, CONTIGUOUS, True),
    (16384, 8, 2, 128, 4, ZIGZAG, True),
    (16384, 8, 2, 128, 4, CONTIGUOUS, False),
    (8192, 6, 2, 64, 4, STRIPED, True),           # d = 64, g = 3
]


@pytest.mark.parametrize("S,h,n_kv,d,N,layout,causal", PEAKED)
def test_peaked_forward(orc, S, h, n_kv, d, N, layout, causal):
    q, k, v = peaked_inputs(orc, 1, S, h, n_kv, d, N, layout, causal, seed=S + layout + d)
    ref_o, ref_l = orc.attn_fwd_rows(q, k, v, causal)
    out, lse = _ring(*_dev(q, k, v), N, layout, causal)
    ra.stream_check()
    _cmp(out, lse, ref_o, ref_l)
    _rel_plain(out.double().cpu().numpy(), ref_o, plain_rows(orc, layout, S, N, causal),
               "peaked")


def test_peaked_block_steps_jump_at_last_step(orc):
    """Block steps over the ring (striped, causal): each query's aligned key
    lies in the last shard it meets, so its running max jumps at the last
    step.  The state after the walk -- m the exact running max, l and O
    relative to it -- and the finalized result match the oracle's recurrence
    over the same blocks in the same order."""
    b, S, h, n_kv, d, N = 1, 2048, 8, 2, 128, 4
    q, k, v = peaked_inputs(orc, b, S, h, n_kv, d, N, STRIPED, True, seed=7)
    _, _, tok = orc.position_map(STRIPED, S, N)
    order = orc.ring_order(N)
    qd, kd, vd = _dev(q, k, v)
    scale = 1.0 / np.sqrt(d)
    for i in range(N):
        qt = tok[i].astype(np.int64)
        st_ref = orc.new_state(b, qt.size, h, d)
        qi = q[:, torch.from_numpy(qt)].contiguous()
        qit = torch.from_numpy(qt).cuda()
        qid = qd[:, qit].contiguous()
        st = ra.new_state(b, qt.size, h, d, "cuda")
        for s_ in range(N):
            kt = tok[order[i, s_]].astype(np.int64)
            ktc = torch.from_numpy(kt)
            orc.block_update(qi, k[:, ktc].contiguous(), v[:, ktc].contiguous(), tok[i],
                             tok[order[i, s_]], True, scale, st_ref)
            ra.block_step(qid, kd[:, ktc.cuda()].contiguous(), vd[:, ktc.cuda()].contiguous(),
                          st, qit.int(), ktc.cuda().int(), True)
        ra.stream_check()
        m, l, o = (t.double().cpu().numpy() for t in st)
        rm, rl, ro = st_ref
        assert np.abs(m - rm).max() <= 1e-4
        assert (np.abs(l - rl) / rl).max() <= 1e-3
        out, lse = ra.finalize(st, lse=torch.full_like(st[0], float("nan")))
        r_out, r_lse = orc.finalize(st_ref)
        _cmp(out, lse, r_out, r_lse)


def test_peaked_block_step_max_in_last_tile(orc):
    """One block step on a running state, whose block's last key tile holds
    keys aligned with every query: the row max jumps in the block's last tile,
    and the epilogue re-references the merged state to the exact new max."""
    b, Lq, Lk, h, n_kv, d = 1, 256, 640, 4, 2, 128
    g = h // n_kv
    q, _, _ = make_inputs(b, Lq, h, n_kv, d, seed=91)
    _, k, v = make_inputs(b, Lk, h, n_kv, d, seed=92)
    k0, v0 = make_inputs(b, 384, h, n_kv, d, seed=93)[1:]
    kf = k.float()
    for r in range(Lq):           # keys 512 + r % 128 of the last tile align with query r
        for kh in range(n_kv):
            kf[0, 512 + r % 128, kh] = 0.0
    for r in range(Lq):
        for kh in range(n_kv):
            kf[0, 512 + r % 128, kh] += 1.5 * q[0, r, kh * g + r % g].float() / np.sqrt(2.0)
    k = kf.to(torch.bfloat16)
    q_pos = np.arange(10000, 10000 + Lq, dtype=np.int32)
    k0_pos = np.arange(384, dtype=np.int32)
    k_pos = np.arange(1000, 1000 + Lk, dtype=np.int32)
    scale = 1.0 / np.sqrt(d)
    st_ref = orc.new_state(b, Lq, h, d)
    orc.block_update(q, k0, v0, q_pos, k0_pos, True, scale, st_ref)
    orc.block_update(q, k, v, q_pos, k_pos, True, scale, st_ref)
    qd, kd, vd, k0d, v0d = _dev(q, k, v, k0, v0)
    qp, kp, k0p = (torch.from_numpy(a).cuda() for a in (q_pos, k_pos, k0_pos))
    st = ra.new_state(b, Lq, h, d, "cuda")
    ra.block_step(qd, k0d, v0d, st, qp, k0p, True)
    ra.block_step(qd, kd, vd, st, qp, kp, True)
    ra.stream_check()
    m, l, o = (t.double().cpu().numpy() for t in st)
    rm, rl, ro = st_ref
    assert np.abs(m - rm).max() <= 1e-4
    assert (np.abs(l - rl) / rl).max() <= 1e-3
    out, lse = ra.finalize(st, lse=torch.full_like(st[0], float("nan")))
    r_out, r_lse = orc.finalize(st_ref)
    _cmp(out, lse, r_out, r_lse)


@pytest.mark.parametrize("layout", [CONTIGUOUS, STRIPED, ZIGZAG])
def test_block_steps_over_ring_reproduce_full_attention(orc, layout):
    """ra_block_step over the N shards in ring order, then ra_finalize,
    equals the direct definition (the pages' exactness claim)."""
    b, S, h, n_kv, d, N = 1, 1024, 8, 2, 128, 4
    q, k, v = make_inputs(b, S, h, n_kv, d, seed=99)
    ref_o, ref_l = orc.attn_fwd_rows(q, k, v, True)
    _, _, tok = orc.position_map(layout, S, N)
    order = orc.ring_order(N)
    out, lse = _nan_out(b, S, h, d, "cpu")
    qd, kd, vd = _dev(q, k, v)
    for i in range(N):
        qt = torch.from_numpy(tok[i].astype(np.int64)).cuda()
        qi = qd[:, qt].contiguous()
        st = ra.new_state(b, qi.shape[1], h, d, "cuda")
        for s in range(N):
            kt = torch.from_numpy(tok[order[i, s]].astype(np.int64)).cuda()
            ra.block_step(qi, kd[:, kt].contiguous(), vd[:, kt].contiguous(), st,
                          qt.int(), kt.int(), True)
        o_i, l_i = ra.finalize(st)
        out[:, qt.cpu()] = o_i.cpu()
        lse[:, :, qt.cpu()] = l_i.cpu()
    ra.stream_check()
    _cmp(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("Lq,Lk,causal,g,d,splits", [
    (256, 4096, True, 4, 128, 0), (256, 4096, True, 4, 128, 1), (256, 4096, True, 4, 128, 5),
    (200, 1000, True, 2, 64, 3), (128, 2048, False, 1, 128, 0), (384, 640, True, 3, 128, 64),
    # splits of >= 512 visible keys per row take the plain bf16 P path
    (256, 16384, True, 4, 128, 2), (128, 12288, False, 2, 64, 0),
])
def test_chunked_prefill_matches_oracle(orc, Lq, Lk, causal, g, d, splits):
    """The last Lq tokens of an Lk-token sequence attend to all Lk keys
    (their own included), keys split over concurrent block steps."""
    n_kv = 2
    h = g * n_kv
    q, _, _ = make_inputs(1, Lq, h, n_kv, d, seed=Lq + 5)
    _, k, v = make_inputs(1, Lk, h, n_kv, d, seed=Lk + 6)
    q_pos = np.arange(Lk - Lq, Lk, dtype=np.int32)
    k_pos = np.arange(Lk, dtype=np.int32)
    st = orc.new_state(1, Lq, h, d)
    orc.block_update(q, k, v, q_pos, k_pos, causal, 1.0 / np.sqrt(d), st)
    ref_o, ref_l = orc.finalize(st)
    qd, kd, vd = _dev(q, k, v)
    qp, kp = (torch.from_numpy(x).cuda() for x in (q_pos, k_pos))
    out, lse = _nan_out(1, Lq, h, d)
    ra.chunked_prefill(qd, kd, vd, qp, kp, causal, n_splits=splits, out=out, lse=lse)
    ra.stream_check()
    _cmp(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("sort_keys", [True, False])
def test_chunked_prefill_irregular_positions(orc, sort_keys):
    """Causal prefill with positions that are neither contiguous nor (for the
    keys) sorted: the leading key tiles every row of a query tile sees in
    full run without the mask and the rest with it, so the split point
    differs from tile to tile; the result must not depend on it."""
    Lq, Lk, h, n_kv, d = 384, 5000, 4, 2, 128
    rng = np.random.default_rng(17 + sort_keys)
    q, _, _ = make_inputs(1, Lq, h, n_kv, d, seed=18)
    _, k, v = make_inputs(1, Lk, h, n_kv, d, seed=19)
    q_pos = np.sort(rng.choice(np.arange(2000, 9000), Lq, replace=False)).astype(np.int32)
    k_pos = rng.choice(9000, Lk, replace=False).astype(np.int32)
    if sort_keys:
        k_pos = np.sort(k_pos)
    st = orc.new_state(1, Lq, h, d)
    orc.block_update(q, k, v, q_pos, k_pos, True, 1.0 / np.sqrt(d), st)
    ref_o, ref_l = orc.finalize(st)
    qd, kd, vd = _dev(q, k, v)
    qp, kp = (torch.from_numpy(x).cuda() for x in (q_pos, k_pos))
    for splits in (0, 3):
        out, lse = _nan_out(1, Lq, h, d)
        ra.chunked_prefill(qd, kd, vd, qp, kp, True, n_splits=splits, out=out, lse=lse)
        ra.stream_check()
        _cmp(out, lse, ref_o, ref_l)


def test_chunked_prefill_batch_of_two(orc):
    """b = 2: the split states and their combination are per batch row."""
    b, Lq, Lk, h, n_kv, d = 2, 200, 1500, 4, 2, 128
    q, _, _ = make_inputs(b, Lq, h, n_kv, d, seed=61)
    _, k, v = make_inputs(b, Lk, h, n_kv, d, seed=62)
    q_pos = np.arange(Lk - Lq, Lk, dtype=np.int32)
    k_pos = np.arange(Lk, dtype=np.int32)
    st = orc.new_state(b, Lq, h, d)
    orc.block_update(q, k, v, q_pos, k_pos, True, 1.0 / np.sqrt(d), st)
    ref_o, ref_l = orc.finalize(st)
    qd, kd, vd = _dev(q, k, v)
    qp, kp = (torch.from_numpy(x).cuda() for x in (q_pos, k_pos))
    out, lse = _nan_out(b, Lq, h, d)
    ra.chunked_prefill(qd, kd, vd, qp, kp, True, n_splits=4, out=out, lse=lse)
    ra.stream_check()
    _cmp(out, lse, ref_o, ref_l)


def test_block_step_batch_of_two_non_causal(orc):
    b, Lq, Lk, h, n_kv, d = 2, 256, 384, 8, 2, 64
    q, _, _ = make_inputs(b, Lq, h, n_kv, d, seed=71)
    _, k, v = make_inputs(b, Lk, h, n_kv, d, seed=72)
    pos_q = np.arange(Lq, dtype=np.int32)
    pos_k = np.arange(Lk, dtype=np.int32)
    st_ref = orc.new_state(b, Lq, h, d)
    orc.block_update(q, k, v, pos_q, pos_k, False, 1.0 / np.sqrt(d), st_ref)
    qd, kd, vd = _dev(q, k, v)
    st = ra.new_state(b, Lq, h, d, "cuda")
    ra.block_step(qd, kd, vd, st, causal=False)
    out, lse = ra.finalize(st, lse=torch.full_like(st[0], float("nan")))
    ra.stream_check()
    r_out, r_lse = orc.finalize(st_ref)
    _cmp(out, lse, r_out, r_lse)


def test_chunked_prefill_without_keys():
    q, k, v = _dev(*make_inputs(1, 128, 4, 2, 64, seed=1))
    pos = torch.arange(128, dtype=torch.int32, device="cuda")
    out, lse = _nan_out(1, 128, 4, 64)
    ra.chunked_prefill(q, k[:, :0].contiguous(), v[:, :0].contiguous(), pos, pos[:0].contiguous(),
                       True, out=out, lse=lse)
    ra.stream_check()
    assert torch.count_nonzero(out).item() == 0
    assert torch.isneginf(lse).all().item()


def test_block_step_state_survives_a_host_round_trip():
    """Checkpoint / resume of the only resumable state, (m, l, O) between
    block steps: stop after ring step k, copy the state to the host and back,
    resume; the result is bit-identical to an uninterrupted walk."""
    b, S, h, n_kv, d, N = 1, 1024, 8, 2, 128, 4
    q, k, v = (t.cuda() for t in make_inputs(b, S, h, n_kv, d, seed=41))
    _, _, tok = ra.position_map(STRIPED, S, N)
    order = ra.ring_order(N).cpu().numpy()
    i = 2
    qt = tok[i].long()
    qi = q[:, qt].contiguous()
    results = []
    for stop in (None, 1):
        st = ra.new_state(b, qi.shape[1], h, d, "cuda")
        for s_ in range(N):
            kt = tok[int(order[i, s_])].long()
            ra.block_step(qi, k[:, kt].contiguous(), v[:, kt].contiguous(), st, tok[i],
                          tok[int(order[i, s_])], True)
            if s_ == stop:
                host = [t.cpu() for t in st]
                st = tuple(t.cuda() for t in host)
        results.append(ra.finalize(st))
    ra.stream_check()
    (o1, l1), (o2, l2) = results
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_merge_matches_oracle(orc):
    b, S, h, n_kv, d = 1, 512, 4, 2, 128
    q, k, v = make_inputs(b, S, h, n_kv, d, seed=12)
    pos = np.arange(S, dtype=np.int32)
    sel = np.random.default_rng(0).permutation(S)
    parts_ref, parts_gpu = [], []
    qd, kd, vd = _dev(q, k, v)
    for idx in (np.sort(sel[:200]), np.sort(sel[200:])):
        st = orc.new_state(b, S, h, d)
        ti = torch.from_numpy(idx)
        orc.block_update(q, k[:, ti], v[:, ti], pos, pos[idx], True, 1 / np.sqrt(d), st)
        parts_ref.append(orc.finalize(st))
        sg = ra.new_state(b, S, h, d, "cuda")
        tid = ti.cuda()
        ra.block_step(qd, kd[:, tid].contiguous(), vd[:, tid].contiguous(), sg,
                      torch.from_numpy(pos).cuda(), torch.from_numpy(pos[idx]).cuda(), True)
        parts_gpu.append(ra.finalize(sg))
    o, lse = ra.merge(parts_gpu[0][0], parts_gpu[0][1], parts_gpu[1][0], parts_gpu[1][1],
                      *_nan_out(b, S, h, d))
    ro, rl = orc.merge(parts_ref[0][0], parts_ref[0][1], parts_ref[1][0], parts_ref[1][1])
    ra.stream_check()
    _cmp(o, lse, ro, rl)
    # a side with no keys leaves the other untouched
    empty_o = torch.zeros_like(o)
    empty_l = torch.full_like(lse, float("-inf"))
    o2, l2 = ra.merge(o, lse, empty_o, empty_l)
    assert torch.allclose(o2, o, atol=1e-6) and torch.allclose(l2, lse, atol=1e-6)


# ------------------------------------------------------------------ failure detection
def test_bounded_wait_reports_timeout():
    """A wait on a barrier nothing arrives on runs out and is reported; the
    context stays usable."""
    ra.selftest_wait_timeout(200000)
    with pytest.raises(ra.RAError) as ei:
        ra.stream_check()
    assert ei.value.status == ra.RA_ERR_DEVICE_TIMEOUT
    ra.stream_check()   # cleared
    q, k, v = _dev(*make_inputs(1, 256, 2, 1, 64, seed=1))
    ra.ring_attention(q, k, v, 2, STRIPED, True)
    ra.stream_check()


# ------------------------------------------------------------------ full-size workloads
def _workload_parity(orc, name, layouts=None):
    """The workload's sampled rows against the oracle: the north-star
    max-abs bounds on every sampled row, and on the rows that take the plain
    bf16 path (nearly all of the work) the error relative to max|ref|."""
    w = WORKLOADS[name]
    q, k, v = workload_inputs(w)[:3]
    rows = sample_rows(w.S, w.n_shards, w.rows_per_head, w.seed)
    ref_o, ref_l = orc.attn_fwd_rows(q, k, v, w.causal, rows=rows)
    qd, kd, vd = _dev(q, k, v)
    errs = {}
    for layout in (layouts or w.layouts):
        out, lse = _ring(qd, kd, vd, w.n_shards, layout, w.causal)
        ra.stream_check()
        tag = ("contiguous_", "striped_", "zigzag_")[layout]
        errs[layout] = _cmp(out, lse, ref_o, ref_l, rows, tag=tag)
        plain = plain_rows(orc, layout, w.S, w.n_shards, w.causal)[rows]
        o = out.index_select(1, torch.from_numpy(rows).cuda()).double().cpu().numpy()
        errs[layout] += (_rel_plain(o, ref_o, plain, f"{name} layout {layout}", tag=tag),)
        del out, lse
    return errs


def test_workload_tiny_all_rows(orc):
    _workload_parity(orc, "tiny")


def test_workload_noncausal_32k(orc):
    _workload_parity(orc, "noncausal32k")


@pytest.mark.slow
def test_workload_noncausal_32k_all_rows(orc):
    """The non-causal 32K GQA configuration with the oracle on every one of
    its 32,768 rows, for one query head of each of the 8 KV groups (heads
    0, 4, ..., 28; about 4.4e12 fp64 FLOP, a few minutes on the host).  The
    oracle runs the sub-problem of those heads, which pairs head 4j with KV
    head j exactly as the full problem does."""
    w = WORKLOADS["noncausal32k"]
    q, k, v = workload_inputs(w)[:3]
    g = w.h // w.n_kv
    heads = list(range(0, w.h, g))
    ref_o, ref_l = orc.attn_fwd_rows(q[:, :, heads].contiguous(), k, v, False,
                                     scale=1.0 / np.sqrt(w.d))
    out, lse = _ring(*_dev(q, k, v), w.n_shards, CONTIGUOUS, False)
    ra.stream_check()
    hsel = torch.tensor(heads, device="cuda")
    o = out.index_select(2, hsel)
    l = lse.index_select(1, hsel)
    del out, lse
    err_o, err_l = _cmp(o, l, ref_o, ref_l)
    _rel_plain(o.double().cpu().numpy(), ref_o, np.ones(w.S, dtype=bool), "noncausal32k all rows")


def test_workload_causal_64k_both_layouts(orc):
    _workload_parity(orc, "causal64k")


def test_workload_causal_64k_zigzag(orc):
    _workload_parity(orc, "causal64k", layouts=(ZIGZAG,))


def test_workload_causal_256k_striped(orc):
    _workload_parity(orc, "causal256k")


def test_launch_counter_and_exp2_probe():
    """The library's launch counter sees each kernel it starts (the forward
    is one launch; the backward a pre-pass and the main kernel), and the
    exp2-rate probe runs and writes finite values."""
    q, k, v, do = _dev(*make_inputs(1, 512, 4, 2, 128, seed=9, with_dout=True))
    n0 = ra.launch_count()
    out, lse = ra.ring_attention(q, k, v, 2, STRIPED, True)
    n1 = ra.launch_count()
    ra.ring_attention_bwd(q, k, v, out, lse, do, 2, STRIPED, True)
    n2 = ra.launch_count()
    ra.stream_check()
    assert n1 - n0 == 1 and n2 - n1 == 2
    sink, evaluated = ra.ex2_probe(4)
    ra.stream_check()
    assert evaluated == 32 * sink.numel() and bool(torch.isfinite(sink).all())
