"""GPU checks of the host-buffer pipeline (``ra_pipeline_*``) and of
``ra_host_alloc``: steps submitted back to back on two alternating input sets
give the results of the device-buffer calls (forward bit for bit, gradients
to fp32 summation order) and of the fp64 oracle."""

import numpy as np
import pytest
import torch

from long_context_exact_gb300 import binding as ra
from long_context_exact_gb300.inputs import STRIPED, ZIGZAG, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_exact_gb300 import build as b
    b.build()
    ra.load()


def _device_run(q, k, v, do, N, layout, causal):
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    out, lse = ra.ring_attention(qd, kd, vd, N, layout, causal)
    res = [out.cpu(), lse.cpu()]
    if do is not None:
        dq, dk, dv = ra.ring_attention_bwd(qd, kd, vd, out, lse, do.cuda(), N, layout, causal)
        res += [dq.cpu(), dk.cpu(), dv.cpu()]
    ra.stream_check()
    return res


def _host(t, pinned):
    if not pinned:
        return None, t.contiguous()
    hb = ra.HostBuffer(t.shape, t.dtype)
    hb.tensor.copy_(t)
    return hb, hb.tensor


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("backward", [True, False])
def test_pipeline_matches_device_calls(orc, pinned, backward):
    b, S, h, n_kv, d, N, layout, causal = 1, 1024, 8, 2, 128, 4, STRIPED, True
    sets = [make_inputs(b, S, h, n_kv, d, seed=s, with_dout=True) for s in (11, 12)]
    keep = []
    host_in = []
    for q, k, v, do in sets:
        row = []
        for t in (q, k, v, do):
            hb, ht = _host(t, pinned)
            keep.append(hb)
            row.append(ht)
        host_in.append(row)
    shapes = [(b, S, h, d), (b, h, S), (b, S, h, d), (b, S, n_kv, d), (b, S, n_kv, d)]
    n_out = 5 if backward else 2
    host_out = []
    for _ in range(3):
        row = []
        for shp in shapes[:n_out]:
            hb, ht = _host(torch.full(shp, float("nan")), pinned)
            keep.append(hb)
            row.append(ht)
        host_out.append(row + [None] * (5 - n_out))
    pl = ra.Pipeline(S, N, layout, causal, b, h, n_kv, d, backward=backward)
    try:
        for step in range(3):
            q, k, v, do = host_in[step % 2]
            pl.submit(q, k, v, do if backward else None, *host_out[step])
        pl.sync()
    finally:
        pl.close()
    for step in range(3):
        q, k, v, do = sets[step % 2]
        ref = _device_run(q, k, v, do if backward else None, N, layout, causal)
        got = host_out[step][:n_out]
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
        for a, r in zip(got[2:], ref[2:]):
            assert float((a - r).abs().max()) <= 1e-5
    q, k, v, do = sets[0]
    ro, rl = orc.attn_fwd_rows(q, k, v, causal)
    assert float(np.abs(host_out[0][0].double().numpy() - ro).max()) <= 1e-2
    assert float(np.abs(host_out[0][1].double().numpy() - rl).max()) <= 1e-3
    if backward:
        rq, rk, rv = orc.attn_bwd_rows(q, k, v, do, causal)
        for a, r in zip(host_out[0][2:5], (rq, rk, rv)):
            assert float(np.abs(a.double().numpy() - r).max()) <= 1e-2
    del keep


def test_pipeline_reports_unsupported_shapes():
    # zig-zag with half-blocks that are not whole 128-token tiles
    b, S, h, n_kv, d, N = 1, 768, 4, 2, 128, 4
    q, k, v, do = make_inputs(b, S, h, n_kv, d, seed=1, with_dout=True)
    pl = ra.Pipeline(S, N, ZIGZAG, True, b, h, n_kv, d, backward=True)
    try:
        with pytest.raises(ra.RAError) as ei:
            pl.submit(q, k, v, do)
        assert ei.value.status == ra.RA_ERR_UNSUPPORTED
    finally:
        pl.close()


def test_host_alloc_round_trip():
    hb = ra.HostBuffer((3, 1000), torch.float32)
    hb.tensor.copy_(torch.arange(3000, dtype=torch.float32).view(3, 1000))
    dev = hb.tensor.cuda()
    assert torch.equal(dev.cpu(), hb.tensor)
    assert ra.host_numa_node() >= -1
    hb.free()
    assert ra.HostBuffer((0,), torch.float32).nbytes == 0


def test_pipeline_refuses_short_host_buffers():
    b, S, h, n_kv, d, N = 1, 512, 4, 2, 64, 2
    q, k, v, do = make_inputs(b, S, h, n_kv, d, seed=3, with_dout=True)
    pl = ra.Pipeline(S, N, STRIPED, True, b, h, n_kv, d, backward=True)
    try:
        with pytest.raises(ra.RAError) as ei:
            pl.submit(q[:, : S // 2].contiguous(), k, v, do)
        assert ei.value.status == ra.RA_ERR_INVALID_ARG
        out = torch.empty((b, S, h, d // 2))
        with pytest.raises(ra.RAError):
            pl.submit(q, k, v, do, out=out)
    finally:
        pl.close()
