"""Pins of the FLOP / byte / utilisation accounting used for reporting,
against the worked example printed on the third page."""

import os

import pytest

from long_context_exact_gb300 import accounting as acc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "accounting_worked_example.txt")
S, N, h, n_kv, d, b = 262144, 8, 32, 8, 128, 1


def _golden():
    out = {}
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            k, v, tol = line.split()
            out[k] = (float(v), float(tol))
    return out


def _ours():
    o = {
        "step_flops": acc.ring_step_flops(b, S, N, h, d),
        "step_kv_bytes": acc.ring_step_kv_bytes(b, S, N, n_kv, d),
        "received_bytes": acc.received_bytes(b, S, N, n_kv, d),
        "step_intensity": acc.step_intensity(S, N, h, n_kv),
        "util_half_N8": acc.causal_utilisation_contiguous(8, half_diagonal=True),
    }
    for n in (2, 4, 8, 16, 32):
        o[f"util_N{n}"] = acc.causal_utilisation_contiguous(n)
    return o


@pytest.mark.parametrize("name", sorted(_golden()))
def test_accounting_matches_printed_values(name):
    val, tol = _golden()[name]
    ours = _ours()[name]
    assert abs(ours - val) <= max(tol * abs(val), 1e-9) + (0.0005 if name.startswith("util") else 0)


def test_useful_flops_convention():
    # 4 b S^2 h d non-causal, half of it causal (section 2, first invariant)
    assert acc.fwd_useful_flops(1, S, h, d, False) == 4.0 * S * S * h * d
    assert acc.fwd_useful_flops(1, S, h, d, True) == 2.0 * S * S * h * d
    assert acc.bwd_useful_flops(2, 65536, h, d, True) == 2.5 * 2 * 2.0 * 65536 ** 2 * h * d
    # N steps of one device add up to the device's share of the total
    assert abs(N * acc.ring_step_flops(1, S, N, h, d) * N - acc.fwd_useful_flops(1, S, h, d, False)) < 1.0
