"""Backward on CTA pairs (pair_mode=1, D = 128): parity with the fp64 oracle
on the same seeded inputs as the single-CTA kernel, and agreement with that
kernel to rounding (the two form P and dS with differently ordered fp32
operations, and sum dQ in a different order)."""
import math

import pytest
import torch

from exact_attention_36_gb300 import fa
from exact_attention_36_gb300.inputs import make_qkvdo
from tests._parity import check_backward, sample_rows

pytestmark = pytest.mark.gpu


def _run(B, H, S, causal, seed=0, stress=False, pair_mode=1):
    D = 128
    q, k, v, do = make_qkvdo(B, H, S, D, seed=seed, stress=stress)
    scale = 1.0 / math.sqrt(D)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.backward(qd, kd, vd, o, dod, lse, causal=causal, scale=scale,
                             pair_mode=pair_mode)
    torch.cuda.synchronize()
    assert fa.device_error() == 0
    return q, k, v, do, dq, dk, dv, scale


@pytest.mark.parametrize("S", [1, 2, 100, 127, 128, 129, 255, 256, 257, 300, 383, 640])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths(S, causal):
    # odd numbers of key tiles leave the second CTA of the last pair past S
    q, k, v, do, dq, dk, dv, scale = _run(2, 3, S, causal, seed=S)
    check_backward(q, k, v, do, dq, dk, dv, causal, scale, heads=None)


def test_many_units_per_pair():
    q, k, v, do, dq, dk, dv, scale = _run(3, 40, 768, True, seed=7)
    check_backward(q, k, v, do, dq, dk, dv, True, scale, heads=[(0, 0), (1, 17), (2, 39)])


def test_noncausal_b4_h16_s2048():
    q, k, v, do, dq, dk, dv, scale = _run(4, 16, 2048, False)
    check_backward(q, k, v, do, dq, dk, dv, False, scale, heads=[(0, 0), (3, 15)])


@pytest.mark.parametrize("causal", [False, True])
def test_long_context_s32768_sampled(causal):
    q, k, v, do, dq, dk, dv, scale = _run(1, 16, 32768, causal)
    rows = sample_rows(32768, 64, seed=4)
    check_backward(q, k, v, do, dq, dk, dv, causal, scale, heads=[(0, 15)], rows=rows,
                   cols=rows)


@pytest.mark.parametrize("S,B", [(1024, 16), (4096, 4), (16384, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_stress_sweep(S, B, causal):
    q, k, v, do, dq, dk, dv, scale = _run(B, 16, S, causal, stress=True)
    rows = None if S <= 4096 else sample_rows(S, 128, seed=5)
    check_backward(q, k, v, do, dq, dk, dv, causal, scale, heads=[(0, 0), (B - 1, 15)],
                   rows=rows, cols=rows)


@pytest.mark.parametrize("causal", [False, True])
def test_matches_single_cta_kernel(causal):
    a = _run(2, 4, 1000, causal, seed=3, pair_mode=0)
    b = _run(2, 4, 1000, causal, seed=3, pair_mode=1)
    for x, y in zip(a[4:7], b[4:7]):
        x, y = x.float(), y.float()
        assert ((x - y).norm() / x.norm()).item() <= 2e-3
