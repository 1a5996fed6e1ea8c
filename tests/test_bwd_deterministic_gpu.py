"""Deterministic backward (FlashAttention-4: Algorithm and Kernel Pipelining
Co-Design, Technische samenvatting, Methodologie §3: a deterministic mode
ordered by semaphores): dQ is summed over key tiles in a fixed order, so two
runs on the same inputs agree bit for bit; the results still match the fp64
oracle and the atomic-order backward."""
import math

import pytest
import torch

from exact_attention_36_gb300 import fa
from exact_attention_36_gb300.inputs import make_qkvdo
from tests._parity import check_backward, sample_rows

pytestmark = pytest.mark.gpu


def _inputs(B, H, S, D, causal, seed):
    q, k, v, do = make_qkvdo(B, H, S, D, seed=seed)
    scale = 1.0 / math.sqrt(D)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, causal=causal, scale=scale)
    return (q, k, v, do), (qd, kd, vd, dod, o, lse), scale


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,S,D", [(1, 2, 256, 64), (2, 3, 300, 128), (4, 16, 2048, 128),
                                     (3, 40, 768, 64), (2, 3, 300, 256), (1, 6, 1000, 256)])
def test_deterministic_is_bitwise_repeatable_and_exact(B, H, S, D, causal):
    cpu, (qd, kd, vd, dod, o, lse), scale = _inputs(B, H, S, D, causal, seed=S + D)
    a = fa.backward(qd, kd, vd, o, dod, lse, causal, scale, deterministic=True)
    b = fa.backward(qd, kd, vd, o, dod, lse, causal, scale, deterministic=True)
    torch.cuda.synchronize()
    assert fa.device_error() == 0
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    heads = [(0, 0), (B - 1, H - 1)]
    rows = None if S <= 1024 else sample_rows(S, 128, seed=6)
    check_backward(*cpu, *a, causal, scale, heads=heads, rows=rows, cols=rows)
    # the atomic-order backward differs only by the order of fp32 additions:
    # dQ's, and without a causal mask at D = 64 and 128 (where the fixed order
    # visits the query blocks rotated) dK's and dV's
    c = fa.backward(qd, kd, vd, o, dod, lse, causal, scale)
    if causal or D == 256:
        assert torch.equal(a[1], c[1]) and torch.equal(a[2], c[2])
    for x, y in zip(a, c):
        x, y = x.float(), y.float()
        assert ((x - y).norm() / y.norm()).item() <= 2e-3


def test_deterministic_long_context_sampled():
    cpu, (qd, kd, vd, dod, o, lse), scale = _inputs(1, 16, 32768, 128, True, seed=0)
    a = fa.backward(qd, kd, vd, o, dod, lse, True, scale, deterministic=True)
    b = fa.backward(qd, kd, vd, o, dod, lse, True, scale, deterministic=True)
    torch.cuda.synchronize()
    assert fa.device_error() == 0
    assert torch.equal(a[0], b[0])
    rows = sample_rows(32768, 48, seed=8)
    check_backward(*cpu, *a, True, scale, heads=[(0, 7)], rows=rows, cols=rows)
