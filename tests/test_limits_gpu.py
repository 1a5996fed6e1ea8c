"""Edge sizes of the boundary on the GPU.

  * The largest problems it accepts: B*S*H*D just below 2^31 elements per
    tensor (4 GiB of bf16), so the last heads' elements lie more than 2^32
    bytes past the base pointer and every offset the kernels form must be
    64-bit.  S = 200 gives each head a full and a ragged tile.  Three heads
    (first, middle, last) are compared with the fp64 oracle, all rows; the
    packed form is checked the same way on a pack of about a million tokens.
  * Empty problems (a size of 0): the tensor API returns empty results and
    launches nothing; the C ABI itself rejects them (tested without a GPU).
"""
import math

import pytest
import torch

from exact_attention_36_gb300 import fa
from exact_attention_36_gb300.inputs import make_qkvdo_device, packed_lengths
from tests._parity import check_backward, check_forward

pytestmark = pytest.mark.gpu

LIMIT = 1 << 31  # elements per tensor the boundary accepts: strictly fewer
H = 16
S = 200


def _head(t, b, h):
    """One head of a [B, S, H, D] device tensor as a [1, S, 1, D] host tensor."""
    return t[b:b + 1, :, h:h + 1, :].cpu()


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_largest_fixed_length_problem(D, causal):
    B = (LIMIT - 1) // (S * H * D)
    assert B * S * H * D < LIMIT and (B + 1) * S * H * D >= LIMIT
    scale = 1.0 / math.sqrt(D)
    q, k, v, do = make_qkvdo_device(B, H, S, D, seed=D + int(causal))
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.backward(q, k, v, o, do, lse, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.device_error() == 0
    for b, h in ((0, 0), (B // 2, 7), (B - 1, H - 1)):
        hq, hk, hv, hdo = (_head(t, b, h) for t in (q, k, v, do))
        check_forward(hq, hk, hv, _head(o, b, h), lse[b:b + 1, h:h + 1].cpu(), causal, scale,
                      heads=None)
        check_backward(hq, hk, hv, hdo, _head(dq, b, h), _head(dk, b, h), _head(dv, b, h),
                       causal, scale, heads=None)
    del q, k, v, do, o, lse, dq, dk, dv
    torch.cuda.empty_cache()


@pytest.mark.parametrize("causal", [False, True])
def test_largest_packed_batch(causal):
    D = 128
    t_max = (LIMIT - 1) // (H * D)
    lengths = []
    for L in packed_lengths(8000, 400, seed=9):
        if sum(lengths) + L > t_max:
            break
        lengths.append(L)
    lengths.append(t_max - sum(lengths))  # fill up to the limit exactly
    T = sum(lengths)
    assert T == t_max and max(lengths) <= 400
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.as_tensor(lengths), 0).to(torch.int32)
    scale = 1.0 / math.sqrt(D)
    q, k, v, do = (t[0] for t in make_qkvdo_device(1, H, T, D, seed=11 + int(causal)))
    o, lse = fa.forward_varlen(q, k, v, cu.cuda(), max(lengths), causal=causal, scale=scale)
    dq, dk, dv = fa.backward_varlen(q, k, v, o, do, lse, cu.cuda(), max(lengths),
                                    causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.device_error() == 0
    n = len(lengths)
    for s in (0, n // 2, n - 2, n - 1):
        sl = slice(int(cu[s]), int(cu[s + 1]))
        hq, hk, hv, hdo = (t[None, sl].cpu() for t in (q, k, v, do))
        heads = [(0, 0), (0, H - 1)]
        check_forward(hq, hk, hv, o[None, sl].cpu(), lse[None, :, sl].cpu(), causal, scale,
                      heads=heads)
        check_backward(hq, hk, hv, hdo, dq[None, sl].cpu(), dk[None, sl].cpu(),
                       dv[None, sl].cpu(), causal, scale, heads=heads)
    del q, k, v, do, o, lse, dq, dk, dv
    torch.cuda.empty_cache()


@pytest.mark.parametrize("shape", [(0, 128, 2, 64), (2, 0, 2, 128), (2, 128, 0, 256)])
def test_empty_problems(shape):
    q = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    B, S, Hh, D = shape
    o, lse = fa.forward(q, q, q, causal=True)
    assert o.shape == shape and lse.shape == (B, Hh, S)
    dq, dk, dv = fa.backward(q, q, q, o, q, lse, causal=True)
    assert dq.shape == dk.shape == dv.shape == shape
    # packed form: no tokens at all (every sequence empty)
    qp = torch.empty((0, 2, D), dtype=torch.bfloat16, device="cuda")
    cu = torch.zeros(3, dtype=torch.int32, device="cuda")
    o, lse = fa.forward_varlen(qp, qp, qp, cu, 0)
    assert o.shape == (0, 2, D) and lse.shape == (2, 0)
    dq, dk, dv = fa.backward_varlen(qp, qp, qp, o, qp, lse, cu, 0)
    assert dq.shape == (0, 2, D)
    assert fa.device_error() == 0
    # an unsupported head dim is still an error
    with pytest.raises(fa.FAError):
        fa.forward(torch.empty((0, 4, 1, 96), dtype=torch.bfloat16, device="cuda"),
                   *(torch.empty((0, 4, 1, 96), dtype=torch.bfloat16, device="cuda"),) * 2)
