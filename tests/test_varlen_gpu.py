"""Packed variable-length batches (fa_fwd_varlen / fa_bwd_varlen): every
sequence of the pack is checked against the fp64 oracle run on that sequence
alone, so attention must stay inside each sequence; ragged lengths put
sequence boundaries inside tiles."""
import math

import pytest
import torch

from exact_attention_36_gb300 import fa
from exact_attention_36_gb300.inputs import make_packed, packed_lengths
from tests._parity import check_forward

pytestmark = pytest.mark.gpu


def _fwd(lengths, H, D, causal, seed=0, stress=False):
    q, k, v, do, cu = make_packed(lengths, H, D, seed=seed, stress=stress, with_dout=False)
    scale = 1.0 / math.sqrt(D)
    qd, kd, vd, cud = q.cuda(), k.cuda(), v.cuda(), cu.cuda()
    o, lse = fa.forward_varlen(qd, kd, vd, cud, max(lengths), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.device_error() == 0
    return q, k, v, cu, o.cpu(), lse.cpu(), scale


def _check_fwd_each(q, k, v, cu, o, lse, causal, scale, peaked=False):
    for b in range(cu.numel() - 1):
        a0, a1 = int(cu[b]), int(cu[b + 1])
        if a1 == a0:
            continue
        sl = slice(a0, a1)
        check_forward(q[None, sl], k[None, sl], v[None, sl], o[None, sl], lse[None, :, sl],
                      causal, scale, heads=None, peaked=peaked)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_ragged_mix(D, causal):
    lengths = [1, 127, 128, 129, 300, 2, 640, 257]
    q, k, v, cu, o, lse, scale = _fwd(lengths, 3, D, causal, seed=1)
    _check_fwd_each(q, k, v, cu, o, lse, causal, scale)


@pytest.mark.parametrize("causal", [False, True])
def test_forward_random_lengths(causal):
    lengths = packed_lengths(12, 1000, seed=2)
    q, k, v, cu, o, lse, scale = _fwd(lengths, 2, 128, causal, seed=2)
    _check_fwd_each(q, k, v, cu, o, lse, causal, scale)


def test_forward_matches_fixed_length_kernel():
    # equal lengths: the packed call must give the fixed-length call's bits
    B, H, S, D = 3, 4, 700, 128
    q, k, v, _, cu = make_packed([S] * B, H, D, seed=5, with_dout=False)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = fa.forward_varlen(qd, kd, vd, cu.cuda(), S, causal=True)
    o2, lse2 = fa.forward(qd.view(B, S, H, D), kd.view(B, S, H, D), vd.view(B, S, H, D),
                          causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o.view(B, S, H, D), o2)
    assert torch.equal(lse.view(H, B, S).permute(1, 0, 2), lse2)


def test_forward_empty_sequences_and_stress():
    lengths = [0, 513, 0, 64, 1025, 0]
    q, k, v, cu, o, lse, scale = _fwd(lengths, 2, 128, True, seed=3, stress=True)
    _check_fwd_each(q, k, v, cu, o, lse, True, scale, peaked=True)


def test_bad_offsets_are_reported_and_skipped():
    # a sequence longer than max_seqlen: its rows are left alone, the others
    # computed, and the device error word says why
    H, D = 2, 64
    q, k, v, _, cu = make_packed([200, 100], H, D, seed=4, with_dout=False)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.full_like(qd, 7.0)
    lse = torch.full((H, 300), 7.0, device="cuda")
    fa.fwd_varlen(qd, kd, vd, o, lse, cu.cuda(), 100, False, 0.125)
    torch.cuda.synchronize()
    assert fa.device_error() == 0x300
    assert (o[:200] == 7.0).all() and (lse[:, :200] == 7.0).all()
    _check_fwd_each(q[200:], k[200:], v[200:], torch.tensor([0, 100], dtype=torch.int32),
                    o[200:].cpu(), lse[:, 200:].cpu(), False, 0.125)
