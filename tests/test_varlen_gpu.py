"""Packed variable-length batches (fa_fwd_varlen / fa_bwd_varlen): every
sequence of the pack is checked against the fp64 oracle run on that sequence
alone, so attention must stay inside each sequence; ragged lengths put
sequence boundaries inside tiles."""
import math

import pytest
import torch

from exact_attention_36_gb300 import fa
from exact_attention_36_gb300.inputs import make_packed, packed_lengths
from tests._parity import check_backward, check_forward

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


def _bwd(lengths, H, D, causal, seed=0, stress=False):
    q, k, v, do, cu = make_packed(lengths, H, D, seed=seed, stress=stress)
    scale = 1.0 / math.sqrt(D)
    qd, kd, vd, dod, cud = q.cuda(), k.cuda(), v.cuda(), do.cuda(), cu.cuda()
    mx = max(lengths)
    o, lse = fa.forward_varlen(qd, kd, vd, cud, mx, causal=causal, scale=scale)
    dq, dk, dv = fa.backward_varlen(qd, kd, vd, o, dod, lse, cud, mx, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.device_error() == 0
    return q, k, v, do, cu, dq.cpu(), dk.cpu(), dv.cpu(), scale


def _check_bwd_each(q, k, v, do, cu, dq, dk, dv, causal, scale):
    for b in range(cu.numel() - 1):
        a0, a1 = int(cu[b]), int(cu[b + 1])
        if a1 == a0:
            continue
        sl = slice(a0, a1)
        check_backward(q[None, sl], k[None, sl], v[None, sl], do[None, sl], dq[None, sl],
                       dk[None, sl], dv[None, sl], causal, scale, heads=None)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_ragged_mix(D, causal):
    lengths = [1, 127, 128, 129, 300, 2, 640, 257]
    args = _bwd(lengths, 3, D, causal, seed=1)
    _check_bwd_each(*args[:8], causal, args[8])


@pytest.mark.parametrize("causal", [False, True])
def test_backward_random_lengths_and_stress(causal):
    lengths = packed_lengths(10, 900, seed=6)
    args = _bwd(lengths, 2, 128, causal, seed=6, stress=True)
    _check_bwd_each(*args[:8], causal, args[8])


def test_backward_matches_fixed_length_kernel():
    B, H, S, D = 3, 4, 700, 128
    q, k, v, do, cu = make_packed([S] * B, H, D, seed=5)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.forward_varlen(qd, kd, vd, cu.cuda(), S, causal=True)
    dq, dk, dv = fa.backward_varlen(qd, kd, vd, o, dod, lse, cu.cuda(), S, causal=True)
    shp = (B, S, H, D)
    o2, lse2 = fa.forward(qd.view(shp), kd.view(shp), vd.view(shp), causal=True)
    dq2, dk2, dv2 = fa.backward(qd.view(shp), kd.view(shp), vd.view(shp), o2, dod.view(shp), lse2,
                                causal=True)
    torch.cuda.synchronize()
    # dK, dV are reduced in a fixed order in both; dQ's fp32 sums run in
    # atomic order
    assert torch.equal(dk.view(shp), dk2) and torch.equal(dv.view(shp), dv2)
    assert ((dq.view(shp).float() - dq2.float()).norm() / dq2.float().norm()).item() <= 1e-3


def test_backward_d256_random_lengths_and_stress():
    lengths = packed_lengths(6, 700, seed=8)
    args = _bwd(lengths, 2, 256, True, seed=8, stress=True)
    _check_bwd_each(*args[:8], True, args[8])


def test_backward_d256_matches_fixed_length_kernel():
    B, H, S, D = 2, 2, 300, 256
    q, k, v, do, cu = make_packed([S] * B, H, D, seed=9)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.forward_varlen(qd, kd, vd, cu.cuda(), S, causal=False)
    dq, dk, dv = fa.backward_varlen(qd, kd, vd, o, dod, lse, cu.cuda(), S, causal=False)
    shp = (B, S, H, D)
    o2, lse2 = fa.forward(qd.view(shp), kd.view(shp), vd.view(shp), causal=False)
    dq2, dk2, dv2 = fa.backward(qd.view(shp), kd.view(shp), vd.view(shp), o2, dod.view(shp), lse2,
                                causal=False)
    torch.cuda.synchronize()
    assert torch.equal(dk.view(shp), dk2) and torch.equal(dv.view(shp), dv2)
    assert ((dq.view(shp).float() - dq2.float()).norm() / dq2.float().norm()).item() <= 1e-3


@pytest.mark.parametrize("D,causal,H", [(128, False, 24), (128, True, 24), (64, True, 2),
                                         (256, True, 2)])
def test_backward_deterministic_packed(D, causal, H):
    # fixed-order dQ over a packed batch: bit-for-bit repeatable, exact per
    # sequence, and the atomic order's result up to the order of additions
    # (H = 24 gives several rounds of the persistent grid)
    lengths = [300, 1, 777, 128, 0, 513] if D != 256 else [300, 1, 200, 129]
    q, k, v, do, cu = make_packed(lengths, H, D, seed=11)
    scale = 1.0 / math.sqrt(D)
    qd, kd, vd, dod, cud = q.cuda(), k.cuda(), v.cuda(), do.cuda(), cu.cuda()
    mx = max(lengths)
    o, lse = fa.forward_varlen(qd, kd, vd, cud, mx, causal=causal, scale=scale)
    a = fa.backward_varlen(qd, kd, vd, o, dod, lse, cud, mx, causal=causal, scale=scale,
                           deterministic=True)
    b = fa.backward_varlen(qd, kd, vd, o, dod, lse, cud, mx, causal=causal, scale=scale,
                           deterministic=True)
    c = fa.backward_varlen(qd, kd, vd, o, dod, lse, cud, mx, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.device_error() == 0
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    for x, y in zip(a, c):
        x, y = x.float(), y.float()
        assert ((x - y).norm() / y.norm()).item() <= 2e-3
    _check_bwd_each(q, k, v, do, cu, a[0].cpu(), a[1].cpu(), a[2].cpu(), causal, scale)
