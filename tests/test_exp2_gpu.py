"""The exp2 approximations on the device (FlashAttention-4: Algorithm and
Kernel Pipelining Co-Design, Technische samenvatting, Methodologie §2: 2^x
emulated by a degree-3 polynomial on the FMA pipes; accuracy gate 2^-9
relative on [-127, 0]).

Two independent checks: an exhaustive sweep of every fp32 in the range on the
device against CUDA's double-precision exp2, and a seeded sample copied back
and compared with the oracle's 2^x (C library exp2, double)."""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_36_gb300 import fa

pytestmark = pytest.mark.gpu

GATE = 2.0 ** -9


def test_full_range_polynomial_exhaustive_minus127_to_0():
    err, x = fa.exp2_sweep(-127.0, 0.0, variant=1)
    assert err <= GATE, (err, x)


def test_kernel_polynomial_exhaustive_on_its_range():
    # the softmax kernel's variant: valid on [-125, 16] (16 = largest rescale
    # threshold, the most an exponent argument can exceed 0)
    err, x = fa.exp2_sweep(-125.0, 16.0, variant=0)
    assert err <= GATE, (err, x)
    assert err <= 1e-4  # the degree-3 fit itself is ~7.5e-5


def test_two_lane_polynomial_matches_scalar_kernel_polynomial():
    # the softmax evaluates the polynomial with f32x2 instructions; same
    # rounding per lane, so the two forms agree bit for bit
    g = torch.Generator().manual_seed(9)
    x = (-140.0 + 160.0 * torch.rand(1 << 20, generator=g)).cuda()
    assert torch.equal(fa.exp2_eval(x, 3), fa.exp2_eval(x, 0))
    err, xm = fa.exp2_sweep(-125.0, 16.0, variant=3)
    assert err <= GATE, (err, xm)


def test_kernel_polynomial_clamps_below_minus125():
    x = torch.tensor([-125.5, -126.0, -127.0, -150.0, -1e30, float("-inf")], device="cuda")
    y = fa.exp2_eval(x, variant=0).cpu().double()
    assert (y > 0).all() and (y <= 2.0 ** -124).all()


def test_degree5_polynomial_exhaustive_minus127_to_0():
    # the pages allow degree 3 or 5; degree 5 is the tighter one (fit ~1.6e-7)
    err, x = fa.exp2_sweep(-127.0, 0.0, variant=4)
    assert err <= GATE, (err, x)
    assert err <= 1e-6


def test_degree5_kernel_form_on_its_range():
    # the two-lane degree-5 form the softmax instances evaluate (clamp at -125)
    err, x = fa.exp2_sweep(-125.0, 16.0, variant=5)
    assert err <= GATE, (err, x)
    assert err <= 1e-6


def test_mufu_reference_range():
    err, x = fa.exp2_sweep(-126.0, 16.0, variant=2)
    assert err <= 2.0 ** -20, (err, x)


@pytest.mark.parametrize("variant,lo,hi", [(1, -127.0, 0.0), (0, -125.0, 16.0), (2, -126.0, 16.0),
                                            (4, -127.0, 0.0), (5, -125.0, 16.0)])
def test_sampled_against_oracle_exp2(variant, lo, hi):
    g = torch.Generator().manual_seed(variant)
    x = lo + (hi - lo) * torch.rand(1 << 20, generator=g, dtype=torch.float64)
    x = x.float()
    y = fa.exp2_eval(x.cuda(), variant).cpu().double().numpy()
    ref = oracle.exp2(x.double().numpy())
    rel = np.abs(y - ref) / np.maximum(ref, 2.0 ** -126)
    assert rel.max() <= GATE
