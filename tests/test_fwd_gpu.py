"""Forward parity: the sm_103a kernel (through the C ABI) against the fp64
oracle on seeded inputs, from tiny and ragged shapes up to the long-context
workload, causal and not, plus the numerics knobs (rescale threshold, MUFU /
polynomial exp2 split) that must not change the result beyond rounding."""
import math

import pytest
import torch

from exact_attention_36_gb300 import fa
from exact_attention_36_gb300.inputs import make_qkvdo
from tests._parity import check_forward, sample_rows

pytestmark = pytest.mark.gpu


def _run(B, H, S, D, causal, seed=0, stress=False, **kw):
    q, k, v, _ = make_qkvdo(B, H, S, D, seed=seed, stress=stress, with_dout=False)
    scale = 1.0 / math.sqrt(D)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = fa.forward(qd, kd, vd, causal=causal, scale=scale, **kw)
    torch.cuda.synchronize()
    assert fa.device_error() == 0
    return q, k, v, o, lse, scale


@pytest.mark.parametrize("causal", [False, True])
def test_small_config_all_heads(causal):
    # 1 x 2 x 256 x 64: the small workload the oracle finishes in seconds
    q, k, v, o, lse, scale = _run(1, 2, 256, 64, causal)
    check_forward(q, k, v, o, lse, causal, scale, heads=None)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("S", [1, 2, 127, 128, 129, 255, 256, 257, 300, 511, 640])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths(S, D, causal):
    q, k, v, o, lse, scale = _run(2, 3, S, D, causal, seed=S)
    check_forward(q, k, v, o, lse, causal, scale, heads=None)


def test_batch_head_layout_many_units():
    # more work units than SMs: every CTA runs several units, both serpentine
    # directions, and rows from distinct (b, h) pairs must not mix
    q, k, v, o, lse, scale = _run(3, 40, 768, 64, True, seed=7)
    check_forward(q, k, v, o, lse, True, scale, heads=[(0, 0), (1, 17), (2, 39), (2, 20)])


def test_noncausal_b4_h16_s2048_d128_all_heads():
    q, k, v, o, lse, scale = _run(4, 16, 2048, 128, False)
    check_forward(q, k, v, o, lse, False, scale, heads=None)


def test_causal_b2_h16_s8192_d128():
    q, k, v, o, lse, scale = _run(2, 16, 8192, 128, True)
    check_forward(q, k, v, o, lse, True, scale, heads=[(0, 0), (1, 15), (1, 6)])


@pytest.mark.parametrize("causal", [False, True])
def test_long_context_b1_h16_s32768_d128_sampled_rows(causal):
    q, k, v, o, lse, scale = _run(1, 16, 32768, 128, causal)
    rows = sample_rows(32768, 96, seed=1)
    check_forward(q, k, v, o, lse, causal, scale, heads=[(0, 0), (0, 15)], rows=rows)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("S,B", [(1024, 16), (4096, 4), (16384, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_stress_sweep(S, B, D, causal):
    # Q ~ N(0, 4^2), 1 % of keys x8: the running maximum jumps, so the
    # conditional rescale fires
    q, k, v, o, lse, scale = _run(B, 16, S, D, causal, stress=True)
    rows = None if S <= 4096 else sample_rows(S, 128, seed=2)
    check_forward(q, k, v, o, lse, causal, scale, heads=[(0, 0), (B - 1, 15)], rows=rows,
                  peaked=True, case=f"B{B}_H16_S{S}_D{D}_{'causal' if causal else 'noncausal'}")


@pytest.mark.parametrize("tau", [0.0, 8.0, 16.0])
@pytest.mark.parametrize("groups", [0, 1, 2, 8])
def test_numerics_knobs_do_not_change_result(tau, groups):
    # rescale threshold 0 = rescale whenever the maximum grows; exp2 from MUFU
    # only, mixed, or polynomial only
    q, k, v, o, lse, scale = _run(2, 4, 1024, 128, True, stress=True,
                                  rescale_threshold=tau, poly_exp2_groups=groups)
    check_forward(q, k, v, o, lse, True, scale, heads=[(0, 0), (1, 3)], peaked=True)
    _, _, _, o_ref, lse_ref, _ = _run(2, 4, 1024, 128, True, stress=True,
                                      rescale_threshold=0.0, poly_exp2_groups=0)
    assert (o.float() - o_ref.float()).abs().max().item() <= 2e-2
    assert (lse - lse_ref).abs().max().item() <= 1e-3


@pytest.mark.parametrize("degree", [3, 5])
@pytest.mark.parametrize("groups", [1, 2, 8])
def test_polynomial_columns_are_taken(groups, degree):
    # the split really moves exponentials to the polynomial: its values differ
    # from MUFU's in the last bits, so the row sums (fp32, before the bf16
    # rounding of P) and hence some LSE values differ from the MUFU-only run
    q, k, v, _ = make_qkvdo(1, 4, 512, 128, seed=13, with_dout=False)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    _, lse0 = fa.forward(qd, kd, vd, poly_exp2_groups=0)
    _, lse1 = fa.forward(qd, kd, vd, poly_exp2_groups=groups, poly_exp2_degree=degree)
    torch.cuda.synchronize()
    assert not torch.equal(lse0, lse1)
    assert (lse0 - lse1).abs().max().item() <= 1e-4


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("groups", [1, 2, 8])
def test_degree5_polynomial_instances(D, groups):
    # the pages allow a polynomial of degree 3 or 5: the degree-5 instances
    # against the oracle, and against the MUFU-only result of the same inputs
    q, k, v, o, lse, scale = _run(2, 4, 1024, D, True, stress=True, poly_exp2_groups=groups,
                                  poly_exp2_degree=5)
    check_forward(q, k, v, o, lse, True, scale, heads=[(0, 0), (1, 3)], peaked=True)
    _, _, _, o_ref, lse_ref, _ = _run(2, 4, 1024, D, True, stress=True, poly_exp2_groups=0)
    assert (o.float() - o_ref.float()).abs().max().item() <= 2e-2
    assert (lse - lse_ref).abs().max().item() <= 1e-3
    # with every exponential on the degree-5 polynomial (relative error ~2e-7
    # against MUFU's ~2^-22) the non-peaked inputs match the oracle as closely
    # as the MUFU path does
    q, k, v, o, lse, scale = _run(1, 3, 700, D, False, seed=5, poly_exp2_groups=groups,
                                  poly_exp2_degree=5)
    check_forward(q, k, v, o, lse, False, scale, heads=None)


@pytest.mark.parametrize("D", [64, 256])
@pytest.mark.parametrize("groups,degree", [(0, 3), (2, 3), (2, 5)])
def test_numerics_knobs_other_head_dims(D, groups, degree):
    q, k, v, o, lse, scale = _run(1, 3, 700, D, True, stress=True, rescale_threshold=0.0,
                                  poly_exp2_groups=groups, poly_exp2_degree=degree)
    check_forward(q, k, v, o, lse, True, scale, heads=None, peaked=True)


def test_deterministic_repeat():
    a = _run(1, 4, 1000, 128, True, seed=3)
    b = _run(1, 4, 1000, 128, True, seed=3)
    assert torch.equal(a[3], b[3]) and torch.equal(a[4], b[4])


def test_rejects_bad_arguments():
    q = torch.zeros(1, 128, 1, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FAError, match="INVALID_ARG"):
        fa.forward(q, q, q, scale=-1.0)
    with pytest.raises(fa.FAError, match="UNSUPPORTED"):
        x = torch.zeros(1, 128, 1, 96, dtype=torch.bfloat16, device="cuda")
        fa.forward(x, x, x)
    with pytest.raises(fa.FAError, match="INVALID_ARG"):
        fa.forward(q, q, q, poly_exp2_groups=1, poly_exp2_degree=4)
