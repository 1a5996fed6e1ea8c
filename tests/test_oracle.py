"""Pins for the fp64 CPU oracle (no GPU).

The CUDA kernels are checked against the oracle, so it is itself checked against
things that do not come from it: hand-derived closed forms (tests/golden),
invariants of softmax attention and of its gradient, a library routine
(torch's CPU float64 scaled_dot_product_attention and autograd), and central
finite differences.  Each check is chosen to catch a plausible slip in the
oracle: a dropped scale, a wrong sign, an off-by-one causal mask, a
transposed operand, a missing Delta term.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from exact_attention_36_gb300.inputs import make_qkvdo

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def _rand_head(S, D, seed, qscale=1.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((S, D)) * qscale
    k = rng.standard_normal((S, D))
    v = rng.standard_normal((S, D))
    do = rng.standard_normal((S, D))
    return q, k, v, do


# ---------------------------------------------------------------- golden


def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_hand_worked_examples(case):
    q, k, v, do = (np.array(case[n], dtype=np.float64) for n in ("q", "k", "v", "dout"))
    o, lse = oracle.forward_head(q, k, v, case["causal"], case["scale"])
    np.testing.assert_allclose(o, case["o"], rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(lse, case["lse"], rtol=1e-14, atol=1e-14)
    g = oracle.backward_head(q, k, v, do, case["causal"], case["scale"])
    np.testing.assert_allclose(g["lse"], case["lse"], rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(g["delta"], case["delta"], rtol=1e-14, atol=1e-14)
    for name in ("dq", "dk", "dv"):
        np.testing.assert_allclose(g[name], case[name], rtol=1e-13, atol=1e-14, err_msg=name)


# ---------------------------------------------------------------- forward closed forms


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_mean_of_visible_values(causal):
    S, D = 37, 8
    q, k, v, _ = _rand_head(S, D, 1)
    k[:] = k[0]  # every key identical -> every visible score equal
    o, lse = oracle.forward_head(q, k, v, causal, 0.3)
    for i in range(S):
        n = i + 1 if causal else S
        np.testing.assert_allclose(o[i], v[:n].mean(axis=0), rtol=1e-12, atol=1e-12)
        s = 0.3 * float(q[i] @ k[0])
        np.testing.assert_allclose(lse[i], s + math.log(n), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_gives_log_count(causal):
    S, D = 29, 4
    _, k, v, _ = _rand_head(S, D, 2)
    q = np.zeros((S, D))
    o, lse = oracle.forward_head(q, k, v, causal, 0.5)
    counts = np.arange(1, S + 1) if causal else np.full(S, S)
    np.testing.assert_allclose(lse, np.log(counts), rtol=1e-13, atol=1e-13)
    prefix_mean = np.cumsum(v, axis=0) / np.arange(1, S + 1)[:, None]
    want = prefix_mean if causal else np.broadcast_to(v.mean(axis=0), (S, D))
    np.testing.assert_allclose(o, want, rtol=1e-12, atol=1e-12)


def test_causal_row0_is_v0():
    S, D = 16, 8
    q, k, v, _ = _rand_head(S, D, 3, qscale=3.0)
    o, lse = oracle.forward_head(q, k, v, True, 0.25)
    np.testing.assert_array_equal(o[0], v[0])
    np.testing.assert_allclose(lse[0], 0.25 * float(q[0] @ k[0]), rtol=1e-14)


def test_rows_of_p_sum_to_one_and_mask_is_zero():
    # V = identity (S == D) makes O equal to the attention matrix P itself.
    S = D = 24
    q, k, _, _ = _rand_head(S, D, 4, qscale=2.0)
    v = np.eye(S)
    for causal in (False, True):
        p, lse = oracle.forward_head(q, k, v, causal, 0.7)
        np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=1e-13)
        assert (p >= 0).all()
        if causal:
            assert np.count_nonzero(np.triu(p, 1)) == 0
            assert (p[np.tril_indices(S)] > 0).all()
        # P_ij = exp(s_ij - LSE_i) for the visible entries
        s = 0.7 * q @ k.T
        want = np.exp(s - lse[:, None])
        if causal:
            want = np.tril(want)
        np.testing.assert_allclose(p, want, rtol=1e-12, atol=1e-300)


def test_key_permutation_invariance():
    S, D = 50, 16
    q, k, v, _ = _rand_head(S, D, 5)
    perm = np.random.default_rng(0).permutation(S)
    o1, l1 = oracle.forward_head(q, k, v, False, 0.25)
    o2, l2 = oracle.forward_head(q, k[perm], v[perm], False, 0.25)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=1e-13)


def test_one_dominant_key_selects_its_value():
    S, D = 32, 8
    q, k, v, _ = _rand_head(S, D, 6)
    q[:] = 1.0
    k[:] = 0.0
    k[7] = 60.0  # score 0.5*8*60 = 240 above the rest
    o, lse = oracle.forward_head(q, k, v, False, 0.5)
    np.testing.assert_allclose(o, np.broadcast_to(v[7], (S, D)), rtol=0, atol=1e-90)
    np.testing.assert_allclose(lse, 240.0, rtol=1e-15)


def test_row_subset_matches_full():
    S, D = 40, 8
    q, k, v, _ = _rand_head(S, D, 7)
    o, lse = oracle.forward_head(q, k, v, True, 0.3)
    rows = [0, 5, 39, 17]
    o2, l2 = oracle.forward_head(q, k, v, True, 0.3, rows=rows)
    np.testing.assert_array_equal(o2, o[rows])
    np.testing.assert_array_equal(l2, lse[rows])


# ---------------------------------------------------------------- library routine


@pytest.mark.parametrize("S,D,causal", [(64, 16, False), (64, 16, True), (33, 8, True),
                                        (129, 32, False)])
def test_matches_torch_float64_sdpa_and_autograd(S, D, causal):
    q, k, v, do = _rand_head(S, D, 10 + S + D, qscale=2.0)
    scale = 1.0 / math.sqrt(D)
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    with torch.nn.attention.sdpa_kernel(torch.nn.attention.SDPBackend.MATH):
        to = torch.nn.functional.scaled_dot_product_attention(
            tq[None, None], tk[None, None], tv[None, None], is_causal=causal, scale=scale)[0, 0]
    to.backward(torch.tensor(do))
    s = scale * (tq.detach() @ tk.detach().T)
    if causal:
        s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
    tlse = torch.logsumexp(s, dim=-1)

    o, lse = oracle.forward_head(q, k, v, causal, scale)
    np.testing.assert_allclose(o, to.detach().numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, tlse.numpy(), rtol=1e-12, atol=1e-12)
    g = oracle.backward_head(q, k, v, do, causal, scale)
    np.testing.assert_allclose(g["dq"], tq.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(g["dk"], tk.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(g["dv"], tv.grad.numpy(), rtol=1e-10, atol=1e-11)


# ---------------------------------------------------------------- backward pins


def _loss(q, k, v, do, causal, scale):
    o, _ = oracle.forward_head(q, k, v, causal, scale)
    return float((o * do).sum())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S,D", [(5, 3), (8, 4), (1, 2)])
def test_backward_matches_central_finite_differences(S, D, causal):
    q, k, v, do = _rand_head(S, D, 20 + S * D + causal)
    scale = 0.8
    g = oracle.backward_head(q, k, v, do, causal, scale)
    h = 1e-6
    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            old = x[idx]
            x[idx] = old + h
            lp = _loss(q, k, v, do, causal, scale)
            x[idx] = old - h
            lm = _loss(q, k, v, do, causal, scale)
            x[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(g[name], fd, rtol=0, atol=1e-6, err_msg=name)


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_invariants(causal):
    S, D = 45, 16
    q, k, v, do = _rand_head(S, D, 30, qscale=2.0)
    g = oracle.backward_head(q, k, v, do, causal, 0.25, want_o=True)
    # shifting every key by the same vector shifts each score row by a constant
    np.testing.assert_allclose(g["dk"].sum(axis=0), 0.0, atol=1e-12)
    # every P row sums to one
    np.testing.assert_allclose(g["dv"].sum(axis=0), do.sum(axis=0), rtol=1e-12, atol=1e-12)
    # Delta_i = sum_j P_ij dP_ij equals dO_i . O_i
    np.testing.assert_allclose(g["delta"], (do * g["o"]).sum(axis=1), rtol=1e-12, atol=1e-12)
    o, lse = oracle.forward_head(q, k, v, causal, 0.25)
    np.testing.assert_allclose(g["o"], o, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(g["lse"], lse, rtol=1e-14)


def test_backward_row_and_column_subsets_match_full():
    S, D = 33, 8
    q, k, v, do = _rand_head(S, D, 40)
    full = oracle.backward_head(q, k, v, do, True, 0.4)
    rows, cols = [32, 0, 11], [3, 32, 0]
    sub = oracle.backward_head(q, k, v, do, True, 0.4, rows=rows, cols=cols)
    np.testing.assert_array_equal(sub["dq"], full["dq"][rows])
    np.testing.assert_array_equal(sub["dk"], full["dk"][cols])
    np.testing.assert_array_equal(sub["dv"], full["dv"][cols])


def test_multihead_wrapper_slices_bshd_layout():
    q, k, v, do = make_qkvdo(2, 3, 20, 8, seed=3)
    res = oracle.forward(q, k, v, True, 0.3, heads=[(1, 2), (0, 0)])
    q64 = q.double().numpy()
    o, lse = oracle.forward_head(q64[1, :, 2], k.double().numpy()[1, :, 2],
                                 v.double().numpy()[1, :, 2], True, 0.3)
    np.testing.assert_array_equal(res[(1, 2)][0], o)
    np.testing.assert_array_equal(res[(1, 2)][1], lse)


# ---------------------------------------------------------------- exp2 reference


def test_exp2_reference_exact_points():
    x = np.array([0.0, 1.0, -1.0, 10.0, -126.0, -127.0, -149.0, 0.5, -0.5, 3.25])
    y = oracle.exp2(x)
    want = [1.0, 2.0, 0.5, 1024.0, 2.0 ** -126, 2.0 ** -127, 2.0 ** -149,
            math.sqrt(2.0), 1.0 / math.sqrt(2.0), 8.0 * 2.0 ** 0.25]
    np.testing.assert_allclose(y, want, rtol=2e-16, atol=0)


# ---------------------------------------------------------------- inputs recipe


def test_input_recipe_is_seeded_and_stress_scales_one_percent_of_keys():
    a = make_qkvdo(1, 2, 300, 8, seed=5)
    b = make_qkvdo(1, 2, 300, 8, seed=5)
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16 and x.shape == (1, 300, 2, 8)
        assert torch.equal(x, y)
    qs, ks, vs, ds = make_qkvdo(1, 2, 300, 8, seed=5, stress=True)
    # 3 of 300 key rows per head are scaled by 8: they stand out in norm
    norms = ks.float().norm(dim=-1)  # [1, S, H]
    for h in range(2):
        top = norms[0, :, h].topk(3).values
        assert (top > 8).all()
    assert qs.float().abs().max() > 8  # Q ~ N(0, 4^2)


def test_row_stats_and_dq_rows_match_full_backward():
    S, D = 40, 8
    q, k, v, do = _rand_head(S, D, 50)
    full = oracle.backward_head(q, k, v, do, True, 0.4)
    rows = [39, 2, 17]
    lse, delta = oracle.row_stats_head(q, k, v, do, True, 0.4, rows)
    np.testing.assert_array_equal(lse, full["lse"][rows])
    np.testing.assert_array_equal(delta, full["delta"][rows])
    lf = np.zeros(S); df = np.zeros(S)
    lf[rows] = lse
    df[rows] = delta
    dq = oracle.dq_rows_head(q, k, v, do, lf, df, True, 0.4, rows)
    np.testing.assert_array_equal(dq, full["dq"][rows])
