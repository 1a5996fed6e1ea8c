"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
binding and compare with the fp64 CPU oracle on the same seeded inputs.

Tolerances (stated by the task for this method, not by the pages):
  forward  O:   |O_gpu - O_ref| <= 1e-2 + ulp_bf16(O_ref)/2   (max abs; the
                half-ulp term only matters where |O_ref| >= 2, where bf16
                rounding of the output alone can exceed 1e-2)
           LSE: |LSE_gpu - LSE_ref| <= 1e-3
  backward dQ, dK, dV: relative L2 error <= 2e-2 over the checked heads.
                The denominator has a floor of 1e-3 RMS: where the exact
                gradient vanishes (e.g. S = 1, where dS = 0 identically) a
                relative error is undefined and the check becomes absolute.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle

# When set, the checks append one JSON line per checked case to this file
# (the per-case errors behind the gates, for a written test report).
REPORT = os.environ.get("FA_PARITY_REPORT")


def _record(entry):
    if REPORT:
        with open(REPORT, "a") as f:
            f.write(json.dumps(entry) + "\n")

O_ATOL = 1e-2
LSE_ATOL = 1e-3
GRAD_REL_L2 = 2e-2


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, 2.0 ** (e - 8), 0.0)


def check_forward(q, k, v, o, lse, causal, scale, heads, rows=None, peaked=False, case=None):
    """Compare GPU o [B,S,H,D] / lse [B,H,S] with the oracle on the listed
    heads (and rows).  Returns (max O error, max LSE error).

    peaked=True (the stress inputs: scores ~30x the N(0,1) scale, nearly
    one-hot rows): P enters the PV product rounded to bf16 (relative 2^-9,
    FlashAttention-4 pages: bf16 quantisation dominates).  With p_j the fp32
    probabilities, l their sum and P_j = p_j (1 + e_j), |e_j| <= 2^-9, the
    product moves O by |sum_j p_j e_j V_j| / l <= 2^-9 max|V| (the fp32 sums
    add relative errors of order 2^-24, far below that).  With the output's
    own half-ulp that can exceed the plain gate, so the bound asserted is
    1e-2 + ulp/2 + 2^-9 max|V|, and at most 1e-5 of the elements may exceed
    the plain gate.

    case: a label; with FA_PARITY_REPORT set, the errors are recorded."""
    ref = oracle.forward(q, k, v, causal, scale, heads=heads, rows=rows)
    o_cpu = o.float().cpu()
    lse_cpu = lse.cpu()
    worst_o = worst_l = 0.0
    for (b, h), (o_ref, lse_ref) in ref.items():
        if rows is None:
            og = o_cpu[b, :, h].double().numpy()
            lg = lse_cpu[b, h].double().numpy()
        else:
            idx = torch.as_tensor(rows, dtype=torch.long)
            og = o_cpu[b, idx, h].double().numpy()
            lg = lse_cpu[b, h, idx].double().numpy()
        err = np.abs(og - o_ref)
        tol = O_ATOL + half_ulp_bf16(o_ref)
        over = int((err > tol).sum())
        vmax = float(np.abs(_f64_head(v, b, h)).max())
        if case is not None:
            _record({"dir": "fwd", "case": case, "head": [b, h], "o_max_err": float(err.max()),
                     "o_ref_max_abs": float(np.abs(o_ref).max()), "v_max_abs": vmax,
                     "over_plain_gate": over, "elements": int(err.size),
                     "lse_max_err": float(np.abs(lg - lse_ref).max()), "peaked": peaked})
        if peaked:
            assert over <= max(1, int(1e-5 * err.size)), (
                f"{over} of {err.size} O elements above the plain gate in head {(b, h)}")
            tol = tol + 2.0 ** -9 * vmax
        bad = err > tol
        assert not bad.any(), (
            f"O mismatch head {(b, h)}: max err {err.max():.4g}, "
            f"{int(bad.sum())} elements over tolerance; first at {np.argwhere(bad)[0]}")
        lerr = np.abs(lg - lse_ref)
        assert lerr.max() <= LSE_ATOL, f"LSE mismatch head {(b, h)}: {lerr.max():.4g}"
        worst_o = max(worst_o, float(err.max()))
        worst_l = max(worst_l, float(lerr.max()))
    return worst_o, worst_l


def _f64_head(x, b, h):
    return x[b, :, h].double().numpy()


def rel_l2(got: np.ndarray, want: np.ndarray) -> float:
    floor = 1e-3 * np.sqrt(want.size)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), floor))


def check_backward(q, k, v, dout, dq, dk, dv, causal, scale, heads, rows=None, cols=None,
                   case=None):
    """Compare GPU gradients with the oracle's (exact fp64) gradients on the
    listed heads (rows of dQ / key columns of dK, dV).  Returns the worst
    relative L2 error per tensor."""
    ref = oracle.backward(q, k, v, dout, causal, scale, heads=heads, rows=rows, cols=cols)
    got = {"dq": dq.float().cpu(), "dk": dk.float().cpu(), "dv": dv.float().cpu()}
    sel = {"dq": rows, "dk": cols, "dv": cols}
    acc = {n: ([], []) for n in got}
    for (b, h), g in ref.items():
        for name in got:
            idx = sel[name]
            t = got[name][b, :, h] if idx is None else got[name][b, torch.as_tensor(idx), h]
            acc[name][0].append(t.double().numpy())
            acc[name][1].append(g[name])
    worst = {}
    for name, (gs, ws) in acc.items():
        worst[name] = rel_l2(np.concatenate(gs), np.concatenate(ws))
    if case is not None:
        _record({"dir": "bwd", "case": case, **{f"{n}_rel_l2": e for n, e in worst.items()}})
    for name, e in worst.items():
        assert e <= GRAD_REL_L2, f"{name} relative L2 error {e:.4g} > {GRAD_REL_L2}"
    return worst


def sample_rows(S: int, n: int, seed: int = 0):
    """Seeded query rows including the first, last and tile-boundary rows."""
    rng = np.random.default_rng(seed)
    fixed = {0, 1, S - 1, S - 2, min(127, S - 1), min(128, S - 1), min(255, S - 1),
             min(256, S - 1), S // 2}
    picks = set(int(x) for x in rng.integers(0, S, size=n)) | fixed
    return sorted(r for r in picks if 0 <= r < S)
