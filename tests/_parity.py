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

import numpy as np
import torch

import oracle

O_ATOL = 1e-2
LSE_ATOL = 1e-3
GRAD_REL_L2 = 2e-2


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, 2.0 ** (e - 8), 0.0)


def check_forward(q, k, v, o, lse, causal, scale, heads, rows=None, peaked=False):
    """Compare GPU o [B,S,H,D] / lse [B,H,S] with the oracle on the listed
    heads (and rows).  Returns (max O error, max LSE error).

    peaked=True (the stress inputs: scores ~30x the N(0,1) scale, nearly
    one-hot rows): P enters the PV product rounded to bf16 (relative 2^-9,
    FlashAttention-4 pages: bf16 quantisation dominates), which alone can move
    O by up to 2^-9 max|V|; with the output's own half-ulp that can exceed the
    plain gate.  The bound asserted is then 1e-2 + ulp/2 + 2^-8 max|V| (the
    P-rounding bound with a factor 2 for the fp32 products around it), and at
    most 1e-5 of the elements may exceed the plain gate."""
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
        if peaked:
            vmax = float(np.abs(_f64_head(v, b, h)).max())
            over = int((err > tol).sum())
            assert over <= max(1, int(1e-5 * err.size)), (
                f"{over} of {err.size} O elements above the plain gate in head {(b, h)}")
            tol = tol + 2.0 ** -8 * vmax
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


def check_backward(q, k, v, dout, dq, dk, dv, causal, scale, heads, rows=None, cols=None):
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
        e = rel_l2(np.concatenate(gs), np.concatenate(ws))
        assert e <= GRAD_REL_L2, f"{name} relative L2 error {e:.4g} > {GRAD_REL_L2}"
        worst[name] = e
    return worst


def sample_rows(S: int, n: int, seed: int = 0):
    """Seeded query rows including the first, last and tile-boundary rows."""
    rng = np.random.default_rng(seed)
    fixed = {0, 1, S - 1, S - 2, min(127, S - 1), min(128, S - 1), min(255, S - 1),
             min(256, S - 1), S // 2}
    picks = set(int(x) for x in rng.integers(0, S, size=n)) | fixed
    return sorted(r for r in picks if 0 <= r < S)
