"""fa_bwd_noalloc: the backward entry point for callers that cannot allocate
device memory (it takes its scratch from a fixed array inside the library).

Called through the C ABI and compared with fa_bwd, which uses caller-provided
scratch, on two calls in a row with different inputs (the second call must
not see anything left in the shared scratch by the first).  Kept in a file
that pytest collects last."""
import ctypes
import math

import numpy as np
import pytest
import torch

from exact_attention_36_gb300 import fa
from exact_attention_36_gb300.inputs import make_qkvdo
from tests._parity import GRAD_REL_L2, rel_l2

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    L = fa.lib()
    fn = L.fa_bwd_noalloc
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [vp] * 9 + [i, i, i, i, i, f, vp]
    fn.restype = i
    return fn


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_noalloc_matches_fa_bwd_on_two_calls_in_a_row(causal, D):
    # every head dim: D = 256 reaches the array through its own main kernel
    # (dQ^T reduced over 64-row blocks with its own accumulator map)
    fn = _noalloc_fn()
    B, H, S = (2, 4, 1000) if D != 256 else (1, 4, 1000)
    scale = 1.0 / math.sqrt(D)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for seed in (21, 22):
        q, k, v, do = (t.cuda() for t in make_qkvdo(B, H, S, D, seed=seed))
        o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
        ref = fa.backward(q, k, v, o, do, lse, causal=causal, scale=scale)
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        st = fn(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq), _p(dk), _p(dv),
                B, H, S, D, int(causal), scale, stream)
        assert st == fa.FA_OK, lib_status(st)
        torch.cuda.synchronize()
        assert fa.device_error() == 0
        for got, want in zip((dq, dk, dv), ref):
            g = got.float().cpu().numpy().ravel().astype(np.float64)
            w = want.float().cpu().numpy().ravel().astype(np.float64)
            assert np.isfinite(g).all()
            assert rel_l2(g, w) <= GRAD_REL_L2
        # dK and dV do not depend on the scratch's summation order
        assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])


def test_noalloc_rejects_problems_larger_than_its_scratch():
    fn = _noalloc_fn()
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    p = _p(x)
    # B*H*S*D*4 bytes of accumulator > 72 MiB
    st = fn(p, p, p, p, p, p, p, p, p, 1, 16, 16384, 128, 0, 0.1,
            ctypes.c_void_p(0))
    assert st == fa.FA_ERR_INVALID_ARG


def lib_status(st):
    return fa.lib().fa_status_string(st).decode()
