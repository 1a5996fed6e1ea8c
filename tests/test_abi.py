"""C ABI checks that need no GPU: the library builds and loads, exports every
entry point include/fa.h declares, and rejects bad arguments before touching
a device; the exp2 polynomial's coefficients meet the accuracy bound."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from exact_attention_36_gb300 import build as fa_build
from exact_attention_36_gb300 import fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")
COEFFS = os.path.join(ROOT, "exact_attention_36_gb300", "csrc", "exp2_poly_coeffs.h")


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return fa.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("fa_fwd", "fa_fwd_ex", "fa_bwd", "fa_bwd_ex", "fa_bwd_workspace_size",
                 "fa_fwd_varlen", "fa_bwd_varlen", "fa_bwd_deterministic", "fa_bwd_varlen_deterministic",
                 "fa_status_string",
                 "fa_last_cuda_error", "fa_device_error", "fa_exp2_eval", "fa_exp2_sweep"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in enumerate(["FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED",
                                 "FA_ERR_CUDA", "FA_ERR_TIMEOUT"]):
        assert lib.fa_status_string(code).decode() == name


def test_argument_errors_need_no_device(lib):
    null = ctypes.c_void_p(0)
    p = ctypes.c_void_p(0x10000)  # aligned, never dereferenced: the checks fail first
    odd = ctypes.c_void_p(0x10008)
    # null pointer
    assert lib.fa_fwd(null, p, p, p, p, 1, 1, 128, 64, 0, 0.125, null) == fa.FA_ERR_INVALID_ARG
    # misaligned pointer
    assert lib.fa_fwd(p, odd, p, p, p, 1, 1, 128, 64, 0, 0.125, null) == fa.FA_ERR_INVALID_ARG
    # sizes, scale
    for B, H, S, D, sc in ((0, 1, 128, 64, 0.1), (1, 0, 128, 64, 0.1), (1, 1, 0, 64, 0.1),
                           (1, 1, 128, 64, 0.0), (1, 1, 128, 64, float("nan")),
                           (1, 1, 128, 64, float("inf")), (1 << 14, 16, 1 << 14, 128, 0.1)):
        assert lib.fa_fwd(p, p, p, p, p, B, H, S, D, 0, sc, null) == fa.FA_ERR_INVALID_ARG
    # unsupported head dim
    assert lib.fa_fwd(p, p, p, p, p, 1, 1, 128, 96, 0, 0.1, null) == fa.FA_ERR_UNSUPPORTED
    # knobs out of range
    assert lib.fa_fwd_ex(p, p, p, p, p, 1, 1, 128, 64, 0, 0.1, 17.0, 0, -1, null) == \
        fa.FA_ERR_INVALID_ARG
    assert lib.fa_fwd_ex(p, p, p, p, p, 1, 1, 128, 64, 0, 0.1, 8.0, 3, -1, null) == \
        fa.FA_ERR_INVALID_ARG
    for deg in (0, 1, 2, 4, 6, 7):  # the polynomial's degree is 3 or 5
        assert lib.fa_fwd_ex(p, p, p, p, p, 1, 1, 128, 64, 0, 0.1, 8.0, 1, deg, null) == \
            fa.FA_ERR_INVALID_ARG
    ptrs = [p] * 11
    ptrs[6] = null
    assert lib.fa_bwd(*ptrs, 1, 1, 128, 64, 0, 0.1, null) == fa.FA_ERR_INVALID_ARG
    # backward main-kernel choice: CTA pairs exist for D = 128 only
    ok = [p] * 11
    lib.fa_bwd_ex.argtypes = [ctypes.c_void_p] * 11 + [ctypes.c_int] * 5 + \
        [ctypes.c_float, ctypes.c_int, ctypes.c_void_p]
    for mode in (-2, 2):
        assert lib.fa_bwd_ex(*ok, 1, 1, 128, 128, 0, 0.1, mode, null) == fa.FA_ERR_INVALID_ARG
    # CTA pairs exist for D = 128 and 256
    assert lib.fa_bwd_ex(*ok, 1, 1, 128, 64, 0, 0.1, 1, null) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_exp2_sweep(1.0, 0.0, 0, p, null) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_exp2_eval(p, p, -1, 0, null) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_exp2_eval(p, p, 16, 6, null) == fa.FA_ERR_INVALID_ARG


def test_workspace_size(lib):
    B, H, S, D = 2, 3, 1000, 128
    n = B * H * S
    want = (n * D * 4 + 255) // 256 * 256 + (n * 4 + 255) // 256 * 256
    assert lib.fa_bwd_workspace_size(B, H, S, D) == want
    assert lib.fa_bwd_workspace_size(0, H, S, D) == 0
    assert lib.fa_bwd_workspace_size(B, H, S, 96) == 0


def test_semaphore_and_varlen_scratch_sizes(lib):
    # fixed-order mode at D = 64/128: per 128-query block one counter per
    # drain warp and accumulator (4 x 2), one order key per 128-key tile, then
    # the second fp32 accumulator; each part padded to 256 bytes
    def pad(x):
        return (x + 255) // 256 * 256

    B, H, S, D = 2, 3, 1000, 128
    nT = (S + 127) // 128
    want = pad(B * H * 8 * nT * 4) + pad(B * H * nT * 4) + pad(B * H * S * D * 4)
    assert lib.fa_bwd_semaphore_bytes(B, H, S, D) == want
    assert lib.fa_bwd_semaphore_bytes(B, H, 0, D) == 0
    # D = 256: one counter per 64 query rows, half of the head dim and drain warp
    assert lib.fa_bwd_semaphore_bytes(B, H, S, 256) == pad(B * H * 8 * ((S + 63) // 64) * 4)
    # packed batches: counters and keys per sequence and the longest one's
    # tiles, the second accumulator over all tokens
    T, Bs, L = 1234, 5, 700
    nT = (L + 127) // 128
    want = pad(Bs * H * 8 * nT * 4) + pad(Bs * H * nT * 4) + pad(H * T * D * 4)
    assert lib.fa_bwd_varlen_semaphore_bytes(Bs, L, T, H, D) == want
    assert lib.fa_bwd_varlen_semaphore_bytes(Bs, L, T, H, 256) == \
        pad(Bs * H * 8 * ((L + 63) // 64) * 4)
    assert lib.fa_bwd_varlen_semaphore_bytes(Bs, T + 1, T, H, D) == 0
    # packed batches: the accumulator and Delta over all tokens, as fa_bwd's
    assert lib.fa_bwd_varlen_workspace_size(T, H, D) == lib.fa_bwd_workspace_size(1, H, T, D)


def _coeffs(deg):
    text = open(COEFFS).read()
    return [float(re.search(rf"FA_EXP2_P{deg}_C{i} ([-+0-9.e]+)f", text).group(1))
            for i in range(deg + 1)]


@pytest.mark.parametrize("deg", [3, 5])
def test_exp2_polynomial_coefficients_meet_the_bound(deg):
    # the reduced argument f = x - rint(x) lies in [-1/2, 1/2]; the relative
    # error of p(f) against 2^f (C library exp2 through the oracle) bounds
    # the kernel's relative error up to float32 rounding of the evaluation
    c = np.asarray(_coeffs(deg), dtype=np.float32).astype(np.float64)
    f = np.linspace(-0.5, 0.5, 400001)
    p = np.zeros_like(f)
    for ci in c[::-1]:
        p = p * f + ci
    err = np.abs(p / oracle.exp2(f) - 1.0).max()
    assert err <= 2.0 ** -9
    assert err <= (8e-5 if deg == 3 else 2e-7)


def test_empty_problem_rule_needs_no_device(lib):
    # the tensor API answers a problem with a size of 0 with empty results and
    # launches nothing, but still refuses a head dim the kernels do not have
    for D in (64, 128, 256):
        assert fa._empty_problem("fa_fwd", D)
    with pytest.raises(fa.FAError):
        fa._empty_problem("fa_fwd", 96)
