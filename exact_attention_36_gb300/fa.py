"""ctypes binding of libfa_gb300.so (C ABI declared in include/fa.h).

Argument marshalling only: every step of the attention computation runs in
the library's CUDA kernels.  PyTorch supplies device memory and the current
stream.  There is no fallback: if the library is missing or the device is not
supported, calls raise ``FAError``.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libfa_gb300.so")

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)
DEFAULT = -1  # selects the library default for a numerics knob


class FAError(RuntimeError):
    """A libfa_gb300 entry point returned an error status."""

    def __init__(self, where: str, status: int, cuda_err: int = 0):
        self.status = status
        self.cuda_err = cuda_err
        name = lib().fa_status_string(status).decode()
        extra = f" (cuda error {cuda_err})" if status == FA_ERR_CUDA else ""
        super().__init__(f"{where}: {name}{extra}")


_lib = None


def lib():
    """The loaded library (loaded on first use; raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "(there is no CPU fallback)")
        L = ctypes.CDLL(_LIB_PATH)
        vp, i, f, ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_longlong
        L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
        L.fa_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, f, i, i, vp]
        L.fa_fwd_varlen.argtypes = [vp] * 6 + [i, i, i, i, i, i, f, vp]
        L.fa_bwd_workspace_size.argtypes = [i, i, i, i]
        L.fa_bwd_workspace_size.restype = ctypes.c_size_t
        L.fa_bwd.argtypes = [vp] * 11 + [i, i, i, i, i, f, vp]
        L.fa_bwd_ex.argtypes = [vp] * 11 + [i, i, i, i, i, f, i, vp]
        L.fa_bwd_varlen.argtypes = [vp] * 12 + [i, i, i, i, i, i, f, vp]
        L.fa_bwd_varlen_workspace_size.argtypes = [i, i, i]
        L.fa_bwd_varlen_workspace_size.restype = ctypes.c_size_t
        L.fa_bwd_deterministic.argtypes = [vp] * 12 + [i, i, i, i, i, f, vp]
        L.fa_bwd_varlen_deterministic.argtypes = [vp] * 13 + [i, i, i, i, i, i, f, vp]
        L.fa_bwd_semaphore_bytes.argtypes = [i, i, i, i]
        L.fa_bwd_semaphore_bytes.restype = ctypes.c_size_t
        L.fa_bwd_varlen_semaphore_bytes.argtypes = [i, i, i, i, i]
        L.fa_bwd_varlen_semaphore_bytes.restype = ctypes.c_size_t
        L.fa_status_string.argtypes = [i]
        L.fa_status_string.restype = ctypes.c_char_p
        L.fa_last_cuda_error.argtypes = [ctypes.POINTER(i)]
        L.fa_device_error.argtypes = [ctypes.POINTER(i), i]
        L.fa_exp2_eval.argtypes = [vp, vp, ll, i, vp]
        L.fa_exp2_sweep.argtypes = [f, f, i, vp, vp]
        for name in ("fa_fwd", "fa_fwd_ex", "fa_fwd_varlen", "fa_bwd", "fa_bwd_ex", "fa_bwd_varlen",
                     "fa_bwd_deterministic", "fa_bwd_varlen_deterministic",
                     "fa_last_cuda_error",
                     "fa_device_error",
                     "fa_exp2_eval", "fa_exp2_sweep"):
            getattr(L, name).restype = i
        _lib = L
    return _lib


def _check(where: str, st: int):
    if st != FA_OK:
        err = ctypes.c_int(0)
        lib().fa_last_cuda_error(ctypes.byref(err))
        raise FAError(where, st, err.value)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else stream)


def _ptr(t: torch.Tensor):
    return ctypes.c_void_p(t.data_ptr())


def _check_bshd(name, t, shape=None):
    if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.dim() != 4:
        raise ValueError(f"{name}: expected a contiguous CUDA bf16 tensor [B, S, H, D]")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)} != {tuple(shape)}")


# ---------------------------------------------------------------- raw calls


def fwd(q, k, v, o, lse, causal: bool, scale: float, stream=None,
        rescale_threshold: float = DEFAULT, poly_exp2_groups: int = DEFAULT,
        poly_exp2_degree: int = DEFAULT):
    """fa_fwd_ex on caller-provided tensors (o, lse written)."""
    B, S, H, D = q.shape
    st = lib().fa_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, S, D,
                         int(bool(causal)), float(scale), float(rescale_threshold),
                         int(poly_exp2_groups), int(poly_exp2_degree), _stream(stream))
    _check("fa_fwd", st)


def fwd_varlen(q, k, v, o, lse, cu_seqlens, max_seqlen: int, causal: bool, scale: float,
               stream=None):
    """fa_fwd_varlen on caller-provided tensors: q, k, v, o bf16 [T, H, D],
    lse fp32 [H, T], cu_seqlens int32 [B+1] on the device."""
    T, H, D = q.shape
    B = cu_seqlens.numel() - 1
    _check("fa_fwd_varlen", lib().fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                                _ptr(cu_seqlens), B, int(max_seqlen), T, H, D,
                                                int(bool(causal)), float(scale),
                                                _stream(stream)))


def bwd_varlen(q, k, v, o, dout, lse, dq_acc, delta, dq, dk, dv, cu_seqlens, max_seqlen: int,
               causal: bool, scale: float, stream=None):
    """fa_bwd_varlen on caller-provided tensors (packed [T, H, D] layout)."""
    T, H, D = q.shape
    B = cu_seqlens.numel() - 1
    _check("fa_bwd_varlen", lib().fa_bwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq_acc), _ptr(delta),
        _ptr(dq), _ptr(dk), _ptr(dv), _ptr(cu_seqlens), B, int(max_seqlen), T, H, D,
        int(bool(causal)), float(scale), _stream(stream)))


def bwd_varlen_deterministic(q, k, v, o, dout, lse, dq_acc, delta, dq_sem, dq, dk, dv, cu_seqlens,
                             max_seqlen: int, causal: bool, scale: float, stream=None):
    """fa_bwd_varlen_deterministic on caller-provided tensors (packed layout, fixed-order dQ)."""
    T, H, D = q.shape
    B = cu_seqlens.numel() - 1
    _check("fa_bwd_varlen_deterministic", lib().fa_bwd_varlen_deterministic(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq_acc), _ptr(delta),
        _ptr(dq_sem), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(cu_seqlens), B, int(max_seqlen), T, H, D,
        int(bool(causal)), float(scale), _stream(stream)))


def bwd_workspace_size(B: int, H: int, S: int, D: int) -> int:
    return int(lib().fa_bwd_workspace_size(B, H, S, D))


def bwd(q, k, v, o, dout, lse, dq_acc, delta, dq, dk, dv, causal: bool, scale: float,
        stream=None, pair_mode: int = DEFAULT):
    """fa_bwd (pair_mode -1) or fa_bwd_ex on caller-provided tensors (dq, dk,
    dv written).  pair_mode: 0 one CTA per key tile, 1 CTA pairs (D = 128)."""
    B, S, H, D = q.shape
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq_acc),
            _ptr(delta), _ptr(dq), _ptr(dk), _ptr(dv), B, H, S, D, int(bool(causal)),
            float(scale))
    if pair_mode == DEFAULT:
        _check("fa_bwd", lib().fa_bwd(*args, _stream(stream)))
    else:
        _check("fa_bwd_ex", lib().fa_bwd_ex(*args, int(pair_mode), _stream(stream)))


def bwd_deterministic(q, k, v, o, dout, lse, dq_acc, delta, dq_sem, dq, dk, dv, causal: bool,
                      scale: float, stream=None):
    """fa_bwd_deterministic on caller-provided tensors (fixed-order dQ)."""
    B, S, H, D = q.shape
    st = lib().fa_bwd_deterministic(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                                    _ptr(dq_acc), _ptr(delta), _ptr(dq_sem), _ptr(dq), _ptr(dk),
                                    _ptr(dv), B, H, S, D, int(bool(causal)), float(scale),
                                    _stream(stream))
    _check("fa_bwd_deterministic", st)


def bwd_semaphore_bytes(B: int, H: int, S: int, D: int) -> int:
    return int(lib().fa_bwd_semaphore_bytes(B, H, S, D))


def bwd_varlen_semaphore_bytes(B: int, max_seqlen: int, total: int, H: int, D: int) -> int:
    return int(lib().fa_bwd_varlen_semaphore_bytes(B, max_seqlen, total, H, D))


# ---------------------------------------------------------------- tensor API


def _empty_problem(where: str, D: int) -> bool:
    """Called for a problem with no elements (a size of 0, which the C ABI
    rejects): the result is empty and nothing is launched.  The library must
    still load and the head dim must still be one the kernels support."""
    lib()
    if D not in (64, 128, 256):
        raise FAError(where, FA_ERR_UNSUPPORTED)
    return True


def forward(q, k, v, causal: bool = False, scale: float | None = None, stream=None,
            rescale_threshold: float = DEFAULT, poly_exp2_groups: int = DEFAULT,
            poly_exp2_degree: int = DEFAULT):
    """Exact attention forward.  q, k, v: CUDA bf16 [B, S, H, D].

    Returns (o bf16 [B, S, H, D], lse fp32 [B, H, S]); empty tensors when
    B, S or H is 0.
    """
    _check_bshd("q", q)
    _check_bshd("k", k, q.shape)
    _check_bshd("v", v, q.shape)
    B, S, H, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    if q.numel() == 0 and _empty_problem("fa_fwd", D):
        return o, lse
    fwd(q, k, v, o, lse, causal, scale, stream, rescale_threshold, poly_exp2_groups,
        poly_exp2_degree)
    return o, lse


def backward(q, k, v, o, dout, lse, causal: bool = False, scale: float | None = None,
             stream=None, deterministic: bool = False, pair_mode: int = DEFAULT):
    """Exact attention backward.  Returns (dq, dk, dv), bf16 [B, S, H, D].

    deterministic=True sums dQ over key tiles in a fixed order, so repeated
    calls give bitwise-identical results (dK and dV always are).
    pair_mode selects the main kernel: 0 one CTA per key tile, 1 CTA pairs
    (D = 128 only), -1 the library default."""
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _check_bshd(name, t, q.shape)
    B, S, H, D = q.shape
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, S) or not lse.is_contiguous():
        raise ValueError("lse: expected contiguous fp32 [B, H, S]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if q.numel() == 0 and _empty_problem("fa_bwd", D):
        return torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    n = B * H * S
    ws = torch.empty(bwd_workspace_size(B, H, S, D), dtype=torch.uint8, device=q.device)
    acc_bytes = (n * D * 4 + 255) // 256 * 256
    dq_acc = ws[:acc_bytes].view(torch.float32)
    delta = ws[acc_bytes:acc_bytes + n * 4].view(torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    if deterministic:
        sem = torch.empty(bwd_semaphore_bytes(B, H, S, D) // 4, dtype=torch.int32,
                          device=q.device)
        bwd_deterministic(q, k, v, o, dout, lse, dq_acc, delta, sem, dq, dk, dv, causal, scale,
                          stream)
    else:
        bwd(q, k, v, o, dout, lse, dq_acc, delta, dq, dk, dv, causal, scale, stream, pair_mode)
    return dq, dk, dv


def _check_packed(name, t, shape=None):
    if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 3 or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CUDA bf16 tensor [T, H, D]")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)} != {tuple(shape)}")


def _check_cu(cu_seqlens, device):
    if (not cu_seqlens.is_cuda or cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1
            or cu_seqlens.numel() < 2 or not cu_seqlens.is_contiguous()
            or cu_seqlens.device != device):
        raise ValueError("cu_seqlens: expected a contiguous CUDA int32 tensor [B+1]")


def forward_varlen(q, k, v, cu_seqlens, max_seqlen: int, causal: bool = False,
                   scale: float | None = None, stream=None):
    """Exact attention over a packed batch: sequence b is tokens
    [cu_seqlens[b], cu_seqlens[b+1]) of q, k, v (CUDA bf16 [T, H, D]).

    Returns (o bf16 [T, H, D], lse fp32 [H, T])."""
    _check_packed("q", q)
    _check_packed("k", k, q.shape)
    _check_packed("v", v, q.shape)
    _check_cu(cu_seqlens, q.device)
    T, H, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = torch.empty_like(q)
    lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
    if q.numel() == 0 and _empty_problem("fa_fwd_varlen", D):
        return o, lse
    fwd_varlen(q, k, v, o, lse, cu_seqlens, max_seqlen, causal, scale, stream)
    return o, lse


def backward_varlen(q, k, v, o, dout, lse, cu_seqlens, max_seqlen: int, causal: bool = False,
                    scale: float | None = None, stream=None, deterministic: bool = False):
    """Exact attention backward over a packed batch (the forward_varlen
    layout).  Returns (dq, dk, dv), bf16 [T, H, D].  deterministic=True sums
    dQ over key tiles in a fixed order (bitwise-repeatable results)."""
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _check_packed(name, t, q.shape)
    _check_cu(cu_seqlens, q.device)
    T, H, D = q.shape
    if lse.dtype != torch.float32 or tuple(lse.shape) != (H, T) or not lse.is_contiguous():
        raise ValueError("lse: expected contiguous fp32 [H, T]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if q.numel() == 0 and _empty_problem("fa_bwd_varlen", D):
        return torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    n = H * T
    ws = torch.empty(int(lib().fa_bwd_varlen_workspace_size(T, H, D)), dtype=torch.uint8,
                     device=q.device)
    acc_bytes = (n * D * 4 + 255) // 256 * 256
    dq_acc = ws[:acc_bytes].view(torch.float32)
    delta = ws[acc_bytes:acc_bytes + n * 4].view(torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    if deterministic:
        B = cu_seqlens.numel() - 1
        sem = torch.empty(bwd_varlen_semaphore_bytes(B, int(max_seqlen), T, H, D) // 4,
                          dtype=torch.int32, device=q.device)
        bwd_varlen_deterministic(q, k, v, o, dout, lse, dq_acc, delta, sem, dq, dk, dv, cu_seqlens,
                                 max_seqlen, causal, scale, stream)
    else:
        bwd_varlen(q, k, v, o, dout, lse, dq_acc, delta, dq, dk, dv, cu_seqlens, max_seqlen,
                   causal, scale, stream)
    return dq, dk, dv


# ---------------------------------------------------------------- diagnostics


def device_error(clear: bool = True) -> int:
    """Synchronise and return (then clear) the device error word (0 = none)."""
    code = ctypes.c_int(0)
    st = lib().fa_device_error(ctypes.byref(code), int(bool(clear)))
    if st not in (FA_OK, FA_ERR_TIMEOUT):
        _check("fa_device_error", st)
    return code.value


def exp2_eval(x: torch.Tensor, variant: int, stream=None) -> torch.Tensor:
    """Approximate 2^x on the device (variant 0 kernel polynomial, 1 full-range
    polynomial, 2 MUFU, 3 the kernel polynomial in two-lane form, 4 the
    degree-5 full-range polynomial, 5 the degree-5 kernel polynomial in
    two-lane form)."""
    if not x.is_cuda or x.dtype != torch.float32 or not x.is_contiguous():
        raise ValueError("x: expected a contiguous CUDA fp32 tensor")
    y = torch.empty_like(x)
    _check("fa_exp2_eval", lib().fa_exp2_eval(_ptr(x), _ptr(y), x.numel(), variant,
                                              _stream(stream)))
    return y


def exp2_sweep(lo: float, hi: float, variant: int, device="cuda"):
    """Max relative error of a variant over every fp32 in [lo, hi]: (err, x)."""
    out = torch.zeros(2, dtype=torch.float64, device=device)
    _check("fa_exp2_sweep", lib().fa_exp2_sweep(float(lo), float(hi), variant, _ptr(out),
                                                _stream(None)))
    err, x = out.cpu().tolist()
    return err, x
