"""GB300-native (sm_103a) exact attention: fused forward and backward kernels.

The compute path is a C-ABI shared library (``libfa_gb300.so``, declared in
``include/fa.h``) built from ``csrc/``; ``exact_attention_36_gb300.fa`` is the
thin ctypes binding over it.  There is no CPU or PyTorch fallback: every call
fails loudly when the library is missing.

Importing this package is cheap; the library is loaded on first use of
``forward`` / ``backward`` (and the other names re-exported from ``fa``).
"""

__all__ = ["forward", "backward", "forward_varlen", "backward_varlen", "fwd", "bwd",
           "bwd_deterministic", "fwd_varlen", "bwd_varlen", "bwd_varlen_deterministic", "bwd_workspace_size",
           "bwd_semaphore_bytes", "FAError"]


def __getattr__(name):
    if name in __all__ or name in ("lib", "exp2_eval", "exp2_sweep", "device_error"):
        from . import fa
        return getattr(fa, name)
    raise AttributeError(name)
