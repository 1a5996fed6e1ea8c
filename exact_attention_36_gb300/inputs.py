"""Seeded synthetic inputs shared by the tests, the bench and the oracle runs.

This module holds no attention arithmetic: it only draws random tensors.
The pages measure on no dataset; these shapes and distributions stand in for
their workloads (N(0,1) bf16 activations; a stress mix with peaked softmax
rows and a few dominant keys that makes the running row maximum jump).

Recipe (the one reading of "N(0,1) from seed" used everywhere):
  * one CPU ``torch.Generator`` seeded with ``seed``;
  * draw order Q, K, V, dO, each ``torch.randn(B, S, H, D, float32)`` and
    then rounded to bf16 (round to nearest even);
  * ``stress=True``: Q is drawn as 4 * randn; after K is drawn, for every
    (b, h) independently, ``randperm(S)[:round(0.01 * S)]`` picks 1 % of the
    key rows, which are multiplied by 8 (exact in bf16); V and dO are then
    drawn as usual.
  * packed batches (sequences of different lengths back to back): the same
    draw with B = 1 and S = the total token count, split by ``cu_seqlens``;
    a length mix comes from ``packed_lengths`` (its own generator, seeded).
  * problems of several GiB per tensor (``make_qkvdo_device``): one
    ``torch.Generator`` on the device, seeded with ``seed``; Q, K, V, dO in
    that order, each ``torch.randn(B, S, H, D)`` drawn directly in bf16 on
    the device (N(0,1) as torch's device generator rounds it).  The checks
    copy the heads they compare to the host.
"""
from __future__ import annotations

import math

import torch

__all__ = ["make_qkvdo", "make_qkvdo_device", "make_packed", "packed_lengths", "default_scale",
           "WORKLOADS"]


def default_scale(D: int) -> float:
    """Softmax scale 1/sqrt(D)."""
    return 1.0 / math.sqrt(D)


def make_qkvdo(B: int, H: int, S: int, D: int, seed: int = 0, stress: bool = False,
               with_dout: bool = True):
    """Return CPU bf16 tensors (q, k, v, dout) of shape [B, S, H, D].

    dout is None when with_dout is False (it is still drawn last, so the
    Q/K/V values do not depend on with_dout).
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    shape = (B, S, H, D)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    if stress:
        q = q * 4.0
    q = q.to(torch.bfloat16)
    k = torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
    if stress:
        n_hot = int(round(0.01 * S))
        if n_hot > 0:
            for b in range(B):
                for h in range(H):
                    idx = torch.randperm(S, generator=g)[:n_hot]
                    k[b, idx, h, :] = k[b, idx, h, :] * 8
    v = torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
    dout = torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return q, k, v, (dout if with_dout else None)


def make_qkvdo_device(B: int, H: int, S: int, D: int, seed: int = 0, device="cuda"):
    """Return device bf16 tensors (q, k, v, dout) of shape [B, S, H, D], drawn
    on the device (for problems too large to draw on the host)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    shape = (B, S, H, D)
    return tuple(torch.randn(shape, generator=g, dtype=torch.bfloat16, device=device)
                 for _ in range(4))


# The workloads the library is measured and checked on: (name, B, H, S, D,
# causal list, stress).
def packed_lengths(n: int, max_len: int, seed: int = 0, min_len: int = 1) -> list[int]:
    """n sequence lengths drawn uniformly from [min_len, max_len] (seeded), the
    first one max_len so that the longest sequence is exactly max_len."""
    g = torch.Generator().manual_seed(seed)
    rest = torch.randint(min_len, max_len + 1, (n - 1,), generator=g).tolist() if n > 1 else []
    return [max_len] + rest


def make_packed(lengths, H: int, D: int, seed: int = 0, stress: bool = False,
                with_dout: bool = True):
    """A packed batch: q, k, v (, dout) bf16 [T, H, D] with T = sum(lengths),
    and cu_seqlens int32 [len(lengths) + 1] (CPU tensors)."""
    T = int(sum(lengths))
    q, k, v, do = make_qkvdo(1, H, T, D, seed=seed, stress=stress, with_dout=with_dout)
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.as_tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    return q[0], k[0], v[0], (do[0] if do is not None else None), cu


WORKLOADS = {
    "C1": dict(B=1, H=2, S=256, D=64, causal=(False,), stress=False),
    "C2": dict(B=4, H=16, S=2048, D=128, causal=(False,), stress=False),
    "C3": dict(B=2, H=16, S=8192, D=128, causal=(True,), stress=False),
    "C4": dict(B=1, H=16, S=32768, D=128, causal=(False, True), stress=False),
}
# stress sweep: D in {64, 128, 256} x (S, B) in {(1024, 16), (4096, 4), (16384, 1)}, H = 16
for _D in (64, 128, 256):
    for (_S, _B) in ((1024, 16), (4096, 4), (16384, 1)):
        WORKLOADS[f"C5_D{_D}_S{_S}"] = dict(B=_B, H=16, S=_S, D=_D, causal=(False, True),
                                            stress=True)
