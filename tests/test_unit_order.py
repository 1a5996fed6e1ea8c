"""Model of the persistent kernels' work-unit orders (no GPU).

Every kernel runs a persistent grid of G CTAs; in round r CTA c takes unit
r * G + c (even rounds) or r * G + G - 1 - c (odd rounds).  The unit number u
maps to the work it stands for.  These tests restate the maps in Python and
check, for many shapes, the properties the kernels rely on:

  * the map is a bijection of [0, U) onto the units (every unit runs once);
  * without a mask the forward numbers units head by head, so the CTAs of a
    round share few heads;
  * under a causal mask the units are longest-first over all heads, or within
    groups of half a grid of heads when many heads' tensors exceed L2, and
    within each group every unit is at least as long as the next one;
  * the grouping condition itself (more heads than half the grid, their
    tensors above the L2 size) switches on where it should;
  * the D = 256 backward's and both CTA-pair kernels' unit maps are
    bijections too, the D = 128 pairs cover every key tile once, and the
    serpentine rounds hand every unit to exactly one CTA.
"""
import itertools

import pytest

L2_BYTES = 128 << 20


def fwd_group_size(BH, G, S, D):
    """Heads per group of the causal forward order (BH: no grouping)."""
    kv = min(BH, G) * S * D * 4
    return max(1, G // 2) if (2 * BH > G and kv > L2_BYTES) else BH


def fwd_unit(u, BH, P, causal, gs):
    """(bh, p) of forward unit u: query rows [p * rows, (p + 1) * rows)."""
    if not causal:
        return u // P, u % P
    grp, r = divmod(u, gs * P)
    ge = min(gs, BH - grp * gs)
    return grp * gs + r % ge, P - 1 - r // ge


def bwd_group_size(BH, G, S, D):
    """Heads per group of the causal backward order (0: no grouping)."""
    head_bytes = S * D * 8
    return max(1, G // 2) if (2 * BH > G and min(BH, G) * head_bytes > L2_BYTES) else 0


def bwd_unit(u, BH, nT, causal, gs):
    """(bh, key tile j) of backward unit u."""
    if causal and 0 < gs < BH:
        grp, r = divmod(u, gs * nT)
        ge = min(gs, BH - grp * gs)
        return grp * gs + r % ge, r // ge
    if causal:
        return u % BH, u // BH
    return u // nT, u % nT


def rounds(U, G):
    r = 0
    while r * G < U:
        yield [r * G + (G - 1 - c if r & 1 else c) for c in range(G) if r * G + (G - 1 - c if r & 1 else c) < U]
        r += 1


SHAPES = [(B, H, S) for B, H, S in itertools.product((1, 2, 4, 16), (1, 3, 16), (256, 1000, 1024, 2048, 8192, 32768))]


@pytest.mark.parametrize("B,H,S", SHAPES)
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_order_is_a_bijection_and_longest_first(B, H, S, D, causal):
    G = 152
    BH = B * H
    rows = 128 if D == 256 else 256
    P = (S + rows - 1) // rows
    U = BH * P
    gs = fwd_group_size(BH, G, S, D)
    seen = [fwd_unit(u, BH, P, causal, gs) for u in range(U)]
    assert sorted(seen) == [(bh, p) for bh in range(BH) for p in range(P)]
    if causal:
        # within each group of gs heads the work (p + 1 query tiles' worth of
        # key tiles) never grows along the numbering
        for g0 in range(0, BH, gs):
            ps = [p for bh, p in seen if g0 <= bh < g0 + gs]
            assert ps == sorted(ps, reverse=True)
    else:
        # head by head: a round of G CTAs touches at most ceil(G / P) + 1 heads
        for rnd in rounds(U, G):
            heads = {seen[u][0] for u in rnd}
            assert len(heads) <= -(-G // P) + 1


@pytest.mark.parametrize("B,H,S", SHAPES)
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_order_is_a_bijection_and_longest_first(B, H, S, D, causal):
    G = 152
    BH = B * H
    nT = (S + 127) // 128
    U = BH * nT
    gs = bwd_group_size(BH, G, S, D)
    seen = [bwd_unit(u, BH, nT, causal, gs) for u in range(U)]
    assert sorted(seen) == [(bh, j) for bh in range(BH) for j in range(nT)]
    if causal:
        # tile j has nT - j query blocks: within each group j never decreases
        size = gs if 0 < gs < BH else BH
        for g0 in range(0, BH, size):
            js = [j for bh, j in seen if g0 <= bh < g0 + size]
            assert js == sorted(js)


def test_grouping_switches_on_only_for_many_heads_beyond_l2():
    G = 152
    # the bench workload (16 heads of 32k rows) and the causal C3 workload keep
    # plain longest-first order
    assert fwd_group_size(16, G, 32768, 128) == 16
    assert fwd_group_size(32, G, 8192, 128) == 32
    assert bwd_group_size(16, G, 32768, 128) == 0
    assert bwd_group_size(32, G, 8192, 128) == 0
    # 256 heads of 1k-2k rows whose K/V (forward) or Q/dO/accumulators
    # (backward) exceed L2 are grouped by half a grid of heads
    assert fwd_group_size(256, G, 1024, 256) == 76
    assert fwd_group_size(256, G, 2048, 128) == 76
    assert bwd_group_size(256, G, 2048, 128) == 76
    assert bwd_group_size(256, G, 1024, 128) == 76
    # many small heads that fit in L2 are not
    assert fwd_group_size(256, G, 1024, 64) == 256
    assert fwd_group_size(256, G, 1024, 128) == 256
    assert bwd_group_size(256, G, 1024, 64) == 0


def d256_unit(u, nT):
    """(bh, key tile j, output half oh) of D = 256 backward unit u: the two
    halves of a key tile, then the key tiles of a head, are adjacent."""
    return (u >> 1) // nT, (u >> 1) % nT, u & 1


def pair_unit(u, nP):
    """(bh, key-tile pair p) of D = 128 CTA-pair unit u: a head's pairs in a row."""
    return u // nP, u % nP


def split_unit(u, BH, nT, causal):
    """(bh, key tile j) of D = 256 split-pair unit u: tile-major under a causal
    mask (longest first across heads), head by head otherwise."""
    return (u % BH, u // BH) if causal else (u // nT, u % nT)


@pytest.mark.parametrize("B,H,S", SHAPES)
def test_other_backward_unit_maps_are_bijections(B, H, S):
    BH = B * H
    nT = (S + 127) // 128
    seen = [d256_unit(u, nT) for u in range(BH * nT * 2)]
    assert sorted(seen) == [(bh, j, oh) for bh in range(BH) for j in range(nT) for oh in range(2)]
    nP = (nT + 1) // 2
    seen = [pair_unit(u, nP) for u in range(BH * nP)]
    assert sorted(seen) == [(bh, p) for bh in range(BH) for p in range(nP)]
    # each pair covers key tiles 2p and 2p + 1 (the second past the end when
    # nT is odd, which that CTA skips): every key tile exactly once
    tiles = sorted((bh, 2 * p + r) for bh, p in seen for r in range(2) if 2 * p + r < nT)
    assert tiles == [(bh, j) for bh in range(BH) for j in range(nT)]
    for causal in (False, True):
        seen = [split_unit(u, BH, nT, causal) for u in range(BH * nT)]
        assert sorted(seen) == [(bh, j) for bh in range(BH) for j in range(nT)]
        if causal:  # tile j has the most query blocks for j = 0: ascending j
            assert [j for _, j in seen] == sorted(j for _, j in seen)


@pytest.mark.parametrize("G", [1, 2, 7, 76, 152])
@pytest.mark.parametrize("U", [1, 5, 151, 152, 153, 1000])
def test_serpentine_rounds_cover_every_unit_once(G, U):
    # CTA (or pair) c takes unit r * G + c in even rounds and r * G + G - 1 - c
    # in odd rounds, while r * G < U
    got = []
    for c in range(G):
        r = 0
        while r * G < U:
            u = r * G + (G - 1 - c if r & 1 else c)
            if u < U:
                got.append(u)
            r += 1
    assert sorted(got) == list(range(U))
