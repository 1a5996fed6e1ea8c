"""Model of the fixed-order dQ schedule of the deterministic backward (no GPU).

The kernel's CTAs are persistent: CTA c runs the units base + c of even rounds
and base + G - 1 - c of odd rounds.  A unit (head, key tile j) adds its share
of every dQ block it visits in a fixed order, waiting on the block's counter
for its turn.  These tests restate the orders in Python and check, for many
shapes and random per-step delays, that

  * the turns of each block are a permutation 0 .. n-1 of the tiles that
    visit it (every counter reaches its end), and
  * the waits never form a cycle (the run always completes),

for the order by rounds without a causal mask (tiles visit the blocks
rotated, starting at block j) and the order by simulated arrival step under
one (units numbered tile-major).  This is the argument the kernel relies on
for not deadlocking; its bounded waits would report a deadlock as an error
code, not hang.
"""
import random

import pytest


def cta_units(c, U, G):
    r, out = 0, []
    while r * G < U:
        u = r * G + (G - 1 - c if r & 1 else c)
        if u < U:
            out.append(u)
        r += 1
    return out


# ---- without a causal mask: units head-major, blocks rotated, order by rounds


def noncausal_position(bh, j, i, nT, G):
    r = (bh * nT + j) // G
    j0 = min(max(r * G - bh * nT, 0), nT)
    j1 = min((r + 1) * G - bh * nT, nT)

    def in_round(lo, hi):
        return max(0, min(j1, hi) - max(j0, lo))

    if j < i:
        ahead = in_round(j + 1, i + 1)
    elif j > i:
        ahead = in_round(j + 1, nT) + in_round(0, i + 1)
    else:
        ahead = 0
    return j0 + ahead


def noncausal_schedule(BH, nT, G):
    U = BH * nT
    seqs = []
    for c in range(G):
        seq = []
        for u in cta_units(c, U, G):
            bh, j = divmod(u, nT)
            for s in range(nT):
                i = (j + s) % nT
                seq.append((bh, i, noncausal_position(bh, j, i, nT, G)))
        seqs.append(seq)
    return seqs


# ---- causal mask: units tile-major, blocks ascending from j, order by arrival


def causal_schedule(BH, nT, G):
    U = BH * nT

    def coords(u):
        return u % BH, u // BH

    key = {}
    for c in range(G):
        start = 0
        for u in cta_units(c, U, G):
            bh, j = coords(u)
            key[(bh, j)] = start - j
            start += nT - j
    seqs = []
    for c in range(G):
        seq = []
        for u in cta_units(c, U, G):
            bh, j = coords(u)
            for i in range(j, nT):
                rank = sum(1 for jp in range(i + 1) if (key[(bh, jp)], jp) < (key[(bh, j)], j))
                seq.append((bh, i, rank))
        seqs.append(seq)
    return seqs


def run(seqs, seed):
    """Advance CTAs in random order with random stalls; False on deadlock."""
    rnd = random.Random(seed)
    counter, pos = {}, [0] * len(seqs)
    left = sum(len(s) for s in seqs)
    while left:
        moved = False
        order = list(range(len(seqs)))
        rnd.shuffle(order)
        for c in order:
            if pos[c] == len(seqs[c]) or rnd.random() < 0.3:
                continue
            bh, i, turn = seqs[c][pos[c]]
            if counter.get((bh, i), 0) == turn:
                counter[(bh, i)] = turn + 1
                pos[c] += 1
                left -= 1
                moved = True
        if not moved and not any(
                pos[c] < len(seqs[c]) and counter.get(seqs[c][pos[c]][:2], 0) == seqs[c][pos[c]][2]
                for c in range(len(seqs))):
            return False
    return True


def turns_are_permutations(seqs):
    per_block = {}
    for seq in seqs:
        for bh, i, turn in seq:
            per_block.setdefault((bh, i), []).append(turn)
    return all(sorted(t) == list(range(len(t))) for t in per_block.values())


SHAPES = [(1, 5, 2), (3, 7, 4), (2, 9, 5), (4, 16, 7), (5, 12, 148), (16, 12, 37), (6, 20, 13)]


@pytest.mark.parametrize("BH,nT,G", SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_fixed_order_schedule_completes(BH, nT, G, causal):
    G = min(G, BH * nT)  # the grid is min(units, SMs)
    seqs = (causal_schedule if causal else noncausal_schedule)(BH, nT, G)
    assert turns_are_permutations(seqs)
    for seed in range(3):
        assert run(seqs, seed)


def test_model_detects_a_cycle():
    # the model itself must be able to fail: two CTAs whose turns cross
    seqs = [[(0, 0, 1), (0, 1, 0)], [(0, 1, 1), (0, 0, 0)]]
    assert turns_are_permutations(seqs)
    assert not run(seqs, 0)
