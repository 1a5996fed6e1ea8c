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
one (units numbered tile-major), for fixed-length batches and for packed
batches (sequences of different lengths, including empty ones and lengths
that are not multiples of 128: units past a sequence's tiles are skipped and
take no steps), and for the ascending order of the head-dim-256 kernel (a
unit is a key tile and one output half; 64-query blocks).  This is the
argument the kernel relies on for not deadlocking; its bounded waits would
report a deadlock as an error code, not hang.  At D = 64 and 128 the places
alternate between two accumulators (place p is the (p // 2)-th term of
accumulator p % 2, under that accumulator's counter); `split` models that.

`run_warps` models the kernel's drain more closely: each of a CTA's four
drain warps has its own counters (its 32 rows of a block) and passes its
turn on a block only when it takes the next block out of Tensor Memory (or
at the end of the unit), and no warp can take block k before all four have
taken block k - 1 (the tensor core reuses that space).
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
# nb[bh]: tiles of head bh's sequence (nT for fixed length; fewer, or 0, in a
# packed batch, whose units are still numbered over the longest sequence's nT)


def noncausal_position(bh, j, i, nT, nb, G):
    r = (bh * nT + j) // G
    j0 = min(max(r * G - bh * nT, 0), nb)
    j1 = min((r + 1) * G - bh * nT, nb)

    def in_round(lo, hi):
        return max(0, min(j1, hi) - max(j0, lo))

    if j < i:
        ahead = in_round(j + 1, i + 1)
    elif j > i:
        ahead = in_round(j + 1, nb) + in_round(0, i + 1)
    else:
        ahead = 0
    return j0 + ahead


def noncausal_schedule(BH, nT, G, nb=None):
    nb = nb or [nT] * BH
    U = BH * nT
    seqs = []
    for c in range(G):
        seq = []
        for u in cta_units(c, U, G):
            bh, j = divmod(u, nT)
            if j >= nb[bh]:
                continue  # past the sequence's end: skipped
            for s in range(nb[bh]):
                i = (j + s) % nb[bh]
                seq.append((bh, i, noncausal_position(bh, j, i, nT, nb[bh], G)))
        seqs.append(seq)
    return seqs


# ---- causal mask: units tile-major, blocks ascending from j, order by arrival


def causal_schedule(BH, nT, G, nb=None):
    nb = nb or [nT] * BH
    U = BH * nT

    def coords(u):
        return u % BH, u // BH

    key = {}
    for c in range(G):
        start = 0
        for u in cta_units(c, U, G):
            bh, j = coords(u)
            key[(bh, j)] = start - j
            start += max(nb[bh] - j, 0)  # skipped units take no steps
    seqs = []
    for c in range(G):
        seq = []
        for u in cta_units(c, U, G):
            bh, j = coords(u)
            for i in range(j, nb[bh]):
                rank = sum(1 for jp in range(i + 1) if (key[(bh, jp)], jp) < (key[(bh, j)], j))
                seq.append((bh, i, rank))
        seqs.append(seq)
    return seqs


# ---- head dim 256: a unit is (head, key tile j, output half); 64-query
# blocks ascending from the first visible one; key tiles take their turns per
# (head, half, block) in ascending order


def d256_schedule(BH, nT, G, causal, lens=None):
    lens = lens or [nT * 128] * BH
    U = BH * nT * 2
    seqs = []
    for c in range(G):
        seq = []
        for u in cta_units(c, U, G):
            oh, j, bh = u & 1, (u >> 1) % nT, (u >> 1) // nT
            if j * 128 >= lens[bh]:
                continue
            nq = (lens[bh] + 63) // 64
            for i in range((j * 128) // 64 if causal else 0, nq):
                seq.append(((bh, oh), i, j))
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


def split(seqs):
    """Places alternating between two accumulators: (head, block, place p)
    becomes turn p // 2 on the counter of (head, accumulator p % 2, block)."""
    return [[((bh, p % 2), i, p // 2) for bh, i, p in seq] for seq in seqs]


def run_warps(seqs, seed, unit_ends, warps=4):
    """Per-warp drains with deferred releases (see the module docstring).
    seqs[c] = [(counter key, turn)], unit_ends[c] = indices of the last block
    of each unit.  False on deadlock."""
    rnd = random.Random(seed)
    counter = {}
    # per CTA and warp: blocks loaded, blocks added (turn taken)
    loaded = [[0] * warps for _ in seqs]
    added = [[0] * warps for _ in seqs]
    left = sum(len(s) for s in seqs) * warps
    while left:
        moved = False
        cand = [(c, q) for c in range(len(seqs)) for q in range(warps)]
        rnd.shuffle(cand)
        for c, q in cand:
            seq, k = seqs[c], added[c][q]
            if k == len(seq) or rnd.random() < 0.3:
                continue
            if loaded[c][q] == k:
                # take block k out of TMEM: needs every warp to have taken k - 1
                if min(loaded[c]) < k:
                    continue
                loaded[c][q] = k + 1
                if k > 0 and (k - 1) not in unit_ends[c]:
                    key = seq[k - 1][0] + (q,)
                    counter[key] = counter.get(key, 0) + 1  # deferred release of k - 1
                moved = True
                continue
            key, turn = seq[k][0] + (q,), seq[k][1]
            if counter.get(key, 0) != turn:
                continue
            added[c][q] = k + 1
            left -= 1
            if k in unit_ends[c]:
                counter[key] = turn + 1  # the unit's last block: released at once
            moved = True
        if not moved:
            stuck = all(added[c][q] == len(seqs[c]) or
                        (loaded[c][q] == added[c][q] and min(loaded[c]) < added[c][q]) or
                        (loaded[c][q] > added[c][q] and
                         counter.get(seqs[c][added[c][q]][0] + (q,), 0) != seqs[c][added[c][q]][1])
                        for c in range(len(seqs)) for q in range(warps))
            if stuck:
                return False
    return True


def warp_view(seqs, lens):
    """(head, block, place) schedules -> per-warp model input: counter key
    (head, block, accumulator), turn = place // 2; unit ends from the per-CTA
    unit lengths."""
    out, ends = [], []
    for seq, ls in zip(seqs, lens):
        out.append([((bh, i, p % 2), p // 2) for bh, i, p in seq])
        e, pos = set(), 0
        for n in ls:
            pos += n
            if n:
                e.add(pos - 1)
        ends.append(e)
    return out, ends


def unit_lengths(BH, nT, G, causal, nb=None):
    nb = nb or [nT] * BH
    out = []
    for c in range(G):
        ls = []
        for u in cta_units(c, BH * nT, G):
            bh, j = (u % BH, u // BH) if causal else divmod(u, nT)
            ls.append(0 if j >= nb[bh] else (nb[bh] - j if causal else nb[bh]))
        out.append(ls)
    return out


def turns_are_permutations(seqs):
    per_block = {}
    for seq in seqs:
        for bh, i, turn in seq:
            per_block.setdefault((bh, i), []).append(turn)
    return all(sorted(t) == list(range(len(t))) for t in per_block.values())


SHAPES = [(1, 5, 2), (3, 7, 4), (2, 9, 5), (4, 16, 7), (5, 12, 148), (16, 12, 37), (6, 20, 13)]


@pytest.mark.parametrize("BH,nT,G", SHAPES)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("two_acc", [False, True])
def test_fixed_order_schedule_completes(BH, nT, G, causal, two_acc):
    G = min(G, BH * nT)  # the grid is min(units, SMs)
    seqs = (causal_schedule if causal else noncausal_schedule)(BH, nT, G)
    if two_acc:
        seqs = split(seqs)
    assert turns_are_permutations(seqs)
    for seed in range(3):
        assert run(seqs, seed)


def packed_tiles(BH, nT, seed):
    """Seeded per-sequence tile counts of a packed batch: lengths 0, 1, exact
    multiples of 128 and ragged ones, the longest sequence at nT tiles."""
    rnd = random.Random(seed)
    lens = [rnd.choice([0, 1, 127, 128, 129, 300, rnd.randrange(1, nT * 128 + 1)])
            for _ in range(BH)]
    lens[rnd.randrange(BH)] = nT * 128  # the longest sequence sizes the launch
    return lens, [(n + 127) // 128 for n in lens]


PACKED = [(3, 4, 5), (5, 6, 7), (8, 3, 4), (6, 9, 148), (12, 5, 17)]


@pytest.mark.parametrize("BH,nT,G", PACKED)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("two_acc", [False, True])
def test_packed_batch_schedule_completes(BH, nT, G, causal, seed, two_acc):
    G = min(G, BH * nT)
    _, nb = packed_tiles(BH, nT, seed)
    seqs = (causal_schedule if causal else noncausal_schedule)(BH, nT, G, nb)
    if two_acc:
        seqs = split(seqs)
    assert turns_are_permutations(seqs)
    for s in range(3):
        assert run(seqs, s)


@pytest.mark.parametrize("BH,nT,G", [(1, 4, 3), (2, 5, 7), (3, 8, 11), (4, 6, 148)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("packed", [False, True])
def test_head_dim_256_ascending_order_completes(BH, nT, G, causal, packed):
    G = min(G, BH * nT * 2)
    lens = packed_tiles(BH, nT, BH + nT)[0] if packed else None
    seqs = d256_schedule(BH, nT, G, causal, lens)
    assert turns_are_permutations(seqs)
    for s in range(3):
        assert run(seqs, s)


@pytest.mark.parametrize("BH,nT,G", SHAPES[:5] + PACKED[:3])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("packed", [False, True])
def test_per_warp_drains_with_deferred_release_complete(BH, nT, G, causal, packed):
    G = min(G, BH * nT)
    nb = packed_tiles(BH, nT, BH * 7 + nT)[1] if packed else None
    seqs = (causal_schedule if causal else noncausal_schedule)(BH, nT, G, nb)
    wseqs, ends = warp_view(seqs, unit_lengths(BH, nT, G, causal, nb))
    for s in range(3):
        assert run_warps(wseqs, s, ends)


def test_warp_model_detects_crossed_deferred_releases():
    # two CTAs, one block each of two units' worth: each waits for the other's
    # release of a block that it releases only after its own next turn
    wseqs = [[((0, 0, 0), 1), ((0, 1, 0), 0)], [((0, 1, 0), 1), ((0, 0, 0), 0)]]
    assert not run_warps(wseqs, 0, [{1}, {1}], warps=1)


def test_model_detects_a_cycle():
    # the model itself must be able to fail: two CTAs whose turns cross
    seqs = [[(0, 0, 1), (0, 1, 0)], [(0, 1, 1), (0, 0, 0)]]
    assert turns_are_permutations(seqs)
    assert not run(seqs, 0)
