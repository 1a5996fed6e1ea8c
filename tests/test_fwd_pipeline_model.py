"""CPU models of the forward kernel's pipeline protocols (no GPU): D = 128
(two ping-pong query tiles, grouped K/V ring), D = 64 (the same tiles, K and V
in single slots released by MMA commits) and D = 256 (one query tile, two S
buffers, a ring of K/V half-slots).

The forward runs, per CTA, a producer warp (the unit's two Q tiles, then K and
V through a ring of four shared-memory slots used as two groups {V_j, K_j+1},
one full and one empty barrier per group), one MMA-issuing thread and the
softmax warps of query tiles 0 and 1 (each also writes its tile's O and LSE).
Per key tile the MMA thread issues PV0(j), S0(j+1), PV1(j), S1(j+1); S and P
of a tile share one TMEM region, O of each tile accumulates in its own.  A
group is released by one thread of tile 1's softmax when it sees S1(j+1)
complete (the group's last reader, issued after every other MMA that reads it)
or, for the unit's last group, O1; Q is released after the unit's last S MMA.
The softmax rescales O in TMEM when the running maximum jumps, between two PV
MMAs.

This module restates each role in the kernel's order (waits with the kernel's
parity expressions) and runs them with random durations, unit lengths and
causal tile counts (tile 0 one key tile short), checking that every role
finishes, that every parity wait sees exactly its phase, and that no buffer
(Q, the K and V slots, S/P and O in TMEM) is written while a previous use is
still read.  Planted mistakes (a wait or a release moved) must be caught.

D = 256: S(j+1) goes into the other of two TMEM S buffers as soon as K_j+1's
halves are in, before P(j) is waited for; K (head-dim halves) and V (key
halves) stream through one ring of five half-slots in the order the MMAs read
them, each released by a commit after its MMAs; a rescale of O waits for
PV(j-1) on its own barrier, since the commit of S(j) no longer covers it.
"""
import random

import pytest

from tests._pipeline_sim import Barrier, Sim, Violation

GROUPS = 2  # slot groups {V_j, K_j+1} of the four-slot ring


def make_bars():
    B = Barrier
    bars = {'q_full': B('q_full', 1), 'q_empty': B('q_empty', 1)}
    for g in range(GROUPS):
        bars[f'kv_full{g}'] = B(f'kv_full{g}', 1)
        bars[f'kv_empty{g}'] = B(f'kv_empty{g}', 1)
    for t in range(2):
        bars[f's_full{t}'] = B(f's_full{t}', 1)
        bars[f'p_full{t}'] = B(f'p_full{t}', 1)
        bars[f'o_full{t}'] = B(f'o_full{t}', 1)
    return bars


def producer(b, units, rng, skip=()):
    ring = 0
    f = rng.uniform(0.1, 5.0)
    for u, (n0, n1) in enumerate(units):
        yield ('wait', b['q_empty'], (u & 1) ^ 1, u - 1)
        yield ('arrive_tx', b['q_full'], 1)
        yield ('tma', b['q_full'], 1, 'Q', u)
        for j in range(-1, n1):
            g, use = ring % GROUPS, ring // GROUPS
            if 'kv_empty' not in skip:
                yield ('wait', b[f'kv_empty{g}'], (use & 1) ^ 1, use - 1)
            has_v, has_k = j >= 0, j + 1 < n1
            yield ('arrive_tx', b[f'kv_full{g}'], int(has_v) + int(has_k))
            if has_v:
                yield ('tma', b[f'kv_full{g}'], 1, f'V{g}', use)
            if has_k:
                yield ('tma', b[f'kv_full{g}'], 1, f'K{g}', use)
            yield ('delay', f * rng.uniform(0, 30))
            ring += 1


def mma(b, units, skip=()):
    ring = 0
    jj = [0, 0]  # S/P tiles seen by each query tile (TMEM S/P uses 2jj, 2jj + 1)
    for u, (n0, n1) in enumerate(units):
        yield ('wait', b['q_full'], u & 1, u)
        g, use = ring % GROUPS, ring // GROUPS
        yield ('wait', b[f'kv_full{g}'], use & 1, use)
        ring += 1
        kk = (f'K{g}', use)
        yield ('mma', [('Q', u), kk], [('SP0', 2 * jj[0])])
        yield ('commit', b['s_full0'])
        yield ('mma', [('Q', u), kk], [('SP1', 2 * jj[1])])
        yield ('commit', b['s_full1'])
        if n1 == 1:
            yield ('commit', b['q_empty'])
        for j in range(n1):
            g, use = ring % GROUPS, ring // GROUPS
            yield ('wait', b[f'kv_full{g}'], use & 1, use)
            ring += 1
            vv, kk = (f'V{g}', use), (f'K{g}', use)
            if j < n0:
                if 'p_full' not in skip:
                    yield ('wait', b['p_full0'], jj[0] & 1, jj[0])
                yield ('mma', [('SP0', 2 * jj[0] + 1), vv], [('O0', (u, 2 * j))])
                jj[0] += 1
                if j + 1 < n0:
                    yield ('mma', [('Q', u), kk], [('SP0', 2 * jj[0])])
                    yield ('commit', b['s_full0'])
                else:
                    yield ('commit', b['o_full0'])
            yield ('wait', b['p_full1'], jj[1] & 1, jj[1])
            yield ('mma', [('SP1', 2 * jj[1] + 1), vv], [('O1', (u, 2 * j))])
            jj[1] += 1
            if j + 1 < n1:
                if 'q_empty_early' in skip and j + 2 == n1:
                    yield ('commit', b['q_empty'])  # planted: before the last S MMA
                yield ('mma', [('Q', u), kk], [('SP1', 2 * jj[1])])
                yield ('commit', b['s_full1'])
                if j + 2 == n1 and 'q_empty_early' not in skip:
                    yield ('commit', b['q_empty'])  # the last S MMA
            else:
                yield ('commit', b['o_full1'])


def softmax(b, units, t, rng, skip=(), grouped=True):
    f = rng.uniform(0.1, 5.0)
    jj = 0
    grp = 0  # groups released (tile 1)
    for u, (n0, n1) in enumerate(units):
        n = n1 if t else n0
        for j in range(n):
            yield ('wait', b[f's_full{t}'], jj & 1, jj)
            if t == 1 and grouped:
                yield ('arrive', b[f'kv_empty{grp % GROUPS}'])
                grp += 1
                if 'release_early' in skip and j == 0:
                    # planted: {V_0, K_1} released with {K_0}, before its readers ran
                    yield ('arrive', b[f'kv_empty{grp % GROUPS}'])
                    grp += 1
            yield ('ld', f'SP{t}', 2 * jj)
            if j > 0 and rng.random() < 0.3:
                # conditional rescale of O between PV(j-1) and PV(j): reads
                # PV(j-1)'s sum, writes the rescaled one
                yield ('ld', f'O{t}', (u, 2 * j - 2))
                yield ('st', f'O{t}', (u, 2 * j - 1))
            yield ('delay', f * rng.uniform(300, 1500))
            yield ('st', f'SP{t}', 2 * jj + 1)
            yield ('arrive', b[f'p_full{t}'])
            jj += 1
        yield ('wait', b[f'o_full{t}'], u & 1, u)
        if t == 1 and grouped and 'release_early' not in skip:
            yield ('arrive', b[f'kv_empty{grp % GROUPS}'])  # the unit's last group
            grp += 1
        yield ('ld', f'O{t}', (u, 2 * (n - 1)))
        yield ('delay', f * rng.uniform(200, 3000))  # staging, stores, LSE


def simulate(seed, skip=()):
    rng = random.Random(seed)
    units = []
    for _ in range(rng.randint(1, 6)):
        n1 = rng.randint(1, 6)
        causal_short = rng.random() < 0.5 and n1 > 1
        units.append((n1 - 1 if causal_short else n1, n1))
    bars = make_bars()
    sim = Sim(rng, bars)
    sim.run([(producer(bars, units, rng, skip), 'producer'),
             (mma(bars, units, skip), 'mma'),
             (softmax(bars, units, 0, rng, skip), 'softmax0'),
             (softmax(bars, units, 1, rng, skip), 'softmax1')])
    sim.check_races()
    return units


def test_pipeline_protocol_holds_under_random_timing():
    for seed in range(400):
        simulate(seed)


@pytest.mark.parametrize("skip,where", [
    # PV0 reading P0 before the softmax wrote it; the MMA thread then also
    # runs two phases ahead of tile 0's S and O waits
    (('p_full',), ('SP0', 'p_full0', 's_full0', 'o_full0')),
    (('kv_empty',), ('K', 'V', 'kv_full')),      # K/V copied over slots still being read
    (('release_early',), ('K', 'V', 'kv_full')),  # a group released before its readers ran
    (('q_empty_early',), ('Q', 'q_full')),        # Q released before the last S MMA is issued
])
def test_planted_mistake_is_caught(skip, where):
    caught = 0
    for seed in range(400):
        try:
            simulate(seed, skip)
        except Violation as e:
            assert any(w in str(e) for w in where), str(e)
            caught += 1
    assert caught > 0


# ---------------------------------------------------------------- D = 64
#
# Single slots: K_j and V_j each in a slot of an eight-slot ring with its own
# full and empty barriers, released by MMA commits (K_j after S1(j), V_j
# after PV1(j)); the softmax warps release nothing.

STAGES = 8


def make_bars_d64():
    B = Barrier
    bars = {'q_full': B('q_full', 1), 'q_empty': B('q_empty', 1)}
    for i in range(STAGES):
        bars[f'kv_full{i}'] = B(f'kv_full{i}', 1)
        bars[f'kv_empty{i}'] = B(f'kv_empty{i}', 1)
    for t in range(2):
        bars[f's_full{t}'] = B(f's_full{t}', 1)
        bars[f'p_full{t}'] = B(f'p_full{t}', 1)
        bars[f'o_full{t}'] = B(f'o_full{t}', 1)
    return bars


def producer_d64(b, units, rng):
    ring = 0
    f = rng.uniform(0.1, 5.0)
    for u, (n0, n1) in enumerate(units):
        yield ('wait', b['q_empty'], (u & 1) ^ 1, u - 1)
        yield ('arrive_tx', b['q_full'], 1)
        yield ('tma', b['q_full'], 1, 'Q', u)
        for j in range(n1):
            for _ in ('K', 'V'):
                sl, use = ring % STAGES, ring // STAGES
                yield ('wait', b[f'kv_empty{sl}'], (use & 1) ^ 1, use - 1)
                yield ('arrive_tx', b[f'kv_full{sl}'], 1)
                yield ('tma', b[f'kv_full{sl}'], 1, f'slot{sl}', use)
                yield ('delay', f * rng.uniform(0, 30))
                ring += 1


def mma_d64(b, units, skip=()):
    ring = 0
    jj = [0, 0]
    for u, (n0, n1) in enumerate(units):
        yield ('wait', b['q_full'], u & 1, u)
        ks, kuse = ring % STAGES, ring // STAGES
        yield ('wait', b[f'kv_full{ks}'], kuse & 1, kuse)
        ring += 1
        yield ('mma', [('Q', u), (f'slot{ks}', kuse)], [('SP0', 2 * jj[0])])
        yield ('commit', b['s_full0'])
        yield ('mma', [('Q', u), (f'slot{ks}', kuse)], [('SP1', 2 * jj[1])])
        yield ('commit', b['s_full1'])
        yield ('commit', b[f'kv_empty{ks}'])
        if n1 == 1:
            yield ('commit', b['q_empty'])
        for j in range(n1):
            vs, vuse = ring % STAGES, ring // STAGES
            yield ('wait', b[f'kv_full{vs}'], vuse & 1, vuse)
            ring += 1
            has_next = j + 1 < n1
            if has_next:
                ns, nuse = ring % STAGES, ring // STAGES
                ring += 1
            next_ready = False
            if j < n0:
                yield ('wait', b['p_full0'], jj[0] & 1, jj[0])
                yield ('mma', [('SP0', 2 * jj[0] + 1), (f'slot{vs}', vuse)], [('O0', (u, 2 * j))])
                jj[0] += 1
                if j + 1 < n0:
                    yield ('wait', b[f'kv_full{ns}'], nuse & 1, nuse)
                    next_ready = True
                    yield ('mma', [('Q', u), (f'slot{ns}', nuse)], [('SP0', 2 * jj[0])])
                    yield ('commit', b['s_full0'])
                else:
                    yield ('commit', b['o_full0'])
            if 'v_release_early' in skip:
                yield ('commit', b[f'kv_empty{vs}'])  # planted: before PV1(j) reads V_j
            yield ('wait', b['p_full1'], jj[1] & 1, jj[1])
            yield ('mma', [('SP1', 2 * jj[1] + 1), (f'slot{vs}', vuse)], [('O1', (u, 2 * j))])
            jj[1] += 1
            if 'v_release_early' not in skip:
                yield ('commit', b[f'kv_empty{vs}'])
            if has_next:
                if not next_ready:
                    yield ('wait', b[f'kv_full{ns}'], nuse & 1, nuse)
                yield ('mma', [('Q', u), (f'slot{ns}', nuse)], [('SP1', 2 * jj[1])])
                yield ('commit', b['s_full1'])
                yield ('commit', b[f'kv_empty{ns}'])
                if j + 2 == n1:
                    yield ('commit', b['q_empty'])
            else:
                yield ('commit', b['o_full1'])


def simulate_d64(seed, skip=()):
    rng = random.Random(seed)
    units = []
    for _ in range(rng.randint(1, 6)):
        n1 = rng.randint(1, 7)
        units.append((n1 - 1 if (rng.random() < 0.5 and n1 > 1) else n1, n1))
    bars = make_bars_d64()
    sim = Sim(rng, bars)
    sim.run([(producer_d64(bars, units, rng), 'producer'),
             (mma_d64(bars, units, skip), 'mma'),
             (softmax(bars, units, 0, rng, skip, grouped=False), 'softmax0'),
             (softmax(bars, units, 1, rng, skip, grouped=False), 'softmax1')])
    sim.check_races()
    return units


def test_d64_pipeline_protocol_holds_under_random_timing():
    for seed in range(400):
        simulate_d64(seed)


def test_d64_planted_mistake_is_caught():
    # V_j's slot released before PV1(j) has read it
    caught = 0
    for seed in range(400):
        try:
            simulate_d64(seed, ('v_release_early',))
        except Violation as e:
            assert 'slot' in str(e) or 'kv_full' in str(e), str(e)
            caught += 1
    assert caught > 0


# ---------------------------------------------------------------- D = 256

HALF_SLOTS = 5  # the ring of 32 KB half-slots: K head-dim halves, V key halves


def make_bars_d256():
    B = Barrier
    bars = {'q_full': B('q_full', 1), 'q_empty': B('q_empty', 1),
            'o_full': B('o_full', 1), 'pv_done': B('pv_done', 1)}
    for i in range(HALF_SLOTS):
        bars[f'hs_full{i}'] = B(f'hs_full{i}', 1)
        bars[f'hs_empty{i}'] = B(f'hs_empty{i}', 1)
    for buf in range(2):
        bars[f's_full{buf}'] = B(f's_full{buf}', 1)
        bars[f'p_full{buf}'] = B(f'p_full{buf}', 1)
    return bars


def producer_d256(b, units, rng, skip=()):
    """Q, then K_0's halves, then per key tile j: K_j+1's halves (if any) and
    V_j's halves: load r goes to half-slot r % 5."""
    ring = [0]
    f = rng.uniform(0.1, 5.0)

    def load_half(what):  # what: 'K' or 'V' (the slot is the same either way)
        hs, use = ring[0] % HALF_SLOTS, ring[0] // HALF_SLOTS
        if 'hs_empty' not in skip:
            yield ('wait', b[f'hs_empty{hs}'], (use & 1) ^ 1, use - 1)
        yield ('arrive_tx', b[f'hs_full{hs}'], 1)
        yield ('tma', b[f'hs_full{hs}'], 1, f'HS{hs}', use)
        yield ('delay', f * rng.uniform(0, 30))
        ring[0] += 1

    for u, n in enumerate(units):
        yield ('wait', b['q_empty'], (u & 1) ^ 1, u - 1)
        yield ('arrive_tx', b['q_full'], 1)
        yield ('tma', b['q_full'], 1, 'Q', u)
        yield from load_half('K')
        yield from load_half('K')
        for j in range(n):
            if j + 1 < n:
                yield from load_half('K')
                yield from load_half('K')
            yield from load_half('V')
            yield from load_half('V')


def mma_d256(b, units, skip=()):
    """S(j+1) into the other S buffer as soon as K_j+1 is in, then [P(j)] PV(j);
    tile g (over the CTA's units) uses S buffer g & 1."""
    kc = [0]
    g = 0

    def next_half():
        hs, use = kc[0] % HALF_SLOTS, kc[0] // HALF_SLOTS
        yield ('wait', b[f'hs_full{hs}'], use & 1, use)
        kc[0] += 1
        return (f'HS{hs}', use), hs

    def issue_s(buf, gg, u):
        for _ in range(2):
            res, hs = yield from next_half()
            yield ('mma', [('Q', u), res], [(f'SB{buf}', 2 * (gg >> 1))])
            yield ('commit', b[f'hs_empty{hs}'])
        yield ('commit', b[f's_full{buf}'])

    for u, n in enumerate(units):
        yield ('wait', b['q_full'], u & 1, u)
        yield from issue_s(g & 1, g, u)
        if n == 1:
            yield ('commit', b['q_empty'])
        for j in range(n):
            if j + 1 < n:
                yield from issue_s((g + 1) & 1, g + 1, u)
                if j + 2 == n:
                    yield ('commit', b['q_empty'])  # the last S MMA
            yield ('wait', b[f'p_full{g & 1}'], (g >> 1) & 1, g >> 1)
            for _ in range(2):
                res, hs = yield from next_half()
                yield ('mma', [(f'SB{g & 1}', 2 * (g >> 1) + 1), res], [('O', (u, 2 * j))])
                yield ('commit', b[f'hs_empty{hs}'])
            yield ('commit', b['pv_done'])
            if j + 1 == n:
                yield ('commit', b['o_full'])
            g += 1


def softmax_d256(b, units, rng, skip=()):
    f = rng.uniform(0.1, 5.0)
    g = 0
    for u, n in enumerate(units):
        for j in range(n):
            buf = g & 1
            yield ('wait', b[f's_full{buf}'], (g >> 1) & 1, g >> 1)
            yield ('ld', f'SB{buf}', 2 * (g >> 1))
            if j > 0 and rng.random() < 0.3:
                # rescale: S(j) was issued before PV(j-1), so wait for that PV
                if 'pv_done' not in skip:
                    yield ('wait', b['pv_done'], (g - 1) & 1, g - 1)
                yield ('ld', 'O', (u, 2 * j - 2))
                yield ('st', 'O', (u, 2 * j - 1))
            yield ('delay', f * rng.uniform(300, 1500))
            yield ('st', f'SB{buf}', 2 * (g >> 1) + 1)
            yield ('arrive', b[f'p_full{buf}'])
            g += 1
        yield ('wait', b['o_full'], u & 1, u)
        yield ('ld', 'O', (u, 2 * (n - 1)))
        yield ('delay', f * rng.uniform(200, 3000))  # direct stores, LSE


def simulate_d256(seed, skip=()):
    rng = random.Random(seed)
    units = [rng.randint(1, 7) for _ in range(rng.randint(1, 6))]
    bars = make_bars_d256()
    sim = Sim(rng, bars)
    sim.run([(producer_d256(bars, units, rng, skip), 'producer'),
             (mma_d256(bars, units, skip), 'mma'),
             (softmax_d256(bars, units, rng, skip), 'softmax')])
    sim.check_races()
    return units


def test_d256_pipeline_protocol_holds_under_random_timing():
    for seed in range(400):
        simulate_d256(seed)


@pytest.mark.parametrize("skip,where", [
    (('pv_done',), ('O',)),             # rescale of O racing PV(j-1), issued after S(j)
    (('hs_empty',), ('HS', 'hs_full')),  # a half-slot refilled while an MMA reads it
])
def test_d256_planted_mistake_is_caught(skip, where):
    caught = 0
    for seed in range(400):
        try:
            simulate_d256(seed, skip)
        except Violation as e:
            assert any(w in str(e) for w in where), str(e)
            caught += 1
    assert caught > 0
