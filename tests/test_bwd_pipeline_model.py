"""CPU model of the single-CTA backward kernel's pipeline protocol (no GPU).

The D = 64/128 backward runs four roles in one CTA: a producer (TMA copies of
K/V per unit, Q and dO per block, and the -LSE / -Delta rows the bias K steps
read), one MMA-issuing thread, the P/dS warps and the dQ-drain warps (which
also write each unit's dK and dV).  They hand buffers to each other through
mbarriers waited on by phase parity.  This module restates, role by role and
in the kernel's order, every wait (with the parity expression the kernel
uses), arrive, TMA copy, MMA and commit, and runs the roles against each other
in a discrete-event simulation with random durations.  It checks that

  * every role finishes (no wait cycle),
  * every wait that passes sees exactly the phase it is meant to see: a parity
    wait cannot tell phase k from phase k + 2, so a barrier two phases ahead of
    a waiter, or a waiter passing before its phase, is reported,
  * no buffer is overwritten while it is still read, and no buffer is read
    before it is written: for every buffer (shared-memory tiles and rows,
    TMEM regions, the dV/dK accumulators) and every use e of it, all accesses
    of use e lie after the writes of use e and before the first write of use
    e + 1.

tcgen05 MMAs from the one issuing thread execute in issue order; a commit
arrives once every MMA issued before it has completed.  Both producer orders
are covered: the unit's K/V copy first (fixed-order instance) and after the
first block's Q and dO copies (atomic order).  The D = 256 kernel (units of
one output half, 64-query blocks, Q in two head-dim halves) has a model of its
own below.  Planted mistakes (a wait left out, a release moved early) must be
caught, which shows the checks can fail; two waits of the P/dS warps (for dS
to have been read, and at D = 256 for the LSE/Delta rows) turned out to be
implied by other orderings, so leaving them out is not a mistake the model
can catch.
"""
import random

import pytest

from tests._pipeline_sim import Barrier, Sim, Violation


def make_bars():
    B = Barrier
    return {
        'kv_full': B('kv_full', 1), 'kv_empty': B('kv_empty', 1),
        'q_full0': B('q_full0', 2), 'q_full1': B('q_full1', 2),
        'q_empty0': B('q_empty0', 1), 'q_empty1': B('q_empty1', 1),
        'do_full': B('do_full', 2), 'do_empty': B('do_empty', 1),
        's_full': B('s_full', 1), 'dp_full': B('dp_full', 1),
        'p_ready': B('p_ready', 1), 'ds_ready': B('ds_ready', 1),
        'dq_full': B('dq_full', 1), 'dq_empty': B('dq_empty', 1),
        'dkdv_full': B('dkdv_full', 1), 'dv_empty': B('dv_empty', 1),
        'dk_empty': B('dk_empty', 1),
    }


def producer(bars, units, kv_first, rng, skip=()):
    b = bars
    f = rng.uniform(0.1, 5.0)
    n = 0
    for u, nb in enumerate(units):
        kv_par = (u & 1) ^ 1

        def load_kv(u=u, kv_par=kv_par):
            yield ('wait', b['kv_empty'], kv_par, u - 1)
            yield ('arrive_tx', b['kv_full'], 2)
            yield ('tma', b['kv_full'], 1, 'K', u)
            yield ('tma', b['kv_full'], 1, 'V', u)
        if kv_first:
            yield from load_kv()
        for i in range(nb):
            st = n & 1
            first = (i == 0) and not kv_first
            yield ('delay', f * rng.uniform(0, 50))  # the -LSE / -Delta loads are issued
            if 'q_empty' not in skip:
                yield ('wait', b[f'q_empty{st}'], ((n >> 1) & 1) ^ 1, (n >> 1) - 1)
            yield ('arrive_tx', b[f'q_full{st}'], 1)
            yield ('tma', b[f'q_full{st}'], 1, f'Q{st}', n >> 1)

            def q_rows(st=st, n=n):
                yield ('delay', f * rng.uniform(0, 1500))  # the loads' latency
                yield ('st', f'Lb{st}', n >> 1)
                yield ('arrive', b[f'q_full{st}'])
            if not first:
                yield from q_rows()
            yield ('wait', b['do_empty'], (n & 1) ^ 1, n - 1)
            yield ('arrive_tx', b['do_full'], 1)
            yield ('tma', b['do_full'], 1, 'dO', n)
            if first:
                yield from load_kv()
                yield from q_rows()
            yield ('st', 'Db', n)
            yield ('arrive', b['do_full'])
            n += 1


def mma(bars, units, skip=()):
    b = bars
    n = 0
    ph_p = ph_ds = ph_dqe = 0
    for u, nb in enumerate(units):
        yield ('wait', b['kv_full'], u & 1, u)
        st = n & 1
        yield ('wait', b[f'q_full{st}'], (n >> 1) & 1, n >> 1)
        yield ('mma', [('K', u), (f'Q{st}', n >> 1), (f'Lb{st}', n >> 1)], [('X', 2 * n)])
        yield ('commit', b['s_full'])
        if n > 0:
            yield ('wait', b['dq_empty'], ph_dqe, n - 1)
            ph_dqe ^= 1
        yield ('wait', b['do_full'], n & 1, n)
        yield ('mma', [('V', u), ('dO', n), ('Db', n)], [('Y', 2 * n)])
        yield ('commit', b['dp_full'])
        for i in range(nb):
            st = n & 1
            first, has_next = i == 0, i + 1 < nb
            yield ('wait', b['p_ready'], ph_p, n)
            ph_p ^= 1
            if first and u > 0 and 'dv_empty' not in skip:
                yield ('wait', b['dv_empty'], (u - 1) & 1, u - 1)
            yield ('mma', [('X', 2 * n + 1), ('dO', n)], [('dVacc', u)])
            yield ('commit', b['do_empty'])
            if has_next:
                st2 = (n + 1) & 1
                yield ('wait', b[f'q_full{st2}'], ((n + 1) >> 1) & 1, (n + 1) >> 1)
                yield ('mma', [('K', u), (f'Q{st2}', (n + 1) >> 1), (f'Lb{st2}', (n + 1) >> 1)],
                       [('X', 2 * n + 2)])
                yield ('commit', b['s_full'])
            yield ('wait', b['ds_ready'], ph_ds, n)
            ph_ds ^= 1
            yield ('mma', [('dS', n), ('K', u)], [('Y', 2 * n + 1)])
            yield ('commit', b['dq_full'])
            if first and u > 0 and 'dk_empty' not in skip:
                yield ('wait', b['dk_empty'], (u - 1) & 1, u - 1)
            yield ('mma', [('dS', n), (f'Q{st}', n >> 1)], [('dKacc', u)])
            yield ('commit', b[f'q_empty{st}'])
            if has_next:
                if 'dq_empty' not in skip:
                    yield ('wait', b['dq_empty'], ph_dqe, n)
                ph_dqe ^= 1
                yield ('wait', b['do_full'], (n + 1) & 1, n + 1)
                yield ('mma', [('V', u), ('dO', n + 1), ('Db', n + 1)], [('Y', 2 * n + 2)])
                yield ('commit', b['dp_full'])
            else:
                yield ('commit', b['dkdv_full'])
                yield ('commit', b['kv_empty'])
            n += 1


def softmax(bars, units, rng, skip=()):
    b = bars
    f = rng.uniform(0.1, 5.0)
    n = 0
    for nb in units:
        for _ in range(nb):
            yield ('wait', b['s_full'], n & 1, n)
            yield ('ld', 'X', 2 * n)
            yield ('delay', f * rng.uniform(300, 1500))
            yield ('st', 'X', 2 * n + 1)
            yield ('arrive', b['p_ready'])
            yield ('wait', b['dp_full'], n & 1, n)
            if n > 0:
                # the previous block's dQ and dK MMAs have read dS (also implied
                # by dp_full: dP(i) is issued after dK(i-1) and MMAs complete in
                # order)
                yield ('wait', b[f'q_empty{(n - 1) & 1}'], ((n - 1) >> 1) & 1, (n - 1) >> 1)
            yield ('ld', 'Y', 2 * n)
            yield ('delay', f * rng.uniform(100, 800))
            yield ('st', 'dS', n)
            yield ('arrive', b['ds_ready'])
            n += 1


def drain(bars, units, rng):
    b = bars
    f = rng.uniform(0.1, 5.0)
    n = 0
    for u, nb in enumerate(units):
        for _ in range(nb):
            yield ('wait', b['dq_full'], n & 1, n)
            yield ('ld', 'Y', 2 * n + 1)
            yield ('arrive', b['dq_empty'])
            yield ('delay', f * rng.uniform(200, 2000))  # staging and reductions
            n += 1
        yield ('wait', b['dkdv_full'], u & 1, u)
        yield ('ld', 'dVacc', u)
        yield ('arrive', b['dv_empty'])
        yield ('delay', f * rng.uniform(200, 2000))  # dV stores
        yield ('ld', 'dKacc', u)
        yield ('arrive', b['dk_empty'])
        yield ('delay', f * rng.uniform(200, 2000))  # dK stores


def simulate(seed, kv_first, skip=()):
    rng = random.Random(seed)
    units = [rng.randint(1, 5) for _ in range(rng.randint(1, 9))]
    bars = make_bars()
    sim = Sim(rng, bars)
    sim.run([(producer(bars, units, kv_first, rng, skip), 'producer'),
             (mma(bars, units, skip), 'mma'),
             (softmax(bars, units, rng, skip), 'softmax'),
             (drain(bars, units, rng), 'drain')])
    sim.check_races()
    return units


@pytest.mark.parametrize("kv_first", [False, True])
def test_pipeline_protocol_holds_under_random_timing(kv_first):
    for seed in range(300):
        simulate(seed, kv_first)


@pytest.mark.parametrize("skip,where", [
    (('dv_empty',), 'dVacc'),   # first dV of a unit not waiting for the dV epilogue's read
    (('dk_empty',), 'dKacc'),   # first dK likewise
    # dP(i+1) written over dQ(i) before the drain has read it; the MMA thread
    # can then also run two dQ phases ahead of the drain's parity wait, and its
    # later dq_empty waits see the wrong phase
    (('dq_empty',), ('Y', 'dq_full', 'dq_empty')),
    (('q_empty',), 'Q'),        # Q_i+2 copied over Q_i while dK(i) may still read it
])
def test_planted_missing_wait_is_caught(skip, where):
    caught = 0
    for seed in range(300):
        try:
            simulate(seed, False, skip)
        except Violation as e:
            wheres = where if isinstance(where, tuple) else (where,)
            assert any(w in str(e) for w in wheres), str(e)
            caught += 1
    assert caught > 0


# ---------------------------------------------------------------- D = 256
#
# A unit is (key tile, output half oh); queries stream in 64-row blocks.  Q
# comes in two head-dim halves with their own barriers (dK of half oh reads
# only Q half oh, so the other, "early" half is released once S^T is done and
# the next block's copy of it loads while dP, dV and dK run); LSE and Delta
# go through two shared-memory buffers by block parity.  The MMAs of a block
# run in order S^T (early half first), dP^T, dV, dK, dQ^T; TMEM X holds S^T
# then P^T, Y holds dP^T, then dS^T (written by the softmax warps), then dQ^T.


def make_bars_d256():
    B = Barrier
    bars = {}
    for name in ('kv_full', 'kv_empty', 'do_full', 'do_empty', 's_full', 'dp_full', 'p_ready',
                 'ds_ready', 'dq_full', 'dq_empty', 'dkdv_full', 'dkdv_empty'):
        bars[name] = B(name, 1)
    for i in range(2):
        bars[f'qh_full{i}'] = B(f'qh_full{i}', 1)
        bars[f'qh_empty{i}'] = B(f'qh_empty{i}', 1)
        bars[f'st_full{i}'] = B(f'st_full{i}', 1)
    return bars


def producer_d256(b, units, rng):
    f = rng.uniform(0.1, 5.0)
    n = 0
    for u, (nb, oh) in enumerate(units):
        yield ('wait', b['kv_empty'], (u & 1) ^ 1, u - 1)
        yield ('arrive_tx', b['kv_full'], 2)
        yield ('tma', b['kv_full'], 1, 'K', u)
        yield ('tma', b['kv_full'], 1, 'V', u)
        eh, lh = 1 - oh, oh
        for _ in range(nb):
            yield ('delay', f * rng.uniform(0, 50))  # LSE / Delta loads issued

            def load_q_half(hs, n=n):
                yield ('wait', b[f'qh_empty{hs}'], (n & 1) ^ 1, n - 1)
                yield ('arrive_tx', b[f'qh_full{hs}'], 1)
                yield ('tma', b[f'qh_full{hs}'], 1, f'Qh{hs}', n)
            yield from load_q_half(eh)
            yield ('delay', f * rng.uniform(0, 1500))  # the loads' latency
            # buffer n & 1 was last read by the softmax of block n-2, whose dS
            # preceded dQ^T(n-2) and so S^T(n-1), whose first half's release
            # (or a later one) the early-half wait above has seen
            yield ('st', f'ST{n & 1}', n >> 1)
            yield ('arrive', b[f'st_full{n & 1}'])
            yield ('wait', b['do_empty'], (n & 1) ^ 1, n - 1)
            yield ('arrive_tx', b['do_full'], 1)
            yield ('tma', b['do_full'], 1, 'dO', n)
            yield from load_q_half(lh)
            n += 1


def mma_d256(b, units, skip=()):
    n = 0
    for u, (nb, oh) in enumerate(units):
        yield ('wait', b['kv_full'], u & 1, u)
        eh, lh = 1 - oh, oh
        for i in range(nb):
            for g2 in range(2):
                hs = lh if g2 else eh
                if g2 == 0 and 'qh_early' in skip:
                    yield ('commit', b[f'qh_empty{eh}'])  # planted: before S^T reads it
                yield ('wait', b[f'qh_full{hs}'], n & 1, n)
                yield ('mma', [('K', u), (f'Qh{hs}', n)], [('X', 2 * n)])
                if g2 == 0 and 'qh_early' not in skip:
                    yield ('commit', b[f'qh_empty{eh}'])  # dK reads only half lh
            yield ('commit', b['s_full'])
            if n > 0 and 'dq_empty' not in skip:
                yield ('wait', b['dq_empty'], (n - 1) & 1, n - 1)
            yield ('wait', b['do_full'], n & 1, n)
            yield ('mma', [('V', u), ('dO', n)], [('Y', 3 * n)])
            yield ('commit', b['dp_full'])
            yield ('wait', b['p_ready'], n & 1, n)
            if i == 0 and u > 0 and 'dkdv_empty' not in skip:
                yield ('wait', b['dkdv_empty'], (u - 1) & 1, u - 1)
            yield ('mma', [('X', 2 * n + 1), ('dO', n)], [('dVacc', u)])
            yield ('commit', b['do_empty'])
            yield ('wait', b['ds_ready'], n & 1, n)
            yield ('mma', [('Y', 3 * n + 1), (f'Qh{lh}', n)], [('dKacc', u)])
            yield ('commit', b[f'qh_empty{lh}'])
            yield ('mma', [('K', u), ('dS', n)], [('Y', 3 * n + 2)])
            yield ('commit', b['dq_full'])
            if i + 1 == nb:
                yield ('commit', b['dkdv_full'])
                yield ('commit', b['kv_empty'])
            n += 1


def softmax_d256(b, units, rng, skip=()):
    f = rng.uniform(0.1, 5.0)
    n = 0
    for nb, _ in units:
        for _ in range(nb):
            # (also implied: the stats are written before the late Q half's
            # copy, which S^T waits for)
            yield ('wait', b[f'st_full{n & 1}'], (n >> 1) & 1, n >> 1)
            yield ('wait', b['s_full'], n & 1, n)
            yield ('ld', 'X', 2 * n)
            yield ('ld', f'ST{n & 1}', n >> 1)
            yield ('delay', f * rng.uniform(300, 1500))
            yield ('st', 'X', 2 * n + 1)
            yield ('arrive', b['p_ready'])
            yield ('wait', b['dp_full'], n & 1, n)
            if n > 0:
                # the dQ MMA of the previous block has read dS (also implied by
                # dp_full: dP^T(i) is issued after dQ^T(i-1))
                yield ('wait', b['dq_full'], (n - 1) & 1, n - 1)
            yield ('ld', 'Y', 3 * n)
            yield ('ld', f'ST{n & 1}', n >> 1)
            yield ('delay', f * rng.uniform(100, 800))
            yield ('st', 'Y', 3 * n + 1)
            yield ('st', 'dS', n)
            yield ('arrive', b['ds_ready'])
            n += 1


def drain_d256(b, units, rng):
    f = rng.uniform(0.1, 5.0)
    n = 0
    for u, (nb, _) in enumerate(units):
        for _ in range(nb):
            yield ('wait', b['dq_full'], n & 1, n)
            yield ('ld', 'Y', 3 * n + 2)
            yield ('arrive', b['dq_empty'])
            yield ('delay', f * rng.uniform(200, 2000))  # staging and reductions
            n += 1
        yield ('wait', b['dkdv_full'], u & 1, u)
        yield ('ld', 'dVacc', u)
        yield ('ld', 'dKacc', u)
        yield ('arrive', b['dkdv_empty'])
        yield ('delay', f * rng.uniform(200, 3000))  # stores


def simulate_d256(seed, skip=()):
    rng = random.Random(seed)
    units = [(rng.randint(1, 6), rng.randint(0, 1)) for _ in range(rng.randint(1, 8))]
    bars = make_bars_d256()
    sim = Sim(rng, bars)
    sim.run([(producer_d256(bars, units, rng), 'producer'),
             (mma_d256(bars, units, skip), 'mma'),
             (softmax_d256(bars, units, rng, skip), 'softmax'),
             (drain_d256(bars, units, rng), 'drain')])
    sim.check_races()
    return units


def test_d256_pipeline_protocol_holds_under_random_timing():
    for seed in range(400):
        simulate_d256(seed)


@pytest.mark.parametrize("skip,where", [
    (('dq_empty',), ('Y', 'dq_full', 'dq_empty')),      # dP^T over dQ^T before the drain read it
    (('qh_early',), ('Qh', 'qh_full')),                 # early Q half released before S^T read it
    (('dkdv_empty',), ('dVacc', 'dKacc', 'dkdv_full')),  # next unit's dV over the unread accumulator
])
def test_d256_planted_missing_wait_is_caught(skip, where):
    caught = 0
    for seed in range(400):
        try:
            simulate_d256(seed, skip)
        except Violation as e:
            assert any(w in str(e) for w in where), str(e)
            caught += 1
    assert caught > 0
