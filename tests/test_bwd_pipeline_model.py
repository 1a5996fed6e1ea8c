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
first block's Q and dO copies (atomic order).  Planted mistakes (a wait left
out) must be caught, which shows the checks can fail.
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
