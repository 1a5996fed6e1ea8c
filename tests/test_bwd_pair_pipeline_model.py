"""CPU model of the D = 256 CTA-pair backward's protocol (no GPU).

A cluster of two CTAs works on one 128-key tile with all 256 head-dim
columns, split by role:

  rank 0  S^T (K, Q in two stages, -LSE rows), P^T into TMEM, dV, and dQ^T
          for d in [0, 128) from dS^T that rank 1 sends back;
  rank 1  dP^T (V, dO, -Delta rows) into two TMEM stages, dS^T = P^T o dP^T
          with P^T that rank 0 sends, dK, and dQ^T for d in [128, 256).

Each rank has a producer, an MMA-issuing thread on its own tensor pipe,
four P^T (rank 0) or dS^T (rank 1) warps and four drain warps.  Each
P/dS warp sends its 32 key rows to the other CTA as one bulk copy that
completes on the receiver's barrier, after arming it remotely; a receiver
frees a buffer with a remote arrive once its values have been used.  Rank 0
issues each block's dQ^T one block late.  Queries stream in blocks of 64.

The model restates every role of both ranks in the kernel's order (waits
with the kernel's parity expressions, local and remote arrives, copies, MMAs
and commits) and checks, under random durations, that every role finishes,
that every parity wait sees exactly its phase, and that no buffer on either
CTA (K, V, Q, dO, the bias rows, the P^T and dS^T buffers of both sides, the
TMEM stages and accumulators) is written while a previous use still reads it.
Planted mistakes must be caught.
"""
import random

import pytest

from tests._pipeline_sim import Barrier, Sim, Violation

W = 4  # P/dS warps and drain warps per CTA


def make_bars():
    B = Barrier
    bars = {}
    for r in range(2):
        def add(name, count):
            bars[f'{r}.{name}'] = B(f'{r}.{name}', count)
        add('KvFull', 1)
        add('KvEmpty', 1)
        for st in range(2):
            add(f'QFull{st}', 2 if r == 0 else 1)  # rank 0: TMA + -LSE rows
            add(f'QEmpty{st}', 1)
            add(f'XFull{st}', 1)
            add(f'PReady{st}', W)
            add(f'DsrFull{st}', W)  # rank 0: dS^T landed (4 remote expect_tx + bytes)
            add(f'DsrFree{st}', 1)  # rank 1: rank 0's dS^T stage free (remote)
        add('DoFull', 1 if r == 0 else 2)  # rank 1: TMA + -Delta rows
        add('DoEmpty', 1)
        for q in range(W):
            add(f'PrFree{q}', 1)  # rank 0: rank 1's warp q has used its P^T rows
            add(f'PrFull{q}', 1)  # rank 1: P^T rows of warp q landed
        add('DsStaged', W)
        add('DsFree', 1)
        add('DqFull', 1)
        add('DqEmpty', W)
        add('AccFull', 1)
        add('AccEmpty', W)
    return bars


def producer(b, r, units, rng):
    f = rng.uniform(0.1, 5.0)
    nq = ndo = 0

    def load_q():
        nonlocal nq
        st, use = (nq & 1, nq >> 1) if r == 0 else (0, nq)
        yield ('delay', f * rng.uniform(0, 50))
        yield ('wait', b[f'{r}.QEmpty{st}'], (use & 1) ^ 1, use - 1)
        yield ('arrive_tx', b[f'{r}.QFull{st}'], 1)
        yield ('tma', b[f'{r}.QFull{st}'], 1, f'{r}.Q{st}', use)
        if r == 0:
            yield ('delay', f * rng.uniform(0, 1500))  # -LSE loads
            yield ('st', f'0.Lb{st}', use)
            yield ('arrive', b[f'0.QFull{st}'])
        nq += 1

    def load_do():
        nonlocal ndo
        yield ('delay', f * rng.uniform(0, 50))
        yield ('wait', b[f'{r}.DoEmpty'], (ndo & 1) ^ 1, ndo - 1)
        yield ('arrive_tx', b[f'{r}.DoFull'], 1)
        yield ('tma', b[f'{r}.DoFull'], 1, f'{r}.dO', ndo)
        if r == 1:
            yield ('delay', f * rng.uniform(0, 1500))  # -Delta loads
            yield ('st', '1.Db', ndo)
            yield ('arrive', b['1.DoFull'])
        ndo += 1

    for u, nb in enumerate(units):
        yield ('wait', b[f'{r}.KvEmpty'], (u & 1) ^ 1, u - 1)
        yield ('arrive_tx', b[f'{r}.KvFull'], 1)
        yield ('tma', b[f'{r}.KvFull'], 1, f'{r}.KV', u)
        if r == 0:  # Q one block ahead of dO (S^T is issued a block early)
            yield from load_q()
            for i in range(nb):
                if i + 1 < nb:
                    yield from load_q()
                yield from load_do()
        else:       # dO one block ahead of Q (dP^T is issued a block early)
            yield from load_do()
            for i in range(nb):
                if i + 1 < nb:
                    yield from load_do()
                yield from load_q()


def mma(b, r, units, skip=()):
    pipe = r
    n = 0

    def X(st, m, part):  # TMEM stage st, its m-th use: part 0 S^T / dP^T, 1 P^T
        return [(f'{r}.X{st}q{q}', 2 * m + part) for q in range(W)]

    for u, nb in enumerate(units):
        yield ('wait', b[f'{r}.KvFull'], u & 1, u)
        if r == 0:
            def issue_s(nb_):
                st = nb_ & 1
                yield ('wait', b[f'0.QFull{st}'], (nb_ >> 1) & 1, nb_ >> 1)
                yield ('mma', [('0.KV', u), (f'0.Q{st}', nb_ >> 1), (f'0.Lb{st}', nb_ >> 1)],
                       X(st, nb_ >> 1, 0), pipe)
                yield ('commit', b[f'0.XFull{st}'], pipe)
                yield ('commit', b[f'0.QEmpty{st}'], pipe)

            def issue_dq0(nb_):
                st = nb_ & 1
                yield ('wait', b[f'0.DsrFull{st}'], (nb_ >> 1) & 1, nb_ >> 1)
                if nb_ > 0 and 'dq_empty' not in skip:
                    yield ('wait', b['0.DqEmpty'], (nb_ - 1) & 1, nb_ - 1)
                yield ('mma', [('0.KV', u)] + [(f'0.DSR{st}q{q}', nb_ >> 1) for q in range(W)],
                       [('0.TdQ', nb_)], pipe)
                yield ('commit', b['0.DqFull'], pipe)

            yield from issue_s(n)
            for i in range(nb):
                st = n & 1
                first = i == 0
                if i + 1 < nb:
                    yield from issue_s(n + 1)
                yield ('wait', b[f'0.PReady{st}'], (n >> 1) & 1, n >> 1)
                if first and u > 0:
                    yield ('wait', b['0.AccEmpty'], (u - 1) & 1, u - 1)
                yield ('wait', b['0.DoFull'], n & 1, n)
                yield ('mma', X(st, n >> 1, 1) + [('0.dO', n)], [('0.Acc', u)], pipe)
                yield ('commit', b['0.DoEmpty'], pipe)
                if not first:
                    yield from issue_dq0(n - 1)
                n += 1
            yield from issue_dq0(n - 1)  # the unit's last block
        else:
            def issue_dp(nb_):
                yield ('wait', b['1.DoFull'], nb_ & 1, nb_)
                yield ('mma', [('1.KV', u), ('1.dO', nb_), ('1.Db', nb_)],
                       X(nb_ & 1, nb_ >> 1, 0), pipe)
                yield ('commit', b[f'1.XFull{nb_ & 1}'], pipe)
                yield ('commit', b['1.DoEmpty'], pipe)

            yield from issue_dp(n)
            for i in range(nb):
                first = i == 0
                if i + 1 < nb:
                    yield from issue_dp(n + 1)
                yield ('wait', b['1.DsStaged'], n & 1, n)
                if first and u > 0:
                    yield ('wait', b['1.AccEmpty'], (u - 1) & 1, u - 1)
                yield ('wait', b['1.QFull0'], n & 1, n)
                yield ('mma', [(f'1.DSL{q}', n) for q in range(W)] + [('1.Q0', n)],
                       [('1.Acc', u)], pipe)
                yield ('commit', b['1.QEmpty0'], pipe)
                if n > 0 and 'dq_empty' not in skip:
                    yield ('wait', b['1.DqEmpty'], (n - 1) & 1, n - 1)
                yield ('mma', [('1.KV', u)] + [(f'1.DSL{q}', n) for q in range(W)],
                       [('1.TdQ', n)], pipe)
                yield ('commit', b['1.DqFull'], pipe)
                n += 1
        yield ('commit', b[f'{r}.AccFull'], pipe)
        yield ('commit', b[f'{r}.KvEmpty'], pipe)


def pwarp(b, q, units, rng, skip=()):
    """Rank 0's P^T warp q: P^T into TMEM, then its rows to rank 1."""
    f = rng.uniform(0.1, 5.0)
    n = 0
    key = f'0.pcopy{q}'
    for nb in units:
        for _ in range(nb):
            st = n & 1
            yield ('wait', b[f'0.XFull{st}'], (n >> 1) & 1, n >> 1)
            yield ('ld', f'0.X{st}q{q}', 2 * (n >> 1))
            yield ('delay', f * rng.uniform(200, 1200))
            yield ('st', f'0.X{st}q{q}', 2 * (n >> 1) + 1)
            yield ('arrive', b[f'0.PReady{st}'])
            yield ('wait_read', key)  # the previous copy has read the staging rows
            yield ('st', f'0.PS{q}', n)
            if 'pr_free' not in skip:
                yield ('wait', b[f'0.PrFree{q}'], (n & 1) ^ 1, n - 1)
            yield ('arrive_tx', b[f'1.PrFull{q}'], 1)  # remote
            yield ('copy', b[f'1.PrFull{q}'], 1, f'0.PS{q}', n, f'1.PR{q}', n, key)
            n += 1


def dswarp(b, q, units, rng, skip=()):
    """Rank 1's dS^T warp q: dP^T from TMEM and P^T from rank 0 give dS^T,
    staged for the dK / dQ^T MMAs and sent to rank 0."""
    f = rng.uniform(0.1, 5.0)
    n = 0
    key = f'1.dscopy{q}'
    for nb in units:
        for _ in range(nb):
            st = n & 1
            yield ('wait', b[f'1.XFull{st}'], (n >> 1) & 1, n >> 1)
            yield ('ld', f'1.X{st}q{q}', 2 * (n >> 1))
            yield ('wait', b[f'1.PrFull{q}'], n & 1, n)
            if 'pr_free_early' in skip:
                yield ('arrive', b[f'0.PrFree{q}'])  # planted: released before the rows are read
            yield ('ld', f'1.PR{q}', n)
            if 'ds_free' not in skip:
                yield ('wait', b['1.DsFree'], (n & 1) ^ 1, n - 1)
            yield ('wait_read', key)
            yield ('delay', f * rng.uniform(100, 800))
            yield ('st', f'1.DSL{q}', n)
            if 'pr_free_early' not in skip:
                yield ('arrive', b[f'0.PrFree{q}'])  # remote: P^T rows used
            yield ('arrive', b['1.DsStaged'])
            yield ('wait', b[f'1.DsrFree{st}'], ((n >> 1) & 1) ^ 1, (n >> 1) - 1)
            yield ('arrive_tx', b[f'0.DsrFull{st}'], 1)  # remote
            yield ('copy', b[f'0.DsrFull{st}'], 1, f'1.DSL{q}', n, f'0.DSR{st}q{q}', n >> 1, key)
            n += 1


def drainwarp(b, r, q, units, rng):
    f = rng.uniform(0.1, 5.0)
    n = 0
    for u, nb in enumerate(units):
        for _ in range(nb):
            yield ('wait', b[f'{r}.DqFull'], n & 1, n)
            yield ('ld', f'{r}.TdQ', n)
            yield ('arrive', b[f'{r}.DqEmpty'])
            if q == 0:  # the signaller: this block's dS^T has been read
                if r == 0:
                    yield ('arrive', b[f'1.DsrFree{n & 1}'])  # remote
                else:
                    yield ('arrive', b['1.DsFree'])
            yield ('delay', f * rng.uniform(200, 2000))
            n += 1
        yield ('wait', b[f'{r}.AccFull'], u & 1, u)
        yield ('ld', f'{r}.Acc', u)
        yield ('arrive', b[f'{r}.AccEmpty'])
        yield ('delay', f * rng.uniform(200, 2000))


def simulate(seed, skip=()):
    rng = random.Random(seed)
    units = [rng.randint(1, 6) for _ in range(rng.randint(1, 6))]
    bars = make_bars()
    sim = Sim(rng, bars)
    procs = []
    for r in range(2):
        procs.append((producer(bars, r, units, rng), f'{r}.producer'))
        procs.append((mma(bars, r, units, skip), f'{r}.mma'))
        for q in range(W):
            procs.append((drainwarp(bars, r, q, units, rng), f'{r}.drain{q}'))
    for q in range(W):
        procs.append((pwarp(bars, q, units, rng, skip), f'0.p{q}'))
        procs.append((dswarp(bars, q, units, rng, skip), f'1.ds{q}'))
    sim.run(procs)
    sim.check_races()
    return units


def test_pair_protocol_holds_under_random_timing():
    for seed in range(250):
        simulate(seed)


@pytest.mark.parametrize("skip,where", [
    (('pr_free',), ('PR', 'PrFull')),            # P^T rows sent before rank 1 used the last ones
    # the receiver freeing the P^T rows when they land rather than once they
    # are read: a fault the GPU parity tests once caught in this kernel
    (('pr_free_early',), ('PR', 'PrFull')),
    (('ds_free',), ('DSL', 'DsFree')),           # dS^T restaged before the dK / dQ^T MMAs read it
    (('dq_empty',), ('TdQ', 'DqFull', 'DqEmpty')),  # dQ^T over the one the drain has not read
])
def test_pair_planted_mistake_is_caught(skip, where):
    caught = 0
    for seed in range(250):
        try:
            simulate(seed, skip)
        except Violation as e:
            assert any(w in str(e) for w in where), str(e)
            caught += 1
    assert caught > 0
