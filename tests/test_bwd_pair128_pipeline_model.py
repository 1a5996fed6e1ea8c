"""CPU model of the D = 128 CTA-pair backward's protocol (no GPU).

A cluster of two CTAs owns a pair of key tiles (CTA r holds tile 2p + r);
both stream the same 128-query blocks.  One thread of CTA 0 issues every MMA
for the pair (tcgen05 .cta_group::2): each MMA reads operands from both CTAs'
shared memory and Tensor Memory and writes both CTAs' Tensor Memory, and each
commit arrives on the barrier of the same slot in both CTAs.  The issuer
waits on its own CTA's "copy landed" barriers and on CTA 0 barriers that a
relay thread of CTA 1 arrives on once CTA 1's copies have landed.  The P^T /
dS^T warps and drain warps of both CTAs arrive on CTA 0's barriers (eight
arrivals).  For dQ each CTA's softmax stages the other CTA's half of dS and
sends it as one bulk copy that completes on the receiver's barrier, which its
own copier thread arms; CTA 1's dS relay forwards that completion to CTA 0.

TMEM per CTA: X holds S^T then P^T; Y holds dP^T, then dS^T in its first 64
columns (the dK MMA's A operand) while dQ lands in its other 64 columns.

The model restates every role of both CTAs in the kernel's order and checks,
under random durations, that every role finishes, that every parity wait sees
exactly its phase, and that no buffer of either CTA is written while a
previous use still reads it.  Planted mistakes must be caught.
"""
import random

import pytest

from tests._pipeline_sim import Barrier, Sim, Violation

W = 4  # P/dS warps and drain warps per CTA
LOADS = ('Qs', 'DOs', 'DOd', 'Qd')  # per-block copies: S^T's B, dP^T's B, dV's B, dK's B


def make_bars():
    B = Barrier
    bars = {}
    for r in range(2):
        def add(name, count):
            bars[f'{r}.{name}'] = B(f'{r}.{name}', count)
        add('KvFull', 1)
        add('KvEmpty', 1)
        for x in LOADS:
            add(f'{x}Full', 2 if x == 'Qs' else 1)  # Qs: TMA + LSE/Delta written
            add(f'{x}Empty', 1)
            add(f'Pk{x}', 1)  # CTA 0: CTA 1's copy landed (relayed)
        add('PkKv', 1)
        add('SFull', 1)
        add('DpFull', 1)
        add('PReady', 2 * W)   # CTA 0's is used: eight warps of both CTAs
        add('DsReady', 2 * W)
        add('DqFull', 1)
        add('DqEmpty', 2 * W)
        add('DkdvFull', 1)
        add('DkdvEmpty', 2 * W)
        add('DsIn', 1)         # the other CTA's dS rows landed (armed by own copier)
        add('PkDs', 1)
        add('Staged', W)
    return bars


def both(name, use, quarters=False):
    """The resource on both CTAs (optionally per lane quarter)."""
    out = []
    for r in range(2):
        if quarters:
            out += [(f'{r}.{name}q{q}', use) for q in range(W)]
        else:
            out.append((f'{r}.{name}', use))
    return out


def producer(b, r, units, rng):
    f = rng.uniform(0.1, 5.0)
    n = 0
    for u, nb in enumerate(units):
        yield ('wait', b[f'{r}.KvEmpty'], (u & 1) ^ 1, u - 1)
        yield ('arrive_tx', b[f'{r}.KvFull'], 1)
        yield ('tma', b[f'{r}.KvFull'], 1, f'{r}.KV', u)
        for _ in range(nb):
            yield ('delay', f * rng.uniform(0, 50))
            yield ('wait', b[f'{r}.QsEmpty'], (n & 1) ^ 1, n - 1)
            yield ('arrive_tx', b[f'{r}.QsFull'], 1)
            yield ('tma', b[f'{r}.QsFull'], 1, f'{r}.Qs', n)
            # the stats stage was last read by the dS phase of block n - 2,
            # which finished before dK(n - 2), whose release the Qd wait of
            # block n - 1 saw
            yield ('delay', f * rng.uniform(0, 1500))
            yield ('st', f'{r}.ST{n & 1}', n >> 1)
            yield ('arrive', b[f'{r}.QsFull'])
            for x in ('DOs', 'DOd', 'Qd'):
                yield ('wait', b[f'{r}.{x}Empty'], (n & 1) ^ 1, n - 1)
                yield ('arrive_tx', b[f'{r}.{x}Full'], 1)
                yield ('tma', b[f'{r}.{x}Full'], 1, f'{r}.{x}', n)
            n += 1


def relay(b, units, skip=()):
    """CTA 1: forwards each of its landed copies to CTA 0, in load order."""
    n = 0
    for u, nb in enumerate(units):
        yield ('wait', b['1.KvFull'], u & 1, u)
        yield ('arrive', b['0.PkKv'])
        for _ in range(nb):
            for x in LOADS:
                if not ('relay_early' in skip and x == 'DOd'):
                    yield ('wait', b[f'1.{x}Full'], n & 1, n)
                yield ('arrive', b[f'0.Pk{x}'])
            n += 1


def ds_relay(b, units):
    n = 0
    for nb in units:
        for _ in range(nb):
            yield ('wait', b['1.DsIn'], n & 1, n)
            yield ('arrive', b['0.PkDs'])
            n += 1


def issuer(b, units, skip=()):
    n = 0

    def commit(slot):  # a pair commit arrives on the slot in both CTAs
        yield ('commit', b[f'0.{slot}'])
        yield ('commit', b[f'1.{slot}'])

    def wait_pair(x, k):  # own copy landed and CTA 1's (relayed)
        yield ('wait', b[f'0.{x}Full'], k & 1, k)
        yield ('wait', b[f'0.Pk{x}'], k & 1, k)

    def issue_s(k, u):
        yield ('mma', both('KV', u) + both('Qs', k) + both(f'ST{k & 1}', k >> 1),
               both('X', 2 * k, quarters=True))
        yield from commit('SFull')
        yield from commit('QsEmpty')

    def issue_dp(k, u):
        yield ('mma', both('KV', u) + both('DOs', k) + both(f'ST{k & 1}', k >> 1),
               both('Ylo', 2 * k, quarters=True) + both('Yhi', 2 * k, quarters=True))
        yield from commit('DpFull')
        yield from commit('DOsEmpty')

    for u, nb in enumerate(units):
        yield ('wait', b['0.KvFull'], u & 1, u)
        yield ('wait', b['0.PkKv'], u & 1, u)
        yield from wait_pair('Qs', n)
        yield from issue_s(n, u)
        if n > 0:
            yield ('wait', b['0.DqEmpty'], (n - 1) & 1, n - 1)
        yield from wait_pair('DOs', n)
        yield from issue_dp(n, u)
        for i in range(nb):
            first, has_next = i == 0, i + 1 < nb
            yield ('wait', b['0.PReady'], n & 1, n)
            if first and u > 0:
                yield ('wait', b['0.DkdvEmpty'], (u - 1) & 1, u - 1)
            yield from wait_pair('DOd', n)
            yield ('mma', both('X', 2 * n + 1, quarters=True) + both('DOd', n), both('dV', u))
            yield from commit('DOdEmpty')
            if has_next:
                yield from wait_pair('Qs', n + 1)
                yield from issue_s(n + 1, u)
            yield ('wait', b['0.DsReady'], n & 1, n)
            yield from wait_pair('Qd', n)
            yield ('mma', both('Ylo', 2 * n + 1, quarters=True) + both('Qd', n), both('dK', u))
            yield from commit('QdEmpty')
            if 'ds_in' not in skip:
                yield ('wait', b['0.DsIn'], n & 1, n)
                yield ('wait', b['0.PkDs'], n & 1, n)
            yield ('mma', both('DSo', n) + both('DSi', n) + both('KV', u),
                   both('Yhi', 2 * n + 1, quarters=True))
            yield from commit('DqFull')
            if has_next:
                if 'dq_empty' not in skip:
                    yield ('wait', b['0.DqEmpty'], n & 1, n)
                yield from wait_pair('DOs', n + 1)
                yield from issue_dp(n + 1, u)
            else:
                yield from commit('DkdvFull')
                yield from commit('KvEmpty')
            n += 1


def softmax_warp(b, r, q, units, rng, skip=()):
    f = rng.uniform(0.1, 5.0)
    peer = r ^ 1
    copier = q == 0
    n = 0
    for nb in units:
        for _ in range(nb):
            yield ('wait', b[f'{r}.QsFull'], n & 1, n)  # the block's LSE / Delta
            yield ('wait', b[f'{r}.SFull'], n & 1, n)
            yield ('ld', f'{r}.Xq{q}', 2 * n)
            yield ('ld', f'{r}.ST{n & 1}', n >> 1)
            yield ('delay', f * rng.uniform(300, 1500))
            yield ('st', f'{r}.Xq{q}', 2 * n + 1)
            yield ('arrive', b['0.PReady'])
            yield ('wait', b[f'{r}.DpFull'], n & 1, n)
            if n > 0:
                # the previous dQ MMA has read both CTAs' dS (and so the copies
                # of the outgoing halves have landed); also implied by DpFull:
                # dP^T(i) is issued after dQ(i-1)
                yield ('wait', b[f'{r}.DqFull'], (n - 1) & 1, n - 1)
            yield ('ld', f'{r}.Yloq{q}', 2 * n)
            yield ('ld', f'{r}.Yhiq{q}', 2 * n)
            yield ('delay', f * rng.uniform(100, 800))
            yield ('st', f'{r}.Yloq{q}', 2 * n + 1)   # dS^T for the dK MMA
            yield ('st', f'{r}.DSo', n)                # own half of the dQ operand
            yield ('st', f'{r}.DSx', n)                # the other CTA's half, outgoing
            yield ('arrive', b[f'{r}.Staged'])
            if copier:
                yield ('wait', b[f'{r}.Staged'], n & 1, n)
                yield ('arrive_tx', b[f'{r}.DsIn'], 1)  # the other CTA's half comes in
                yield ('copy', b[f'{peer}.DsIn'], 1, f'{r}.DSx', n, f'{peer}.DSi', n, f'{r}.dscopy')
            yield ('arrive', b['0.DsReady'])
            n += 1


def drain_warp(b, r, q, units, rng):
    f = rng.uniform(0.1, 5.0)
    n = 0
    for u, nb in enumerate(units):
        for _ in range(nb):
            yield ('wait', b[f'{r}.DqFull'], n & 1, n)
            yield ('ld', f'{r}.Yhiq{q}', 2 * n + 1)
            yield ('arrive', b['0.DqEmpty'])
            yield ('delay', f * rng.uniform(200, 2000))
            n += 1
        yield ('wait', b[f'{r}.DkdvFull'], u & 1, u)
        yield ('ld', f'{r}.dV', u)
        yield ('ld', f'{r}.dK', u)
        yield ('arrive', b['0.DkdvEmpty'])
        yield ('delay', f * rng.uniform(200, 2000))


def simulate(seed, skip=()):
    rng = random.Random(seed)
    units = [rng.randint(1, 5) for _ in range(rng.randint(1, 6))]
    bars = make_bars()
    sim = Sim(rng, bars)
    procs = [(issuer(bars, units, skip), '0.mma'), (relay(bars, units, skip), '1.relay'),
             (ds_relay(bars, units), '1.dsrelay')]
    for r in range(2):
        procs.append((producer(bars, r, units, rng), f'{r}.producer'))
        for q in range(W):
            procs.append((softmax_warp(bars, r, q, units, rng, skip), f'{r}.sm{q}'))
            procs.append((drain_warp(bars, r, q, units, rng), f'{r}.drain{q}'))
    sim.run(procs)
    sim.check_races()
    return units


def test_pair128_protocol_holds_under_random_timing():
    for seed in range(250):
        simulate(seed)


@pytest.mark.parametrize("skip,where", [
    # dQ issued before the dS halves landed (their staging is then also
    # rewritten while the copy still reads it)
    (('ds_in',), ('DSi', 'DSx', 'DsIn', 'PkDs')),
    (('dq_empty',), ('Yhi', 'DqFull', 'DqEmpty')),      # dP^T over dQ the drains have not read
    (('relay_early',), ('DOd', 'DOdFull', 'PkDOd')),   # CTA 1's dO columns forwarded unlanded
])
def test_pair128_planted_mistake_is_caught(skip, where):
    caught = 0
    for seed in range(250):
        try:
            simulate(seed, skip)
        except Violation as e:
            assert any(w in str(e) for w in where), str(e)
            caught += 1
    assert caught > 0
