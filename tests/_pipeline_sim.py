"""Discrete-event simulator for the CPU models of the kernels' pipeline
protocols (test infrastructure).

Roles are Python generators that yield the actions of the kernel's threads:
mbarrier waits by phase parity, arrives (with expected transaction bytes),
TMA copies that land after a random latency, tensor-pipe MMAs that execute in
issue order, commits that arrive once every MMA issued before them has
completed, thread loads and stores, and delays.  The simulator runs them with
random durations and reports

  * a wait cycle (some role never finishes),
  * a parity wait that passes on the wrong phase or that its barrier has run
    two phases past (a parity cannot tell phase k from k + 2),
  * a buffer written while a previous use still reads it, or read before the
    write of its use has finished (every access names the buffer and its use;
    uses are ordered, and all accesses of use e must lie after the writes of
    use e and before the first write of the next use).
"""
import heapq


class Barrier:
    def __init__(self, name, count):
        self.name, self.count = name, count
        self.pend = 0     # arrivals in the current phase
        self.tx = 0       # bytes still expected in the current phase
        self.done = 0     # completed phases
        self.waiters = []


class Violation(AssertionError):
    pass


class Sim:
    """Discrete-event run of generator processes.  Actions a process yields:
    ('wait', bar, parity, k)       block until phase k of bar completed; the
                                   hardware test is done & 1 != parity
    ('arrive', bar) / ('arrive_tx', bar, n)
    ('tma', bar, n, res, use)      copy into res (use), n units of tx on landing
    ('mma', reads, writes[, pipe]) in-order tensor-pipe op, [(res, use)] lists
    ('commit', bar[, pipe])        arrive when every MMA issued so far to the
                                   pipe (one per SM) is done
    ('ld', res, use) / ('st', res, use)   a thread access
    ('delay', t)
    ('copy', bar, n, src, src_use, dst, dst_use, key)
                                   a bulk copy between shared memories (also
                                   to the other CTA of a pair): reads src and
                                   writes dst until it lands, then n units of
                                   tx complete on bar
    ('wait_read', key)             until the last copy issued under key has
                                   read its source (bulk wait_group.read)
    """

    def __init__(self, rng, bars):
        self.rng = rng
        # per-run scales, so that rare interleavings (a slow drain, a copy that
        # hits in L2, a slow tensor pipe) come up across seeds
        self.tma_lat = (rng.uniform(100, 1000), rng.uniform(1000, 5000))
        self.mma_scale = rng.uniform(0.3, 3.0)
        self.t = 0.0
        self.events = []
        self.seq = 0
        self.bars = bars
        self.pipe_free = {}  # tensor pipe (one per SM) -> when its last MMA ends
        self.acc = {}  # res -> list of (kind, use, start, end, who)
        self.blocked = {}
        self.copy_done = {}  # key -> when the last copy under key has read its source

    def at(self, t, fn):
        self.seq += 1
        heapq.heappush(self.events, (t, self.rng.random(), self.seq, fn))

    def record(self, res, kind, use, start, end, who):
        self.acc.setdefault(res, []).append((kind, use, start, end, who))

    def complete_check(self, b):
        if b.pend == b.count and b.tx == 0:
            b.done += 1
            b.pend = 0
            ws, b.waiters = b.waiters, []
            for w in ws:
                self.try_pass(*w)

    def arrive(self, b, tx=0):
        b.pend += 1
        b.tx += tx
        if b.pend > b.count:
            raise Violation(f"{b.name}: more arrivals than its count in one phase")
        self.complete_check(b)

    def try_pass(self, proc, b, parity, k, entered):
        if b.done >= k + 2:
            raise Violation(f"{b.name}: barrier two phases ahead of a waiter for phase {k}")
        if (b.done & 1) != parity:
            if b.done != k + 1:
                raise Violation(f"{b.name}: wait for phase {k} passed with {b.done} phases done")
            self.blocked.pop(proc, None)
            wake = 0.0 if self.t == entered else self.rng.uniform(50, 300)
            self.at(self.t + wake, lambda p=proc: self.step(p))
            return True
        b.waiters.append((proc, b, parity, k, entered))
        self.blocked[proc] = (b.name, k)
        return False

    def step(self, proc):
        gen, who = proc
        while True:
            try:
                a = next(gen)
            except StopIteration:
                return
            op = a[0]
            if op == 'wait':
                _, b, parity, k = a
                if not self.try_pass(proc, b, parity, k, self.t):
                    return
                return  # resumes from the scheduled wake-up
            if op == 'arrive':
                self.arrive(a[1])
            elif op == 'arrive_tx':
                self.arrive(a[1], a[2])
            elif op == 'tma':
                _, b, n, res, use = a
                land = self.t + self.rng.uniform(*self.tma_lat)
                self.record(res, 'w', use, self.t, land, who + ':tma')

                def landed(b=b, n=n):
                    b.tx -= n
                    self.complete_check(b)
                self.at(land, landed)
            elif op == 'mma':
                reads, writes = a[1], a[2]
                pipe = a[3] if len(a) > 3 else None
                start = max(self.t, self.pipe_free.get(pipe, 0.0))
                end = start + self.rng.uniform(200, 700) * self.mma_scale
                self.pipe_free[pipe] = end
                for res, use in reads:
                    self.record(res, 'r', use, start, end, who + ':mma')
                for res, use in writes:
                    self.record(res, 'w', use, start, end, who + ':mma')
                # issue returns when the pipe takes the MMA
                self.at(max(self.t, start) + self.rng.uniform(5, 60), lambda p=proc: self.step(p))
                return
            elif op == 'copy':
                _, b, n, src, src_use, dst, dst_use, key = a
                land = self.t + self.rng.uniform(*self.tma_lat) * 0.5
                self.record(src, 'r', src_use, self.t, land, who + ':copy')
                self.record(dst, 'w', dst_use, self.t, land, who + ':copy')
                self.copy_done[key] = land

                def copied(b=b, n=n):
                    b.tx -= n
                    self.complete_check(b)
                self.at(land, copied)
            elif op == 'wait_read':
                t_read = self.copy_done.get(a[1], self.t)
                if t_read > self.t:
                    self.at(t_read, lambda p=proc: self.step(p))
                    return
            elif op == 'commit':
                b = a[1]
                pipe = a[2] if len(a) > 2 else None
                self.at(max(self.t, self.pipe_free.get(pipe, 0.0)), lambda b=b: self.arrive(b))
            elif op in ('ld', 'st'):
                _, res, use = a
                d = self.rng.uniform(20, 200)
                self.record(res, 'r' if op == 'ld' else 'w', use, self.t, self.t + d, who)
                self.at(self.t + d, lambda p=proc: self.step(p))
                return
            elif op == 'delay':
                self.at(self.t + a[1], lambda p=proc: self.step(p))
                return
            else:
                raise ValueError(op)

    def run(self, procs):
        for p in procs:
            self.at(0.0, lambda p=p: self.step(p))
        while self.events:
            t, _, _, fn = heapq.heappop(self.events)
            self.t = t
            fn()
        if self.blocked:
            raise Violation(f"deadlock: {sorted(self.blocked.values())}")

    def check_races(self):
        for res, accs in self.acc.items():
            uses = sorted({u for _, u, _, _, _ in accs})
            by = {u: [a for a in accs if a[1] == u] for u in uses}
            for i, u in enumerate(uses):
                writes = [a for a in by[u] if a[0] == 'w']
                reads = [a for a in by[u] if a[0] == 'r']
                if reads and not writes:
                    raise Violation(f"{res} use {u}: read but never written")
                if writes and reads:
                    w_end = max(a[3] for a in writes)
                    r0 = min(reads, key=lambda a: a[2])
                    if r0[2] < w_end - 1e-9:
                        raise Violation(f"{res} use {u}: {r0[4]} reads before the write ends")
                if i + 1 < len(uses):
                    nxt = [a for a in by[uses[i + 1]] if a[0] == 'w']
                    if nxt:
                        w_start = min(a[2] for a in nxt)
                        last = max(by[u], key=lambda a: a[3])
                        if last[3] > w_start + 1e-9:
                            raise Violation(f"{res}: use {uses[i + 1]} written while use {u} "
                                            f"is still accessed ({last[4]})")
