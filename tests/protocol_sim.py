"""Discrete-event engine for the host-side models of the tensor-core kernels'
synchronisation (tests/test_bwd_protocol.py, tests/test_fwd_protocol.py).

A role is a Python generator that yields steps: wait on a barrier for a named
phase, arrive, spend time, read or write buffer regions, issue an MMA to the
in-order tensor pipe, commit (arrive once every MMA issued so far has finished),
start a TMA load (writes its regions, then arrives on its barrier) or a bulk
reduce-add (reads its regions), and wait for older reduce-adds to have read their
sources.  Mbarriers keep their arrival counts and completed phases.  Every
access is recorded with its time interval; `run` reports deadlocks, barrier
phases overtaken before their wait, writes that overlap another access of the
same region, and reads that do not see the version they name.

A wait returns whether its phase completed (`ok = yield ("wait", ...)`).  With a
fault injected (`fault=(role, n)`: that role's n-th wait never completes) the
run takes the kernels' failure path: the failed wait sets the status word, and
from then on every wait that has lasted longer than the status-check interval
returns False, as the kernels' bounded waits do.  Such a run is checked for what
must hold even after a failure: every role ends, no asynchronous operation is
still running when the last role ends, and nothing touches tensor memory after
it is released (version checks are off: the results are flagged as failed)."""
import heapq
from collections import defaultdict


STATUS_CHECK = 100_000  # a wait consults the status word after this long (~50 us)


class Barrier:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.completed = 0
        self.waiters = []


class Sim:
    def __init__(self, rng, jitter, fault=None):
        self.rng = rng
        self.jitter = jitter
        self.fault = fault
        self.status = False
        self.waits_done = defaultdict(int)
        self.finish = {}
        self.queue = []
        self.seq = 0
        self.bars = {}
        self.acc = defaultdict(list)
        self.errors = []
        self.pipe_free = 0
        self.reduce_free = 0
        self.groups = []
        self.live = set()

    # -- infrastructure --------------------------------------------------------
    def d(self, lo, hi):
        v = self.rng.randint(lo, hi)
        if self.rng.random() < self.jitter:  # occasional long stall of one engine or warp
            v += self.rng.randint(2000, 30000)
        return v

    def at(self, t, fn):
        heapq.heappush(self.queue, (t, self.seq, fn))
        self.seq += 1

    def barrier(self, name, count=1):
        self.bars[name] = Barrier(count)

    def arrive(self, name, t):
        b = self.bars[name]
        b.pending -= 1
        assert b.pending >= 0
        if b.pending == 0:
            b.completed += 1
            b.pending = b.count
            keep = []
            for w in b.waiters:
                if b.completed == w["k"] + 1:
                    self.wake(w, t + self.rng.randint(1, 200), True)
                else:
                    keep.append(w)
            b.waiters = keep

    def wake(self, w, t, value):
        if not w["done"]:
            w["done"] = True
            self.at(t, lambda tt: w["resume"](tt, value))

    def set_status(self, t):
        """A wait failed: every pending wait gives up once it has lasted STATUS_CHECK."""
        if self.status:
            return
        self.status = True
        for b in self.bars.values():
            for w in b.waiters:
                self.at(max(t, w["start"] + STATUS_CHECK), lambda tt, w=w: self.wake(w, tt, False))

    def record(self, res, t0, t1, kind, tag, who):
        self.acc[res].append((t0, t1, kind, tag, who))

    def spawn(self, name, gen):
        self.live.add(name)
        self.at(0, lambda t: self.advance(name, gen, t))

    def advance(self, name, gen, t, value=None):
        """Runs one role from time t (the current time of the event loop) until its
        next step that takes time, which resumes it through the event queue: every
        action therefore happens in global time order."""
        def later(dt, v=None):
            self.at(t + dt, lambda tt: self.advance(name, gen, tt, v))

        while True:
            try:
                cmd = gen.send(value)
            except StopIteration:
                self.live.discard(name)
                self.finish[name] = t
                return
            value = None
            op = cmd[0]
            if op == "delay":
                later(cmd[1])
                return
            if op == "wait":
                _, bname, k = cmd
                b = self.bars[bname]
                self.waits_done[name] += 1
                if self.fault == (name, self.waits_done[name]):  # this phase never completes
                    self.set_status(t)
                    later(STATUS_CHECK, False)
                    return
                if b.completed == k + 1:
                    later(1, True)
                    return
                if b.completed > k + 1:
                    self.errors.append(f"{name}: {bname} ran past phase {k} (completed {b.completed}) before the wait")
                    self.live.discard(name)
                    return
                w = {"k": k, "start": t, "done": False,
                     "resume": lambda tt, v: self.advance(name, gen, tt, v)}
                b.waiters.append(w)
                if self.status:
                    self.at(t + STATUS_CHECK, lambda tt: self.wake(w, tt, False))
                return
            if op == "arrive":
                self.arrive(cmd[1], t)
                later(1)
                return
            if op == "access":  # the warp's own loads and stores: (res list, kind, tag or expected)
                _, items, dur = cmd
                for res, kind, tag in items:
                    self.record(res, t, t + dur, kind, tag, name)
                later(dur)
                return
            if op == "mma":
                _, reads, writes = cmd
                start = max(t, self.pipe_free)
                end = start + self.d(300, 900)
                for res, exp in reads:
                    self.record(res, start, end, "R", exp, name)
                for res, tag in writes:
                    self.record(res, start, end, "W", tag, name)
                self.pipe_free = end
                later(self.rng.randint(5, 80))
                return
            if op == "commit":
                bname = cmd[1]
                self.at(max(t, self.pipe_free), lambda tt, b=bname: self.arrive(b, tt))
                later(1)
                return
            if op == "load":
                _, items, bname = cmd
                end = t + self.d(400, 4000)
                for res, tag in items:
                    self.record(res, t, end, "W", tag, name)
                self.at(end, lambda tt, b=bname: self.arrive(b, tt))
                later(1)
                return
            if op == "reduce":
                _, reads = cmd
                start = max(t, self.reduce_free)
                end = start + self.d(800, 3000)
                for res, exp in reads:
                    self.record(res, start, end, "R", exp, name)
                self.reduce_free = end
                self.groups.append(end)
                later(1)
                return
            if op == "wait_read":  # all but the n most recent reduce groups have read their sources
                n = cmd[1]
                older = self.groups[:-n] if n else self.groups
                later(max([t] + older) - t + 1)
                return
            raise ValueError(op)

    def run(self):
        while self.queue:
            t, _, fn = heapq.heappop(self.queue)
            fn(t)
        if self.live:
            self.errors.append(f"deadlock: {sorted(self.live)} never finished")
        if self.fault is not None:
            return self.failure_checks()
        for res, acc in self.acc.items():
            writes = [a for a in acc if a[2] == "W"]
            for w in writes:
                for a in acc:
                    same_op = a[4] == w[4] and a[0] == w[0] and a[1] == w[1]  # an MMA accumulating in place
                    if a is not w and not same_op and a[0] < w[1] and w[0] < a[1]:
                        self.errors.append(f"{res}: {w[4]} writes {w[3]} during {a[4]} {a[2]} {a[3]}")
            for r in acc:
                if r[2] != "R" or r[3] is None:
                    continue
                prior = [w for w in writes if w[1] <= r[0]]
                last = max(prior, key=lambda w: w[1])[3] if prior else None
                if last != r[3]:
                    self.errors.append(f"{res}: {r[4]} reads {last!r}, needs {r[3]!r}")
        return self.errors

    def failure_checks(self):
        """After an injected fault: nothing still running when the last role ends,
        nothing touching a region after its release (a write tagged "freed")."""
        end = max(self.finish.values(), default=0)
        for res, acc in self.acc.items():
            freed = [a for a in acc if a[3] == "freed"]
            for a in acc:
                if a[1] > end:
                    self.errors.append(f"{res}: {a[4]} {a[2]} {a[3]} still running when the last role ended")
                if freed and a[3] != "freed" and a[1] > freed[0][0]:
                    self.errors.append(f"{res}: {a[4]} {a[2]} {a[3]} after the release")
        return self.errors
