"""A host-side model of the tensor-core forward's synchronisation (`fwd_tc_kernel`
in csrc/ra_fwd_tc.cu), run under random timings with the engine of
tests/protocol_sim.py.

Roles as in the kernel: the TMA warp (both Q tiles once, then K and V of each
K/V tile into two-stage rings, each refill after its empty barrier), the MMA
thread (in order: S_A(0), S_B(0); then per tile j: PV_A(j), S_A(j+1), PV_B(j),
S_B(j+1), with the K-empty, V-empty, S-full and O-done commits) and two softmax
warpgroups (one per Q tile, four lane quarters each): wait for S, rescale O when
the running max moves (only after S(j+1), whose commit certifies PV(j)), write P
over the first half of the S columns, arrive on P-full; at the end read O.

Checked over random timings and tile counts: no deadlock, no barrier phase
overtaken before its wait, no write overlapping another access of the same
region, and every read seeing its own tile's version (S_X(j) reads K of tile j,
PV_X(j) reads P_X(j), V of tile j and the O that the softmax left).  Planted
mistakes in the model must be caught.  With a never-completing wait injected at
every wait of every role in turn, the roles follow the kernel's error exits:
every role ends, no MMA or load outlives the last role, and TMEM is not touched
after its release."""
import random

import pytest

from protocol_sim import Sim

QUARTERS = (0, 1, 2, 3)
TILES = (0, 1)  # Q tiles A and B


def S_parts(X, tag=None):
    return [(("S", X, part, q), tag) for part in ("P", "rest") for q in QUARTERS]


def O_all(X, tag=None):
    return [(("O", X, q), tag) for q in QUARTERS]


def producer(sim, n, mut):
    yield ("load", [(("Q", X), "Q") for X in TILES], "QFull")
    j = 0            # tiles whose K load was issued
    last_v = True    # whether the V load of tile j-1 was issued too
    while j < n:
        st = j % 2
        yield ("delay", sim.d(1, 200))
        if "no_kempty_wait" not in mut and j >= 2:
            if not (yield ("wait", f"KEmpty{st}", j // 2 - 1)):
                break
        yield ("load", [(("K", st), f"K{j}")], "KFull0" if "one_kfull" in mut else f"KFull{st}")
        if j >= 2 and not (yield ("wait", f"VEmpty{st}", j // 2 - 1)):
            j += 1  # the K load of this tile is in flight, its V load is not
            last_v = False
            break
        yield ("load", [(("V", st), f"V{j}")], f"VFull{st}")
        j += 1
    # every load this warp issued lands before the CTA may exit
    yield ("wait", "QFull", 0)
    for back in (1, 2):
        if back <= j:
            jj = j - back
            yield ("wait",) + (("KFull0", jj) if "one_kfull" in mut else (f"KFull{jj % 2}", jj // 2))
            if last_v or back > 1:
                yield ("wait", f"VFull{jj % 2}", jj // 2)


def mma(sim, n, mut, state):
    def kfull(j):
        return ("KFull0", j) if "one_kfull" in mut else (f"KFull{j % 2}", j // 2)

    def s_mma(X, j):
        return ("mma", [(("Q", X), "Q"), (("K", j % 2), f"K{j}")], S_parts(X, f"S{X}{j}"))

    def pv_mma(X, j):
        reads = [(r, f"P{X}{j}") for r, _ in S_parts(X) if r[2] == "P"] + [(("V", j % 2), f"V{j}")]
        if j > 0:  # accumulate: O as the softmax left it
            reads += [((("O", X, q)), state.get((X, j, q))) for q in QUARTERS]
        return ("mma", reads, O_all(X, f"O{X}{j}"))

    ok = yield ("wait", "QFull", 0)
    if ok and n > 0:
        ok = yield ("wait",) + kfull(0)
        if ok:
            yield s_mma(0, 0)
            yield ("commit", "SFull0")
            yield s_mma(1, 0)
            yield ("commit", "SFull1")
            yield ("commit", "KEmpty0")
        j = 0
        while ok:
            more = j + 1 < n
            yield ("delay", sim.d(1, 150))
            ok = (yield ("wait", f"VFull{j % 2}", j // 2)) and (yield ("wait", "PFull0", j))
            if not ok:
                break
            yield pv_mma(0, j)
            if "vempty_after_pv_a" in mut:
                yield ("commit", f"VEmpty{j % 2}")
            if more:
                ok = yield ("wait",) + kfull(j + 1)
                if not ok:
                    break
                yield s_mma(0, j + 1)
                yield ("commit", "SFull0")
            else:
                yield ("commit", "ODone0")
            ok = yield ("wait", "PFull1", j)
            if not ok:
                break
            yield pv_mma(1, j)
            if "vempty_after_pv_a" not in mut:
                yield ("commit", f"VEmpty{j % 2}")
            if more:
                yield s_mma(1, j + 1)
                yield ("commit", "SFull1")
                yield ("commit", f"KEmpty{(j + 1) % 2}")
            else:
                yield ("commit", "ODone1")
                break
            j += 1
    elif ok:
        yield ("commit", "ODone0")
        yield ("commit", "ODone1")
    # every MMA issued complete, the epilogue's reads done, then TMEM released
    yield ("commit", "Final")
    yield ("wait", "Final", 0)
    if "no_epidone_wait" not in mut:
        yield ("wait", "EpiDone", 0)
    yield ("access", [(r, "W", "freed") for X in TILES for r, _ in S_parts(X) + O_all(X)], 1)


def softmax(sim, n, X, q, mut, state):
    last_o = None  # the version of this quarter's O as the softmax last saw or made it
    ok = True
    for j in range(n):
        yield ("delay", sim.d(1, 300))
        if "rescale_before_sfull" in mut and j > 0 and sim.rng.random() < 0.5:
            yield ("access", [(("O", X, q), "W", f"R{X}{j}")], sim.d(100, 400))
            last_o = f"R{X}{j}"
        ok = yield ("wait", f"SFull{X}", j)
        if not ok:
            break
        yield ("access", [(r, "R", f"S{X}{j}") for r, _ in S_parts(X) if r[3] == q], sim.d(200, 700))
        if "rescale_before_sfull" not in mut and j > 0 and sim.rng.random() < 0.3:
            # the running max moved: O scaled in TMEM (PV(j-1) is complete: S(j) was committed after it)
            yield ("access", [(("O", X, q), "R", f"O{X}{j - 1}")], sim.d(50, 200))
            yield ("access", [(("O", X, q), "W", f"R{X}{j}")], sim.d(50, 200))
            last_o = f"R{X}{j}"
        elif j > 0 and "rescale_before_sfull" not in mut:
            last_o = f"O{X}{j - 1}"
        state[(X, j, q)] = last_o
        yield ("delay", sim.d(200, 1000))
        yield ("access", [(("S", X, "P", q), "W", f"P{X}{j}")], sim.d(50, 300))
        yield ("arrive", f"PFull{X}")
        last_o = None
    if ok:
        ok = yield ("wait", f"ODone{X}", 0)
    if ok and n > 0:
        yield ("access", [(("O", X, q), "R", f"O{X}{n - 1}")], sim.d(100, 400))
    yield ("arrive", "EpiDone")


def simulate(seed, n, mut=(), jitter=0.05, fault=None, keep=False):
    sim = Sim(random.Random(seed), jitter, fault)
    sim.barrier("QFull")
    for st in (0, 1):
        for b in ("KFull", "KEmpty", "VFull", "VEmpty"):
            sim.barrier(f"{b}{st}")
    for X in TILES:
        sim.barrier(f"SFull{X}")
        sim.barrier(f"PFull{X}", 4)  # the kernel counts 128 threads; here one arrival per warp
        sim.barrier(f"ODone{X}")
    sim.barrier("Final")
    sim.barrier("EpiDone", 8)
    state = {}
    sim.spawn("producer", producer(sim, n, mut))
    sim.spawn("mma", mma(sim, n, mut, state))
    for X in TILES:
        for q in QUARTERS:
            sim.spawn(f"softmax{X}{q}", softmax(sim, n, X, q, mut, state))
    errors = sim.run()
    return (errors, sim) if keep else errors


def test_protocol_holds_under_random_timing():
    for seed in range(400):
        n = seed % 8
        errors = simulate(seed, n, jitter=0.02 if seed % 2 else 0.1)
        assert not errors, f"seed {seed}, {n} tiles: {errors[:3]}"


@pytest.mark.parametrize("mutation", ["no_kempty_wait", "one_kfull", "vempty_after_pv_a", "rescale_before_sfull",
                                      "no_epidone_wait"])
def test_planted_protocol_mistake_is_caught(mutation):
    caught = [s for s in range(400) if simulate(s, 2 + s % 6, (mutation,), jitter=0.1)]
    assert caught, f"{mutation} passed every timing"


def _faults(seed, n):
    """Every wait of every role, in a clean run of the same timing."""
    _, sim = simulate(seed, n, keep=True)
    return [(role, k) for role, count in sorted(sim.waits_done.items()) for k in range(1, count + 1)]


@pytest.mark.parametrize("n", [0, 1, 2, 5])
def test_failure_paths(n):
    """A wait that never completes, at every wait of every role: every role still
    ends, no MMA or load is running when the last one does, and nothing touches
    TMEM after it is released."""
    for seed in (21, 22):
        for fault in _faults(seed, n):
            errors = simulate(seed, n, fault=fault)
            assert not errors, f"seed {seed}, {n} tiles, fault {fault}: {errors[:3]}"
