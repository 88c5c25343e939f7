"""A host-side model of the tensor-core backward's synchronisation
(`bwd_tc_kernel` in csrc/ra_bwd_tc.cu), run under random timings.

The model follows the kernel's roles step by step: the TMA warp (K/V once, Q and
dO tiles into two stages, the dQ reduce-adds), the MMA thread (an in-order
tensor pipe: S^T, dP^T, dV, dQ, dK) and the eight softmax warps (warp w: query
column half h = w / 4, TMEM lane quarter q = w % 4).  Mbarriers keep their
arrival counts and phases; a wait names the phase it is meant for.  TMA loads,
reduce-adds and MMAs are asynchronous engines with random durations; the MMA
commits arrive when every MMA issued before them has finished.  Every read and
write of a buffer region (TMEM columns per half and lane quarter, the shared-
memory dS^T tile, the Q and dO halves of each stage, the LSE row of each stage and
the two halves of the one D row) is recorded with its time interval.

Checked, over many random timings and tile counts:
  * every wait ends (no deadlock);
  * no barrier runs two phases past the phase a waiter asks for before the
    waiter polls it (the parity of the phase would then read as not complete, or
    as complete for the wrong phase);
  * no write overlaps another access of the same region;
  * every read sees the version it needs (the dS pass reads dP^T of its own tile,
    the reduce-add reads the staged dQ of its own tile, ...).
Planted mistakes in the model (a barrier shared by both stages, a staging buffer
reused too early, a missing wait, the next D row loaded before the drains) must be
caught.

Failure paths: with a wait that never completes injected at every wait of every
role in turn, the roles take the kernel's error exits; every role must still
end, no MMA, load or reduce-add may be running when the last one ends, and
nothing may touch TMEM after its release.  This checks the protocol, not
the arithmetic; the GPU parity tests check the kernel itself."""
import random

import pytest

from protocol_sim import Sim

HALVES, QUARTERS = (0, 1), (0, 1, 2, 3)


# -- the kernel's roles ----------------------------------------------------------
def S_all(tag=None):
    return [(("S", h, part, q), tag) for h in HALVES for part in ("P", "dS") for q in QUARTERS]


def DP_all(tag=None):
    return [(("DP", h, q), tag) for h in HALVES for q in QUARTERS]


def DS_all(tag=None):
    return [(("DS", h, q), tag) for h in HALVES for q in QUARTERS]


def DO_all(st, tag=None):
    return [(("DO", st, q), tag) for q in QUARTERS]


def stage_bar(name, i, mut):
    """Per-stage barriers: tile i uses stage i & 1 and that barrier's phase i >> 1."""
    if name == "KDone" and "kdone_single" in mut:
        return "KDone0", i
    return f"{name}{i & 1}", i >> 1


def producer(sim, n, mut):
    yield ("load", [(("K",), "K"), (("V",), "V")], "KV")
    if "dpfull_no_producer" not in mut:
        yield ("arrive", "DPFull")  # tile 0 has no predecessor
    loaded = 0
    drows = [0, 0]  # D row halves loaded

    def load_drow(half, tile):
        drows[half] += 1
        return ("load", [(("D", half), f"D{tile}")], f"DRow{half}")

    for st in range(min(2, n)):
        # the LSE row of the tile comes with its Q tile, on the same barrier
        yield ("load", [(("Q", st), f"Q{st}"), (("LSE", st), f"L{st}")], f"QFull{st}")
        yield ("load", [(res, f"DO{st}") for res, _ in DO_all(st)], f"DOFull{st}")
        loaded += 1
    if loaded:
        yield load_drow(0, 0)
        yield load_drow(1, 0)
    i = 0
    while i < loaded:
        st = i & 1
        yield ("delay", sim.d(1, 300))
        if "drow_no_wait" in mut and i + 1 < loaded:
            yield load_drow(0, i + 1)
            yield load_drow(1, i + 1)
        if not (yield ("wait",) + stage_bar("DrainQ", i, mut)):
            break
        # the D row half of tile i+1 once the warps that read it for tile i have drained
        if i + 1 < loaded and "drow_no_wait" not in mut:
            yield load_drow(0, i + 1)
        if "stage_q_half" in mut:
            yield ("reduce", [(("Q", st), f"stage{i}")])
        else:
            yield ("reduce", DS_all(f"stage{i}"))
        if not (yield ("wait",) + stage_bar("DrainDO", i, mut)):
            break
        if i + 1 < loaded and "drow_no_wait" not in mut:
            yield load_drow(1, i + 1)
        yield ("reduce", DO_all(st, f"stage{i}"))
        yield ("wait_read", 1)
        if "dpfull_no_producer" not in mut:
            yield ("arrive", "DPFull")  # for tile i+1
        yield ("delay", sim.d(1, 100))  # the walk to tile i+2 (and any stall of this warp)
        nxt = i + 2 < n
        if "no_kdone_wait" not in mut:
            if not (yield ("wait",) + stage_bar("KDone", i, mut)):
                break
        if nxt:
            yield ("load", [(("Q", st), f"Q{i + 2}"), (("LSE", st), f"L{i + 2}")], f"QFull{st}")
        yield ("wait_read", 0)
        if nxt:
            yield ("load", [(res, f"DO{i + 2}") for res, _ in DO_all(st)], f"DOFull{st}")
            loaded += 1
        i += 1
    # every reduce-add complete and every load landed before the CTA may exit
    yield ("wait_read", 0)
    yield ("wait", "KV", 0)
    for back in (1, 2):
        if back <= loaded:
            ii = loaded - back
            yield ("wait", f"QFull{ii & 1}", ii >> 1)
            yield ("wait", f"DOFull{ii & 1}", ii >> 1)
    for half in (0, 1):
        if drows[half]:
            yield ("wait", f"DRow{half}", drows[half] - 1)


def mma(sim, n, mut):
    ok = yield ("wait", "KV", 0)
    if ok and n > 0:
        ok = yield ("wait", "QFull0", 0)
        if ok:
            yield ("mma", [(("K",), "K"), (("Q", 0), "Q0")], S_all("S0"))
            yield ("commit", "SFull")
            ok = yield ("wait", "DOFull0", 0)
        if ok:
            yield ("mma", [(("V",), "V")] + DO_all(0, "DO0"), DP_all("dP0"))
            yield ("commit", "DPFull")
    i = 0
    while ok and i < n:
        st = i & 1
        yield ("delay", sim.d(1, 200))
        if not (yield ("wait", "PReady", i)):
            break
        dv_prev = [(("DV", q), f"dV{i - 1}") for q in QUARTERS] if i else []  # accumulate after tile 0
        yield ("mma", [(r, f"P{i}") for r, _ in S_all() if r[2] == "P"] + DO_all(st, f"DO{i}") + dv_prev,
               [(("DV", q), f"dV{i}") for q in QUARTERS])
        if not (yield ("wait", "DSReady", i)):
            break
        yield ("mma", DS_all(f"dSs{i}") + [(("K",), "K")], DP_all(f"dQ{i}"))  # dQ_i over dP^T
        yield ("commit", "DQFull")
        dk_prev = [(("DK", q), f"dK{i - 1}") for q in QUARTERS] if i else []
        yield ("mma", [(r, f"dS{i}") for r, _ in S_all() if r[2] == "dS"] + [(("Q", st), f"Q{i}")] + dk_prev,
               [(("DK", q), f"dK{i}") for q in QUARTERS])
        yield ("commit", stage_bar("KDone", i, mut)[0])
        if i + 1 == n:
            break
        nst = (i + 1) & 1
        if not (yield ("wait", f"QFull{nst}", (i + 1) >> 1)):
            break
        yield ("mma", [(("K",), "K"), (("Q", nst), f"Q{i + 1}")], S_all(f"S{i + 1}"))
        yield ("commit", "SFull")
        if "no_dqempty_wait" not in mut:
            if not (yield ("wait", "DQEmpty", i)):
                break
        if not (yield ("wait", f"DOFull{nst}", (i + 1) >> 1)):
            break
        yield ("mma", [(("V",), "V")] + DO_all(nst, f"DO{i + 1}"), DP_all(f"dP{i + 1}"))
        yield ("commit", "DPFull")
        i += 1
    # every MMA issued so far complete, the epilogue's reads done, then TMEM released
    yield ("commit", "Final")
    yield ("wait", "Final", 0)
    if "no_epidone_wait" not in mut:
        yield ("wait", "EpiDone", 0)
    freed = S_all() + DP_all() + [(("DK", q), None) for q in QUARTERS] + [(("DV", q), None) for q in QUARTERS]
    yield ("access", [(r, "W", "freed") for r, _ in freed], 1)


def softmax(sim, n, h, q, mut):
    ok = True
    for i in range(n):
        st = i & 1
        yield ("delay", sim.d(1, 300))
        ok = yield ("wait", f"QFull{st}", i >> 1)  # the LSE row, loaded with the Q tile
        if not ok:
            break
        ok = yield ("wait", "SFull", i)
        if not ok:
            break
        yield ("access", [(("S", h, "P", q), "R", f"S{i}"), (("S", h, "dS", q), "R", f"S{i}"),
                          (("LSE", st), "R", f"L{i}")], sim.d(200, 700))
        yield ("delay", sim.d(300, 1200))  # probabilities
        yield ("access", [(("S", h, "P", q), "W", f"P{i}")], sim.d(50, 300))
        yield ("arrive", "PReady")
        ok = yield ("wait", f"DRow{h}", i)  # this half of the D row
        if not ok:
            break
        ok = yield ("wait", "DPFull", i)
        if not ok:
            break
        yield ("access", [(("DP", h, q), "R", f"dP{i}"), (("D", h), "R", f"D{i}")], sim.d(100, 400))
        yield ("delay", sim.d(100, 600))
        yield ("access", [(("S", h, "dS", q), "W", f"dS{i}"), (("DS", h, q), "W", f"dSs{i}")], sim.d(50, 300))
        yield ("arrive", "DSReady")
        ok = yield ("wait", "DQFull", i)
        if not ok:
            break
        yield ("access", [(("DP", h, q), "R", f"dQ{i}")], sim.d(100, 400))
        yield ("arrive", "DQEmpty")
        if h == 0:
            if "stage_q_half" in mut:
                yield ("access", [(("Q", st), "W", f"stage{i}")], sim.d(100, 500))
            else:
                yield ("access", [(("DS", hh, q), "W", f"stage{i}") for hh in HALVES], sim.d(100, 500))
            yield ("arrive", stage_bar("DrainQ", i, mut)[0])
        else:
            yield ("access", [(("DO", st, q), "W", f"stage{i}")], sim.d(100, 500))
            yield ("arrive", stage_bar("DrainDO", i, mut)[0])
    if ok:
        ok = yield ("wait", "Final", 0)
    if ok:  # warps 0-3 write dK out, warps 4-7 dV (an empty walk writes zeros)
        yield ("access", [(("DK" if h == 0 else "DV", q), "R", f"{'dK' if h == 0 else 'dV'}{n - 1}" if n else None)],
               sim.d(100, 400))
    yield ("arrive", "EpiDone")


def simulate(seed, n, mut=(), jitter=0.05, fault=None, keep=False):
    rng = random.Random(seed)
    sim = Sim(rng, jitter, fault)
    sim.barrier("KV")
    for st in (0, 1):
        sim.barrier(f"QFull{st}")
        sim.barrier(f"DOFull{st}")
        sim.barrier(f"DrainQ{st}", 4)
        sim.barrier(f"DrainDO{st}", 4)
        sim.barrier(f"KDone{st}")
    sim.barrier("SFull")
    sim.barrier("DPFull", 1 if "dpfull_no_producer" in mut else 2)
    sim.barrier("PReady", 8)
    sim.barrier("DSReady", 8)
    sim.barrier("DQFull")
    sim.barrier("DQEmpty", 8)
    sim.barrier("Final")
    sim.barrier("EpiDone", 8)
    sim.barrier("DRow0")
    sim.barrier("DRow1")
    sim.spawn("producer", producer(sim, n, mut))
    sim.spawn("mma", mma(sim, n, mut))
    for w in range(8):
        sim.spawn(f"softmax{w}", softmax(sim, n, w >> 2, w & 3, mut))
    errors = sim.run()
    return (errors, sim) if keep else errors


def test_protocol_holds_under_random_timing():
    for seed in range(400):
        n = 1 + seed % 7
        errors = simulate(seed, n, jitter=0.02 if seed % 2 else 0.1)
        assert not errors, f"seed {seed}, {n} tiles: {errors[:3]}"


def test_empty_walk():
    assert not simulate(0, 0)


@pytest.mark.parametrize("mutation", ["kdone_single", "stage_q_half", "dpfull_no_producer", "no_dqempty_wait",
                                      "no_kdone_wait", "no_epidone_wait", "drow_no_wait"])
def test_planted_protocol_mistake_is_caught(mutation):
    caught = [s for s in range(400) if simulate(s, 2 + s % 6, (mutation,), jitter=0.1)]
    assert caught, f"{mutation} passed every timing"


def _faults(seed, n):
    """Every wait of every role, in a clean run of the same timing."""
    _, sim = simulate(seed, n, keep=True)
    return [(role, k) for role, count in sorted(sim.waits_done.items()) for k in range(1, count + 1)]


@pytest.mark.parametrize("n", [1, 2, 5])
def test_failure_paths(n):
    """A wait that never completes, at every wait of every role: every role still
    ends, no MMA, load or reduce-add is running when the last one does, and
    nothing touches TMEM after it is released."""
    for seed in (11, 12):
        for fault in _faults(seed, n):
            errors = simulate(seed, n, fault=fault)
            assert not errors, f"seed {seed}, {n} tiles, fault {fault}: {errors[:3]}"


def test_release_without_epilogue_barrier_is_caught_after_a_fault():
    caught = any(simulate(11, 5, ("no_epidone_wait",), fault=f) for f in _faults(11, 5))
    assert caught
