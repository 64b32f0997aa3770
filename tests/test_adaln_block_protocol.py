"""The synchronisation protocol of the 7,168-column AdaLN block kernel
(adaln_block_kernel in csrc/adaln.cu), checked on the CPU by random interleavings.

The kernel's 14 warps are modelled one step at a time: the stats warp publishes
each step's rows and arrives on a named barrier per other warp (count 64); the
other warps form pass 1 of the next step, wait on their own barrier, arrive on
the shared totals barrier (count 448, which only the stats warp waits on),
refill a ring stage with cp.async and emit pass 2.  Named barriers follow the
PTX semantics (a phase completes when its count of threads has arrived; bar.sync
waits for that, bar.arrive does not), and memory ordering follows them too, with
vector clocks: arriving releases, completing a phase acquires for the warps that
wait in it.  Every interleaving must end (no deadlock), no warp may arrive twice
in one phase, every read of a ring stage, of the published rows and of the
totals must be ordered after the write it needs, and every overwrite after the
reads of what it replaces.  A few planted protocol mistakes must be caught, so
the checker is not vacuous."""
import random

import pytest

NW = 14          # warps of the 448-thread CTA
STATS = 2        # the stats warp (no pass 1)


class Protocol:
    stages = 5
    ahead = 3            # steps whose copies are issued before the loop
    wait_pending = 1     # cp.async groups left pending before pass 1 of step q+1
    issue_after_own_barrier = True
    arrive_after_own_barrier = True
    stats_ahead = True   # the stats warp publishes step q+1 before its own pass 2 of step q
    pass2_only = 13      # the warp with neither pass 1 nor the statistics (6 in the abs-max pass)


class Race(AssertionError):
    pass


def simulate(steps: int, seed: int, proto=Protocol) -> None:
    rng = random.Random(seed)
    p1 = [w for w in range(NW) if w not in (STATS, proto.pass2_only)]
    others = [w for w in range(NW) if w != STATS]
    clk = [[0] * NW for _ in range(NW)]

    def tick(w):
        clk[w][w] += 1
        return list(clk[w])

    def ordered(ev, w):
        return all(a <= b for a, b in zip(ev, clk[w]))

    bars = {}
    blocked = set()

    def arrive(w, bid, count, wait):
        b = bars.setdefault(bid, {"count": count, "in": set(), "acc": [0] * NW, "waiting": []})
        if b["count"] != count:
            raise Race(f"barrier {bid} used with counts {b['count']} and {count}")
        if w in b["in"]:
            raise Race(f"warp {w} arrives twice in one phase of barrier {bid}")
        b["in"].add(w)
        b["acc"] = [max(a, c) for a, c in zip(b["acc"], clk[w])]
        if wait:
            b["waiting"].append(w)
            blocked.add(w)
        if 32 * len(b["in"]) == count:
            for x in b["waiting"]:
                clk[x] = [max(a, c) for a, c in zip(clk[x], b["acc"])]
                blocked.discard(x)
            b.update({"in": set(), "acc": [0] * NW, "waiting": []})

    ring = {}       # (stage, copying warp) -> {"step", "landed", "reads"}
    pending = {w: [] for w in range(NW)}
    rows = {}       # slot -> (step, write clock, reads)
    totals = {}     # (slot, warp) -> (step, write clock, reads)
    issued = [0] * NW

    def issue(w):
        s = issued[w]
        issued[w] += 1
        if w in p1 and s < steps:
            key = (s % proto.stages, w)
            old = ring.get(key)
            if old is not None and not all(ordered(r, w) for r in old["reads"]):
                raise Race(f"warp {w} refills stage {key[0]} with step {s} while step {old['step']} is read")
            ring[key] = {"step": s, "landed": None, "reads": []}
        pending[w].append(s)

    def wait_group(w, n):
        while len(pending[w]) > n:
            s = pending[w].pop(0)
            if w in p1 and s < steps:
                ring[(s % proto.stages, w)]["landed"] = tick(w)

    def read_step(w, s, writers):
        for x in writers:
            e = ring.get((s % proto.stages, x))
            if e is None or e["step"] != s or e["landed"] is None or not ordered(e["landed"], w):
                raise Race(f"warp {w} reads step {s} copied by warp {x} before it is there")
            e["reads"].append(tick(w))

    def pass1(w, q):
        if q >= steps or w not in p1:
            return
        read_step(w, q, [w])
        old = totals.get((q & 1, w))
        if old is not None and not all(ordered(r, w) for r in old[2]):
            raise Race(f"warp {w} overwrites its totals of step {old[0]} before they are read")
        totals[(q & 1, w)] = (q, tick(w), [])

    def publish(w, q):
        for x in p1:
            e = totals.get((q & 1, x))
            if e is None or e[0] != q or not ordered(e[1], w):
                raise Race(f"statistics of step {q} before warp {x} posted its totals")
            e[2].append(tick(w))
        old = rows.get(q & 1)
        if old is not None and not all(ordered(r, w) for r in old[2]):
            raise Race(f"rows of step {q} published over step {old[0]} while it is read")
        rows[q & 1] = (q, tick(w), [])

    def emit(w, q):
        e = rows.get(q & 1)
        if e is None or e[0] != q or not ordered(e[1], w):
            raise Race(f"warp {w} emits step {q} before its rows are published")
        e[2].append(tick(w))
        read_step(w, q, p1)

    def program(w):
        for _ in range(proto.ahead):
            issue(w)
        wait_group(w, proto.ahead - 1)
        pass1(w, 0)
        yield ("syncthreads",)
        if w == STATS and proto.stats_ahead and steps > 0:
            publish(w, 0)
            for c in range(len(others)):
                yield ("arrive", 3 + c, 64)
        for q in range(steps):
            if w == STATS and proto.stats_ahead:
                if q + 1 < steps:
                    yield ("sync", 2, 448)
                    publish(w, q + 1)
                    for c in range(len(others)):
                        yield ("arrive", 3 + c, 64)
                issued[w] += 1
                pending[w].append(None)
            elif w == STATS:
                if q > 0:
                    yield ("sync", 2, 448)
                publish(w, q)
                for c in range(len(others)):
                    yield ("arrive", 3 + c, 64)
                issued[w] += 1
                pending[w].append(None)
            else:
                wait_group(w, proto.wait_pending)
                pass1(w, q + 1)
                yield None
                if not proto.issue_after_own_barrier:
                    issue(w)
                if not proto.arrive_after_own_barrier and q + 1 < steps:
                    yield ("arrive", 2, 448)
                yield ("sync", 3 + others.index(w), 64)
                if proto.arrive_after_own_barrier and q + 1 < steps:
                    yield ("arrive", 2, 448)
                if proto.issue_after_own_barrier:
                    issue(w)
            yield None
            emit(w, q)
            yield None
        wait_group(w, 0)

    progs = {w: program(w) for w in range(NW)}
    done, at_syncthreads = set(), set()
    while len(done) < NW:
        ready = [w for w in range(NW) if w not in done | blocked | at_syncthreads]
        if not ready:
            if at_syncthreads and len(at_syncthreads) == NW:
                acc = [max(col) for col in zip(*(clk[x] for x in at_syncthreads))]
                for x in at_syncthreads:
                    clk[x] = list(acc)
                at_syncthreads.clear()
                continue
            raise Race(f"deadlock with warps {sorted(blocked)} waiting")
        w = rng.choice(ready)
        try:
            op = next(progs[w])
        except StopIteration:
            done.add(w)
            continue
        if op is None:
            continue
        if op[0] == "syncthreads":
            at_syncthreads.add(w)
        else:
            arrive(w, op[1], op[2], op[0] == "sync")
    if any(b["in"] for b in bars.values()):
        raise Race("a barrier phase is left incomplete")


class StatsInStep(Protocol):
    stats_ahead = False  # the stats warp publishes step q, then emits it


class AbsMaxPass(Protocol):
    pass2_only = 6


@pytest.mark.parametrize("proto", [Protocol, AbsMaxPass, StatsInStep])
@pytest.mark.parametrize("steps", [0, 1, 2, 3, 4, 7])
def test_protocol_has_no_deadlock_or_race(steps, proto):
    for seed in range(60):
        simulate(steps, seed, proto)


class FourStages(Protocol):
    stages = 4


class IssueBeforeOwnBarrier(Protocol):
    issue_after_own_barrier = False


class ArriveBeforeOwnBarrier(Protocol):
    arrive_after_own_barrier = False


class NoWaitForCopies(Protocol):
    wait_pending = 2


@pytest.mark.parametrize("proto", [FourStages, IssueBeforeOwnBarrier, ArriveBeforeOwnBarrier, NoWaitForCopies])
def test_planted_protocol_mistakes_are_caught(proto):
    with pytest.raises(Race):
        for seed in range(80):
            for steps in (3, 5, 7):
                simulate(steps, seed, proto)
