"""A randomised model of k_attn_tc's mbarrier protocol (attention_tc.cu), run on
the CPU: the copy lane, the MMA lane with its two non-blocking streams (S of a
tile, P.V of a tile) and the four softmax warps, with the parity semantics of
mbarrier waits and random completion times for copies and MMAs.  Every wait
that returns must see exactly the phase it asked for, every MMA must read a
stage that holds its own tile's data, and no buffer may be overwritten while
it is read.  The protocol as built passes on random schedules; the same
protocol without its guard (an item's copy barrier tested before the item
before it in that stage was taken) is caught: a parity test then returns for
a phase two behind."""
import random

import pytest


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.c = count, count, 0   # c = completed phases

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.c += 1
            self.pending = self.count

    def test(self, n):
        """parity test for the completion of phase n"""
        return (self.c & 1) != (n & 1)


class Violation(AssertionError):
    pass


def simulate(n, stages, seed, guard=True):
    R = random.Random(seed)
    full = [Bar(1) for _ in range(stages)]
    empty = [Bar(1) for _ in range(stages)]
    sF, sE = [Bar(1), Bar(1)], [Bar(4), Bar(4)]
    pF, pE = Bar(4), Bar(1)
    oF, oE = [Bar(1), Bar(1)], [Bar(4), Bar(4)]
    item = [None] * stages      # the item a stage holds
    landed = [False] * stages
    reading = [0] * stages      # MMAs in flight on the stage
    s_tile, s_done = [None, None], [False, False]
    o_tile, o_done = [None, None], [False, False]
    p_tile = [None]
    events, clock = [], [0.0]

    def later(fn, lo, hi):
        events.append((clock[0] + R.uniform(lo, hi), fn))

    def expect(bar, k, what):
        if bar.c != k + 1:
            raise Violation(f"{what}: {bar.c} phases complete, waited for #{k}")

    prod = {"u": 0}

    def producer():
        u = prod["u"]
        if u >= 2 * n:
            return False
        st = u % stages
        if u >= stages:
            if not empty[st].test(u // stages - 1):
                return False
            expect(empty[st], u // stages - 1, "empty")
            if reading[st]:
                raise Violation("stage refilled under an MMA")
        item[st], landed[st] = u, False

        def land(st=st, u=u):
            if item[st] != u:
                raise Violation("copy landed in a stage that moved on")
            landed[st] = True
            full[st].arrive()
        later(land, 5, 200)
        prod["u"] += 1
        return True

    m = {"ts": 0, "tp": 0}

    def taken(v):
        return v < 0 or ((v >> 1) < m["tp"] if v & 1 else (v >> 1) < m["ts"])

    def mma():
        did = False
        ts, tp = m["ts"], m["tp"]
        if ts < n and (not guard or taken(2 * ts - stages)):
            u, st = 2 * ts, (2 * ts) % stages
            if full[st].test(u // stages) and (ts < 2 or sE[ts & 1].test((ts >> 1) - 1)):
                expect(full[st], u // stages, "keys")
                if not (item[st] == u and landed[st]):
                    raise Violation("S read a stage without its keys")
                reading[st] += 1
                s_tile[ts & 1], s_done[ts & 1] = ts, False

                def done(st=st, ts=ts):
                    reading[st] -= 1
                    empty[st].arrive()
                    s_done[ts & 1] = True
                    sF[ts & 1].arrive()
                later(done, 2, 20)
                m["ts"] += 1
                did = True
        if tp < m["ts"] and (not guard or taken(2 * tp + 1 - stages)):
            u, st = 2 * tp + 1, (2 * tp + 1) % stages
            if pF.test(tp) and full[st].test(u // stages) and (tp < 2 or oE[tp & 1].test((tp >> 1) - 1)):
                expect(pF, tp, "P")
                expect(full[st], u // stages, "values")
                if not (item[st] == u and landed[st]):
                    raise Violation("P.V read a stage without its values")
                if p_tile[0] != tp:
                    raise Violation("P.V read another tile's P")
                reading[st] += 1
                o_tile[tp & 1], o_done[tp & 1] = tp, False

                def done(st=st, tp=tp):
                    reading[st] -= 1
                    empty[st].arrive()
                    o_done[tp & 1] = True
                    oF[tp & 1].arrive()
                    pE.arrive()
                later(done, 2, 30)
                m["tp"] += 1
                did = True
        return did

    warps = [{"t": 0, "ph": 0} for _ in range(4)]
    at_barrier = [0] * (n + 1)
    wrote = [0] * (n + 1)

    def warp(x):
        t = x["t"]
        if t > n:
            return False
        if t == n:                               # the last tile's O
            if n > 0:
                if not oF[(n - 1) & 1].test((n - 1) >> 1):
                    return False
                expect(oF[(n - 1) & 1], (n - 1) >> 1, "last O")
            x["t"] += 1
            return True
        if x["ph"] == 0:                         # S of tile t
            if not sF[t & 1].test(t >> 1):
                return False
            expect(sF[t & 1], t >> 1, "S")
            if not (s_done[t & 1] and s_tile[t & 1] == t):
                raise Violation("softmax read another tile's S")
            sE[t & 1].arrive()
            at_barrier[t] += 1
            x["ph"] = 1
            return True
        if x["ph"] == 1:                         # named barrier of the four warps
            if at_barrier[t] < 4:
                return False
            x["ph"] = 2
            return True
        if x["ph"] == 2:                         # P of tile t
            if t >= 1:
                if not pE.test(t - 1):
                    return False
                expect(pE, t - 1, "P free")
                if not (o_done[(t - 1) & 1] and o_tile[(t - 1) & 1] == t - 1):
                    raise Violation("P overwritten under P.V")
            wrote[t] += 1
            if wrote[t] == 4:
                p_tile[0] = t
            pF.arrive()
            x["ph"] = 3
            return True
        if t >= 1:                               # O of tile t - 1
            if not oF[(t - 1) & 1].test((t - 1) >> 1):
                return False
            expect(oF[(t - 1) & 1], (t - 1) >> 1, "O")
            oE[(t - 1) & 1].arrive()
        x["t"] += 1
        x["ph"] = 0
        return True

    for _ in range(200000):
        if all(x["t"] > n for x in warps) and m["tp"] >= n:
            return
        actors = ["p", "m", 0, 1, 2, 3]
        R.shuffle(actors)
        moved = False
        for a in actors:
            moved |= producer() if a == "p" else mma() if a == "m" else warp(warps[a])
        if events and (not moved or R.random() < 0.3):
            events.sort(key=lambda e: e[0])
            clock[0], fn = events.pop(0)
            fn()
        elif not moved:
            raise Violation("deadlock")
    raise Violation("no progress")


@pytest.mark.parametrize("stages", [2, 3])
def test_protocol_holds(stages):
    for n in (0, 1, 2, 3, 5, 16):
        for seed in range(60):
            simulate(n, stages, seed)


def test_model_catches_the_unguarded_protocol():
    caught = 0
    for n in (3, 5, 16):
        for seed in range(60):
            try:
                simulate(n, 3, seed, guard=False)
            except Violation:
                caught += 1
    assert caught > 0
