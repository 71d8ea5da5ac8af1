"""A randomised model of k_score_tc's mbarrier protocol (score_tc.cu), run on the
CPU: the copy lane, the MMA lane, the scan group (query operands; without
wrong-side sums also each stage's C_b share) and the four TMEM warps, with the
parity semantics of mbarrier waits, random copy times, and tensor-core MMAs
that complete in issue order with commits that arrive once every earlier MMA
is done.

Checked on every schedule: a wait that returns sees exactly the phase it asked
for; an MMA reads a stage that holds its own piece, the operand of its own
segment and an accumulator no TMEM warp is still reading; no stage, operand,
max_d Q_d slot or C_b slot is overwritten while it is read; the TMEM warps read
each tile's finished accumulator with its own segment's max_d Q_d and C_b.
The protocol as built passes with whole and split halves, with and without
wrong-side sums, over tile ranges that cross segments; the same protocol with
one hand-off left out is caught."""
import random

import pytest

N_ACC, N_C, N_TMEM = 4, 4, 4


class Violation(AssertionError):
    pass


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.c = count, count, 0   # c = completed phases

    def arrive(self, n=1):
        for _ in range(n):
            self.pending -= 1
            if self.pending == 0:
                self.c += 1
                self.pending = self.count

    def test(self, k):
        """parity test for the completion of phase k"""
        return (self.c & 1) != (k & 1)


def simulate(tiles, stages, pieces, wsum, seed, mutate=None):
    """tiles: the segment of each tile of the CTA's range, in order."""
    R = random.Random(seed)
    T = len(tiles)
    per_tile = 2 * pieces
    full = [Bar(1) for _ in range(stages)]
    empty = [Bar(1 if (wsum or mutate == "empty_count") else 1 + 4) for _ in range(stages)]
    accF, accE = [Bar(1) for _ in range(N_ACC)], [Bar(N_TMEM) for _ in range(N_ACC)]
    bqF, bqE = Bar(1), Bar(1)
    qmF, qmE = [Bar(1), Bar(1)], [Bar(N_TMEM), Bar(N_TMEM)]
    cF, cE = [Bar(1) for _ in range(N_C)], [Bar(N_TMEM) for _ in range(N_C)]

    st_item, st_landed, st_reads = [None] * stages, [False] * stages, [0] * stages
    b_seg, b_reads = [None], [0]
    qm_seg = [None, None]
    acc_tile, acc_left, acc_reading = [None] * N_ACC, [0] * N_ACC, [0] * N_ACC
    c_tile = [None] * N_C
    events, clock, mma_tail = [], [0.0], [0.0]

    def later(fn, lo, hi):
        events.append((clock[0] + R.uniform(lo, hi), fn))

    def expect(bar, k, what):
        if bar.c != k + 1:
            raise Violation(f"{what}: {bar.c} phases complete, waited for #{k}")

    def mma(on_done):
        """an MMA issued now; MMAs complete in issue order"""
        mma_tail[0] = max(mma_tail[0], clock[0]) + R.uniform(0.5, 8)
        events.append((mma_tail[0], on_done))

    def commit(bar):
        """arrives once every MMA issued so far has completed"""
        events.append((max(mma_tail[0], clock[0]) + 1e-9, bar.arrive))

    segs = []
    for s in tiles:
        if not segs or segs[-1] != s:
            segs.append(s)

    # ---- copy lane
    P = {"u": 0}

    def producer():
        u = P["u"]
        if u >= per_tile * T:
            return False
        st = u % stages
        if u >= stages:
            if not empty[st].test(u // stages - 1):
                return False
            expect(empty[st], u // stages - 1, "empty")
            if st_reads[st]:
                raise Violation("stage refilled under an MMA")
        st_item[st], st_landed[st] = u, False

        def land(st=st, u=u):
            if st_item[st] != u:
                raise Violation("copy landed in a stage that moved on")
            st_landed[st] = True
            full[st].arrive()
        later(land, 2, 60)
        P["u"] += 1
        return True

    # ---- MMA lane
    M = {"i": 0, "q": 0, "seg": None, "nseg": 0, "phase": "tile"}

    def mma_lane():
        i = M["i"]
        if i >= T:
            return False
        s = tiles[i]
        acc = i % N_ACC
        if M["phase"] == "tile":
            if s != M["seg"]:
                if M["seg"] is not None:
                    commit(bqE)
                M["seg"] = s
                M["phase"] = "operand"
                return True
            M["phase"] = "acc"
            return True
        if M["phase"] == "operand":
            k = M["nseg"]
            if not bqF.test(k):
                return False
            expect(bqF, k, "operand")
            if b_seg[0] != s:
                raise Violation("MMA would read another segment's operand")
            M["nseg"] += 1
            M["phase"] = "acc"
            return True
        if M["phase"] == "acc":
            if i >= N_ACC and mutate != "acc_wait":
                if not accE[acc].test(i // N_ACC - 1):
                    return False
                expect(accE[acc], i // N_ACC - 1, "accumulator free")
            if acc_reading[acc]:
                raise Violation("accumulator overwritten while a TMEM warp reads it")
            if acc_tile[acc] is not None and acc_left[acc]:
                raise Violation("accumulator reused before its MMAs completed")
            acc_tile[acc], acc_left[acc] = i, per_tile
            M["phase"] = "piece"
            return True
        # a piece of tile i
        q = M["q"]
        u = i * per_tile + q
        st = u % stages
        if not full[st].test(u // stages):
            return False
        expect(full[st], u // stages, "piece")
        if not (st_item[st] == u and st_landed[st]):
            raise Violation("MMA read a stage without its piece")
        if b_seg[0] != s:
            raise Violation("MMA read another segment's operand")
        st_reads[st] += 1
        b_reads[0] += 1

        def done(st=st, acc=acc):
            st_reads[st] -= 1
            b_reads[0] -= 1
            acc_left[acc] -= 1
        mma(done)
        commit(empty[st])
        M["q"] += 1
        if M["q"] == per_tile:
            commit(accF[acc])
            M["q"] = 0
            M["i"] += 1
            M["phase"] = "tile"
        return True

    # ---- scan group (four warps moving together between named barriers)
    S = {"built": 0, "i": 0, "q": 0, "seg": None, "used": 0, "phase": "build", "next": 0}
    Q_slot = [None, None]       # the segment whose Q_d a slot holds (the group's own reads)

    def build_step():
        """one operand build: returns None when blocked, True when done"""
        k = S["built"]
        if k >= 1 and mutate != "operand_wait":
            if not bqE.test(k - 1):
                return None
            expect(bqE, k - 1, "operand free")
        if b_reads[0] and k >= 1:
            raise Violation("operand rewritten under an MMA")
        if k >= 2:
            if not qmE[k & 1].test((k >> 1) - 1):
                return None
            expect(qmE[k & 1], (k >> 1) - 1, "max slot free")
        b_seg[0] = segs[k]
        bqF.arrive()
        Q_slot[k & 1] = segs[k]
        qm_seg[k & 1] = segs[k]
        qmF[k & 1].arrive()
        S["built"] += 1
        return True

    def scan():
        if S["phase"] == "build":                 # the first operand, then (with wsum) all of them
            if S["built"] >= len(segs):
                S["phase"] = "done" if wsum else "tiles"
                return True
            r = build_step()
            if r is None:
                return False
            if not wsum:
                S["phase"] = "tiles"
            return True
        if S["phase"] in ("done",):
            return False
        i = S["i"]
        if i >= T:
            return False
        s = tiles[i]
        if S["phase"] == "tiles":
            if s != S["seg"]:
                if S["seg"] is not None:
                    S["phase"] = "rebuild"
                    return True
                S["seg"] = s
                S["used"] += 1
            S["phase"] = "pieces"
            return True
        if S["phase"] == "rebuild":               # the segment before is done: build the next one
            if S["built"] < len(segs):
                r = build_step()
                if r is None:
                    return False
            S["seg"] = s
            S["used"] += 1
            S["phase"] = "pieces"
            return True
        if S["phase"] == "pieces":
            q = S["q"]
            u = i * per_tile + q
            st = u % stages
            if not full[st].test(u // stages):
                return False
            expect(full[st], u // stages, "scan piece")
            if not (st_item[st] == u and st_landed[st]):
                raise Violation("scan read a stage without its piece")
            if Q_slot[(S["used"] - 1) & 1] != s:
                raise Violation("scan weighted C_b with another segment's Q")
            empty[st].arrive(4)
            S["q"] += 1
            if S["q"] == per_tile:
                S["q"] = 0
                S["phase"] = "c"
            return True
        # C_b of tile i to the TMEM warps
        cb = i % N_C
        if i >= N_C:
            if not cE[cb].test(i // N_C - 1):
                return False
            expect(cE[cb], i // N_C - 1, "C slot free")
        c_tile[cb] = i
        cF[cb].arrive()
        S["i"] += 1
        S["phase"] = "tiles"
        return True

    # ---- TMEM warps (independent)
    tw = [{"i": 0, "seg": None, "used": 0, "phase": "tile", "read": False} for _ in range(N_TMEM)]

    def tmem(x):
        i = x["i"]
        if i >= T:
            return False
        s = tiles[i]
        acc = i % N_ACC
        if x["phase"] == "tile":
            if s != x["seg"]:
                b = x["used"] & 1
                if not qmF[b].test(x["used"] >> 1):
                    return False
                expect(qmF[b], x["used"] >> 1, "max_d Q_d")
                if qm_seg[b] != s:
                    raise Violation("TMEM warp took another segment's max_d Q_d")
                qmE[b].arrive()
                x["used"] += 1
                x["seg"] = s
            x["phase"] = "acc"
            return True
        if x["phase"] == "acc":
            if not accF[acc].test(i // N_ACC):
                return False
            expect(accF[acc], i // N_ACC, "accumulator")
            if not (acc_tile[acc] == i and acc_left[acc] == 0):
                raise Violation("TMEM warp read an unfinished or foreign accumulator")
            acc_reading[acc] += 1
            x["read"] = False
            # tcgen05.ld, max, radius and stores; now and then the warp is held up far longer
            lo, hi = (1, 40) if R.random() < 0.9 else (100, 600)
            later(lambda x=x: x.__setitem__("read", True), lo, hi)
            x["phase"] = "release"
            return True
        if x["phase"] == "release":
            if not x["read"]:
                return False
            if acc_tile[acc] != i:
                raise Violation("accumulator overwritten while a TMEM warp read it")
            acc_reading[acc] -= 1
            accE[acc].arrive()
            x["phase"] = "c" if not wsum else "next"
            return True
        if x["phase"] == "c":
            cb = i % N_C
            if not cF[cb].test(i // N_C):
                return False
            expect(cF[cb], i // N_C, "C_b")
            if c_tile[cb] != i:
                raise Violation("TMEM warp took another tile's C_b")
            cE[cb].arrive()
        x["i"] += 1
        x["phase"] = "tile"
        return True

    actors = ["p", "m", "s"] + list(range(N_TMEM))
    for _ in range(400000):
        if P["u"] >= per_tile * T and M["i"] >= T and all(x["i"] >= T for x in tw) \
                and (wsum or S["i"] >= T):
            return
        R.shuffle(actors)
        moved = False
        for a in actors:
            moved |= producer() if a == "p" else mma_lane() if a == "m" else scan() if a == "s" else tmem(tw[a])
        if events and (not moved or R.random() < 0.3):
            events.sort(key=lambda e: e[0])
            clock[0], fn = events.pop(0)
            fn()
        elif not moved:
            raise Violation("deadlock")
    raise Violation("no progress")


# tile ranges of one CTA: within one segment, across segment boundaries, a
# one-tile segment, and more segments than operand and max_d Q_d slots
RANGES = [[0] * 6, [0, 0, 1, 1, 1, 1, 1], [3, 4, 4, 4, 5], [0, 1, 2, 3, 3, 4, 5, 5, 5, 6]]


@pytest.mark.parametrize("pieces,stages", [(1, 2), (1, 3), (2, 4), (2, 5)])
@pytest.mark.parametrize("wsum", [True, False])
def test_protocol_holds(pieces, stages, wsum):
    for tiles in RANGES:
        for seed in range(25):
            simulate(tiles, stages, pieces, wsum, seed)


@pytest.mark.parametrize("mutate,wsum", [("acc_wait", True), ("operand_wait", True), ("empty_count", False)])
def test_model_catches_a_missing_hand_off(mutate, wsum):
    """without the TMEM warps' accumulator release, the scan group's wait for
    the operand to be free, or the scan warps' arrivals on a stage's release,
    some schedule breaks a check"""
    caught = 0
    for tiles in RANGES:
        for seed in range(40):
            try:
                simulate(tiles, 4, 2, wsum, seed, mutate=mutate)
            except Violation:
                caught += 1
    assert caught > 0
