"""A CPU model of the pair kernel's synchronisation (csrc/swa_prefill_tc.cu,
swa_prefill_bf16_pair_sm103), run under random schedules.

The roles are sequential programs that wait on and arrive at barriers in the
kernel's order:

* the producer.  Skewed protocol (the window path, and fixed patterns with
  items of four tiles and more): tile c's barrier carries K(c) and V(c-1).
  The Q tiles go after the item's first key tile on the window path, first
  for the patterns.  Fixed patterns with short items: one stage per tile for
  K and V, the Q tiles first, the item's tile count posted in a four-slot
  ring;
* the MMA warp: per tile, P_A(c-1) V in two halves, S_A(c), P_B(c-1) V, S_B(c);
* the two softmax warpgroups: S read, O rescaled in place, P handed over in two
  halves on hardware named barriers, row statistics posted per item;
* the epilogue warpgroup: row statistics and O read, O freed.

Copies complete in any order; the tensor pipe executes MMAs and commits in
issue order.  Every run checks that

* nothing deadlocks;
* a copy-completed barrier is armed only after its previous phase completed;
* no wait meets a barrier two phases ahead (a parity wait would alias), and
  no named barrier gets a second arrival before it was met;
* a copy never overwrites a shared-memory tile that a queued MMA still reads,
  and every MMA reads the tiles it was issued for;
* S/P and O in tensor memory are each written only once the previous reader
  is done (S by its softmax, P by its P V, O by the epilogue), and O is
  rescaled only when every earlier P V into it has executed;
* a row-statistics slot and a tile-count slot are overwritten only after
  they were read.

Planted protocol mistakes (the last value tile armed without waiting for its
barrier's previous phase; a tile-count ring too short) must be caught, so the
model is not vacuous."""
import random

import pytest

STAGES = 2


class Barrier:
    """An mbarrier: `count` arrivals and, for copy barriers, the armed copies
    complete a phase."""

    def __init__(self, name, count=1):
        self.name, self.count = name, count
        self.done = 0          # completed phases
        self.arrived = 0
        self.pending = 0       # copies still in flight for this phase
        self.armed = False

    def arrive(self):
        self.arrived += 1
        self._check()

    def arm(self, copies):
        assert not self.armed, f"{self.name}: armed again before phase {self.done} completed"
        self.armed = True
        self.pending += copies
        self.arrive()

    def copy_done(self):
        self.pending -= 1
        self._check()

    def _check(self):
        if self.arrived >= self.count and self.pending == 0:
            self.done += 1
            self.arrived -= self.count
            self.armed = False

    def passed(self, phase):
        assert self.done <= phase + 1, f"{self.name}: phase {phase} waited when {self.done} done"
        return self.done > phase


class NamedBarrier:
    """A hardware named barrier met by one arrival of the softmax warpgroup
    (bar.arrive) and one of the MMA warp (bar.sync)."""

    def __init__(self, name):
        self.name, self.arrivals, self.met = name, 0, 0

    def arrive(self):
        assert self.arrivals == self.met, f"{self.name}: arrived twice before being met"
        self.arrivals += 1


class Model:
    def __init__(self, items, skew, q_first, seed, plant=None):
        self.rnd = random.Random(seed)
        self.items, self.skew, self.q_first, self.plant = items, skew, q_first, plant
        self.q_full = [Barrier(f"Q_FULL{x}") for x in range(2)]
        self.q_empty = [Barrier(f"Q_EMPTY{x}") for x in range(2)]
        self.k_full = [Barrier(f"K_FULL{s}") for s in range(STAGES)]
        self.kv_empty = [Barrier(f"KV_EMPTY{s}") for s in range(STAGES)]
        self.v_empty = [Barrier(f"V_EMPTY{s}") for s in range(STAGES)]
        self.s_full = [Barrier(f"S_FULL{x}") for x in range(2)]
        self.o_full = [Barrier(f"O_FULL{x}") for x in range(2)]
        self.o_empty = [Barrier(f"O_EMPTY{x}") for x in range(2)]
        self.row_stats = [[Barrier(f"ROW_STATS{x}.{p}") for p in range(2)] for x in range(2)]
        self.p_half = [NamedBarrier(f"P_HALF{x}") for x in range(2)]
        self.p_all = [NamedBarrier(f"P_ALL{x}") for x in range(2)]
        # shared memory: what each tile buffer holds (None while a copy is in flight)
        self.bufs = {"k": [None] * STAGES, "v": [None] * STAGES, "q": [None, None]}
        self.stats = [[None, None], [None, None]]       # [item parity][head]: (item, read)
        self.info_slots = 1 if plant == "short_info_ring" else 4
        self.item_info = [None] * self.info_slots       # (item, tile count, read)
        # tensor memory per head: the S/P columns and O
        self.s_tile = [None, None]       # tile whose S is in the columns
        self.s_read = [True, True]       # its softmax has read it
        self.p_tile = [[None, None], [None, None]]      # tile of each P half
        self.pv_read = [[True, True], [True, True]]     # its P V has read each half
        self.o_item = [None, None]       # item O accumulates
        self.o_read = [True, True]       # the epilogue has read the previous item's O
        self.copies = []                 # in flight: (buffer kind, index, tag, barrier)
        self.pipe = []                   # queued MMAs and commits, in issue order
        self.procs = {"producer": self.producer(), "mma": self.mma(),
                      "softmax0": self.softmax(0), "softmax1": self.softmax(1),
                      "epilogue": self.epilogue()}
        self.waiting = dict.fromkeys(self.procs)

    # ------------------------------------------------------------------ roles
    def load_q(self, it):
        for x in range(2):
            yield ("wait", self.q_empty[x], it - 1)  # item it-1's last S has run
            self.start_copies([("q", x, ("Q", it))], self.q_full[x])

    def producer(self):
        kv_iter = 0
        for it, n in enumerate(self.items):
            if not self.skew:
                slot = it % self.info_slots
                old = self.item_info[slot]
                assert old is None or old[2], f"tile count of item {old[0]} overwritten unread"
                self.item_info[slot] = (it, n, False)
            if self.q_first:
                yield from self.load_q(it)
            for j in range(n):
                st = kv_iter % STAGES
                if self.skew and kv_iter > 0:
                    vc = kv_iter - 1
                    yield ("wait", self.v_empty[vc % STAGES], vc // STAGES - 1)
                yield ("wait", self.kv_empty[st], kv_iter // STAGES - 1)
                copies = [("k", st, ("K", kv_iter))]
                if not self.skew:
                    copies.append(("v", st, ("V", kv_iter)))
                elif kv_iter > 0:
                    copies.append(("v", (kv_iter - 1) % STAGES, ("V", kv_iter - 1)))
                self.start_copies(copies, self.k_full[st])
                kv_iter += 1
                if j == 0 and not self.q_first:
                    yield from self.load_q(it)
        if self.skew:  # the last tile's V, on the barrier of the tile after it
            st, vc = kv_iter % STAGES, kv_iter - 1
            yield ("wait", self.v_empty[vc % STAGES], vc // STAGES - 1)
            if self.plant != "final_v_unguarded":
                yield ("wait", self.kv_empty[st], kv_iter // STAGES - 1)
            self.start_copies([("v", vc % STAGES, ("V", vc))], self.k_full[st])

    def mma(self):
        c = 0
        prev = None
        for it, n in enumerate(self.items):
            count = n if self.skew else 1
            j = 0
            while j < count:
                st = c % STAGES
                if self.skew:
                    yield ("wait", self.k_full[st], c // STAGES)
                for x in range(2):
                    if prev is not None:
                        yield from self.issue_pv(x, prev)
                    if j == 0:
                        yield ("wait", self.q_full[x], it)
                    if x == 0 and not self.skew:
                        yield ("wait", self.k_full[st], c // STAGES)
                        if j == 0:
                            slot = it % self.info_slots
                            tag, count, _ = self.item_info[slot]
                            assert tag == it, f"MMA read the tile count of item {tag} for {it}"
                            self.item_info[slot] = (tag, count, True)
                    last = j == count - 1
                    self.pipe.append(("S", x, c, st, it))
                    self.pipe.append(("commit", self.s_full[x]))
                    if last:
                        self.pipe.append(("commit", self.q_empty[x]))
                    if self.skew and x == 1:
                        self.pipe.append(("commit", self.kv_empty[st]))
                prev = (c, st, it, j == 0, last)
                c += 1
                j += 1
        if self.skew:
            yield ("wait", self.k_full[c % STAGES], c // STAGES)
        for x in range(2):
            yield from self.issue_pv(x, prev)

    def issue_pv(self, x, prev):
        pc, pst, pit, first, last = prev
        yield ("named", self.p_half[x])
        if first:
            yield ("wait", self.o_empty[x], pit - 1)
        self.pipe.append(("PV", x, pc, pst, 0, pit, first))
        yield ("named", self.p_all[x])
        self.pipe.append(("PV", x, pc, pst, 1, pit, False))
        if x == 1:
            self.pipe.append(("commit", (self.v_empty if self.skew else self.kv_empty)[pst]))
        if last:
            self.pipe.append(("commit", self.o_full[x]))

    def softmax(self, x):
        c = 0
        for it, n in enumerate(self.items):
            for j in range(n):
                yield ("wait", self.s_full[x], c)
                assert self.s_tile[x] == c and not self.s_read[x], f"softmax {x}: S of {c} not there"
                self.s_read[x] = True
                if j > 0:  # O may be rescaled in place: every earlier P V into it has run
                    assert not any(op[0] == "PV" and op[1] == x for op in self.pipe), \
                        f"softmax {x}: O rescaled at tile {c} with a P V queued"
                    assert self.o_item[x] == it and not self.o_read[x], f"softmax {x}: O not item {it}'s"
                for h in range(2):
                    assert self.pv_read[x][h], f"P_{x} half {h} overwritten before its P V read it"
                    self.p_tile[x][h], self.pv_read[x][h] = c, False
                    (self.p_half if h == 0 else self.p_all)[x].arrive()
                    yield ("step",)
                c += 1
            old = self.stats[it & 1][x]
            assert old is None or old[1], f"row statistics of item {old[0]} overwritten unread"
            self.stats[it & 1][x] = (it, False)
            self.row_stats[x][it & 1].arrive()

    def epilogue(self):
        for it in range(len(self.items)):
            for x in range(2):
                yield ("wait", self.row_stats[x][it & 1], it >> 1)
                yield ("wait", self.o_full[x], it)
                assert self.stats[it & 1][x] == (it, False), f"epilogue {x}: statistics of {it} not there"
                self.stats[it & 1][x] = (it, True)
                assert self.o_item[x] == it, f"epilogue {x}: O holds item {self.o_item[x]}, not {it}"
                self.o_read[x] = True
                self.o_empty[x].arrive()

    # ------------------------------------------------------------ async units
    def start_copies(self, copies, bar):
        for kind, idx, tag in copies:
            for op in self.pipe:
                assert not self.reads(op, kind, idx), f"copy of {tag} over a tile {op} still reads"
            self.bufs[kind][idx] = None
            self.copies.append((kind, idx, tag, bar))
        bar.arm(len(copies))

    @staticmethod
    def reads(op, kind, idx):
        if op[0] == "S":
            return (kind == "k" and op[3] == idx) or (kind == "q" and op[1] == idx)
        return op[0] == "PV" and kind == "v" and op[3] == idx

    def land_copy(self):
        kind, idx, tag, bar = self.copies.pop(self.rnd.randrange(len(self.copies)))
        self.bufs[kind][idx] = tag
        bar.copy_done()

    def run_pipe(self):
        op = self.pipe.pop(0)
        if op[0] == "commit":
            op[1].arrive()
        elif op[0] == "S":
            _, x, c, st, it = op
            assert self.bufs["k"][st] == ("K", c), f"S_{x}({c}) read {self.bufs['k'][st]}"
            assert self.bufs["q"][x] == ("Q", it), f"S_{x}({c}) read {self.bufs['q'][x]}"
            assert self.s_read[x], f"S_{x}({c}) overwrote the unread S({self.s_tile[x]})"
            assert all(self.pv_read[x]), f"S_{x}({c}) overwrote P before its P V"
            self.s_tile[x], self.s_read[x] = c, False
        else:
            _, x, c, st, h, it, first = op
            assert self.bufs["v"][st] == ("V", c), f"P_{x}({c}) V read {self.bufs['v'][st]}"
            assert self.p_tile[x][h] == c and not self.pv_read[x][h], f"P_{x}({c}) half {h} not there"
            self.pv_read[x][h] = True
            if first:
                assert self.o_read[x], f"O_{x} of item {it} started before the previous one was read"
                self.o_item[x], self.o_read[x] = it, False

    # ------------------------------------------------------------------ driver
    def runnable(self, name):
        w = self.waiting[name]
        if w is None or w[0] == "step":
            return True
        if w[0] == "wait":
            return w[2] < 0 or w[1].passed(w[2])
        return w[1].arrivals > w[1].met  # named barrier: the softmax has arrived

    def advance(self, name):
        w = self.waiting[name]
        if w is not None and w[0] == "named":
            w[1].met += 1
        try:
            self.waiting[name] = next(self.procs[name])
        except StopIteration:
            del self.procs[name]
            del self.waiting[name]

    def run(self):
        for _ in range(100000):
            moves = [("proc", k) for k in self.procs if self.runnable(k)]
            if self.copies:
                moves.append(("copy", None))
            if self.pipe:
                moves.append(("pipe", None))
            if not moves:
                assert not self.procs, f"deadlock: {self.waiting}"
                return
            kind, name = self.rnd.choice(moves)
            if kind == "copy":
                self.land_copy()
            elif kind == "pipe":
                self.run_pipe()
            else:
                self.advance(name)
        raise AssertionError("did not finish")


def random_items(rnd, max_tiles):
    return [rnd.randint(1, max_tiles) for _ in range(rnd.randint(1, 7))]


# (skewed K/V protocol, Q tiles before the first key tile, tiles per item)
PROTOCOLS = {
    "window": (True, False, 5),
    "pattern_skewed": (True, True, 5),
    "pattern_per_tile_stage": (False, True, 2),
}


@pytest.mark.parametrize("name", list(PROTOCOLS))
def test_pair_kernel_protocol_holds_under_random_schedules(name):
    skew, q_first, max_tiles = PROTOCOLS[name]
    for seed in range(400):
        rnd = random.Random(seed)
        Model(random_items(rnd, max_tiles), skew, q_first, seed).run()


@pytest.mark.parametrize("plant,name,expect", [
    ("final_v_unguarded", "window", "armed again"),
    ("short_info_ring", "pattern_per_tile_stage", "tile count"),
])
def test_model_catches_planted_protocol_mistakes(plant, name, expect):
    skew, q_first, max_tiles = PROTOCOLS[name]
    caught = 0
    for seed in range(400):
        rnd = random.Random(seed)
        try:
            Model(random_items(rnd, max_tiles), skew, q_first, seed, plant=plant).run()
        except AssertionError as e:
            assert expect in str(e), e
            caught += 1
    assert caught > 0
