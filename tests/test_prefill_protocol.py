"""The synchronisation protocol of the persistent tcgen05 prefill kernel
(csrc/prefill_tc.cu), checked on the CPU by a randomised discrete-event
model: no deadlock, every mbarrier wait sees exactly the phase it means
(never one two phases later that passes the same parity test), and every
buffer holds the right data whenever a copy, an MMA, the softmax or the
epilogue touches it.

A CTA works through a list of items, each a pair of query tiles attending
the same keys in steps of 64 (ns steps = the longer tile's count; the
shorter tile's extra keys are masked), the rings holding chunks of 128
keys (two steps).  The model follows the kernel's roles and order:
  * a key producer: per item, query tile 0 once tile 0's last S of the
    previous item has completed (q_empty_0), the keys of the first chunk,
    query tile 1 likewise (q_empty_1), then the keys of the other chunks;
    keys of chunk k (counting over the CTA's items) go into ring stage k % 2
    once both tiles have released the stage's previous chunk;
  * a value producer: the values of chunk k into stage k % 2 likewise; for
    a chunk that holds rows past its sequence's end, the copy signals
    v_land, the producer waits for it, clears those rows and then arrives
    on the stage's full barrier itself;
  * one MMA thread per tile with two S buffers: per item S_t(0) into
    buffer 0 and S_t(1) into buffer 1, each followed by a commit into its
    buffer's barrier (C(0), C(1)); then per step u, once the values of u,
    the keys of u + 2 and P_t(u) are in (one P barrier per buffer, so that
    P_t(u + 2) cannot arrive before the thread has taken P_t(u): it needs
    C(u + 2)), P·V_t(u), S_t(u + 2) into the
    buffer P·V_t(u) has just read (while u + 2 < ns) and a commit into
    that buffer's barrier, C(u + 2).  A commit arrives when every MMA the
    thread issued before it is done.  The first P·V of an item overwrites
    O_t without a barrier of its own: it waits for P_t(0), which the
    warpgroup writes only after it has read the previous item's O_t (the
    model checks that it has);
  * per tile a softmax warpgroup takes every commit once, in order: per
    step u it takes C(u) (S_t(u) is in; unless the previous step took it);
    taking C(v) for v >= 2 means P·V_t(v - 2) is done, and after the
    second step of a chunk (or the item's last) the chunk's values are
    free; it releases the keys of a chunk after its second step (or the
    item's last) and, after the item's last S, the query tile (one arrival
    per tile); reads S_t(u), writes P_t(u) over it; if the row's max grew
    it takes C(u + 1) early (P·V_t(u - 1) is done) and rescales O_t;
    arrives (one arrival per warp); after the item's last step it takes
    C(ns) and C(ns + 1) (the last P·V), reads O_t, then stages its rows in
    the output buffer the two tiles share in turns (tile 0 of an item, tile
    1, tile 0 of the next, ..., each turn waiting for the previous one's
    end on out_free) for a TMA store.
    The two warpgroups run independently of each other;
  * the tensor pipe runs the operations in issue order, a commit arriving
    when everything issued before it has completed.
TMA copies, MMAs and the softmax take random times.  Planted mistakes (a
stage of keys released by one tile alone, keys released after a chunk's
first step, values released after a chunk's first P·V, S issued before the
P·V that reads the buffer it overwrites, O rescaled without waiting for
the previous P·V, both buffers' P on one barrier, a tile staging its rows
without waiting for its turn, an epilogue without its wait, a producer waiting on the wrong parity, query tiles reloaded without
waiting for q_empty, values never released by one tile, rows cleared before
their copy has landed) show that the checks catch each kind of failure:
stale data, a deadlock."""

import pytest

from tests._event_sim import Bar, EventSim

K_STAGES, V_STAGES = 2, 2


class Sim(EventSim):
    def __init__(self, items, seed, mutate=None):
        super().__init__(seed)
        self.items = [tuple(x) for x in items]  # (steps of tile 0, steps of tile 1); both tiles run the longer
        # the last chunk of every other item holds rows past its sequence's end
        self.clears = [i % 2 == 1 for i in range(len(self.items))]
        self.mutate = mutate
        # the stage and query-tile releases take one arrival from each tile's softmax
        self.full_k = [Bar(f"full_k{i}", 1) for i in range(K_STAGES)]
        self.empty_k = [Bar(f"empty_k{i}", 1 if mutate == "k_count_one" else 2) for i in range(K_STAGES)]
        self.full_v = [Bar(f"full_v{i}", 1) for i in range(V_STAGES)]
        self.empty_v = [Bar(f"empty_v{i}", 2) for i in range(V_STAGES)]
        self.v_land = Bar("v_land", 1)
        self.out_free = Bar("out_free", 1)  # turns on the output staging buffer: tile 0, tile 1, tile 0, ...
        self.out_owner = None
        self.s_full = [[Bar(f"s_full{t}.{b}", 1) for b in range(2)] for t in range(2)]
        self.p_full = [[Bar(f"p_full{t}.{b}", 4) for b in range(2)] for t in range(2)]
        if mutate == "one_p_barrier":  # both buffers' P on one barrier
            self.p_full = [[self.p_full[t][0]] * 2 for t in range(2)]
        self.q_full = [Bar(f"q_full{t}", 1) for t in range(2)]
        self.q_empty = [Bar(f"q_empty{t}", 1) for t in range(2)]
        # buffer contents, tagged (item, chunk) for the rings, (item, step) for S / P
        self.k_stage = [None] * K_STAGES
        self.v_stage = [None] * V_STAGES
        self.v_clean = [True] * V_STAGES  # rows past the sequence's end hold no stale copy
        self.k_busy = [0] * K_STAGES  # S operations reading the stage right now
        self.v_busy = [0] * V_STAGES  # P·V operations reading the stage right now
        self.q_tile = [None, None]  # item whose query tile has landed
        self.s_buf = [[None, None], [None, None]]  # per tile and buffer: ("S", i, u) or ("P", i, u)
        self.o_last = [None, None]  # (item, last step accumulated into O_t)
        self.o_busy = [False, False]  # a P·V of the tile is running
        self.o_read = [None, None]  # item whose O_t the epilogue has read
        self.pipe_free = 0.0

    @staticmethod
    def steps(item):
        return max(item)

    def run(self):
        roles = [self.key_producer(), self.value_producer(), self.mma(0), self.mma(1), self.softmax(0),
                 self.softmax(1)]
        return self.run_roles(roles, {"kp", "vp", "mma0", "mma1", "sm0", "sm1"})

    # --- copies and the tensor pipe ---
    def pipe(self, duration, start, end):
        # one tensor pipe, operations in issue order (that keeps each thread's
        # own operations in order too)
        t0 = max(self.now, self.pipe_free)
        self.pipe_free = t0 + duration
        self.at(t0, start)
        self.at(t0 + duration, end)

    def commit(self, bar):
        self.pipe(0.0, lambda: None, lambda: self.arrive(bar))

    # --- roles ---
    def load_q(self, i, t):
        if i > 0 and self.mutate != "no_q_empty_wait":
            yield ("wait", self.q_empty[t], (i - 1) & 1, i, f"key producer q_empty{t} item {i}")
        self.expect_tx(self.q_full[t], 2)
        self.copy(self.q_full[t], 2, lambda t=t, i=i: self.q_tile.__setitem__(t, i))

    def key_producer(self):
        k = 0
        for i, item in enumerate(self.items):
            nch = (self.steps(item) + 1) // 2
            yield from self.load_q(i, 0)
            for c in range(nch):
                if c == 1:
                    yield from self.load_q(i, 1)
                st = k % K_STAGES
                flip = 0 if self.mutate == "producer_parity" else 1
                yield ("wait", self.empty_k[st], ((k // K_STAGES) & 1) ^ flip, k // K_STAGES, f"key producer {i}.{c}")
                if self.k_busy[st]:
                    self.fail(f"keys {i}.{c} copied into stage {st} while an S reads it")
                self.expect_tx(self.full_k[st], 1)
                self.copy(self.full_k[st], 1, lambda st=st, tag=(i, c): self.k_stage.__setitem__(st, tag))
                k += 1
                yield ("delay", self.rng.uniform(0.0, 0.5))
            if nch == 1:
                yield from self.load_q(i, 1)
        self.done.add("kp")

    def value_producer(self):
        k, vl = 0, 0
        for i, item in enumerate(self.items):
            n = (self.steps(item) + 1) // 2
            for c in range(n):
                st = k % V_STAGES
                yield ("wait", self.empty_v[st], ((k // V_STAGES) & 1) ^ 1, k // V_STAGES, f"value producer {i}.{c}")
                if self.v_busy[st]:
                    self.fail(f"values {i}.{c} copied into stage {st} while a P·V reads it")
                clear = self.clears[i] and c == n - 1

                def land(st=st, tag=(i, c), clear=clear):
                    self.v_stage[st] = tag
                    self.v_clean[st] = not clear  # the copy brings rows past the sequence's end

                if clear:
                    self.expect_tx(self.v_land, 1)
                    self.copy(self.v_land, 1, land)
                    if self.mutate != "no_land_wait":
                        yield ("wait", self.v_land, vl & 1, vl + 1, f"value producer land {i}.{c}")
                    vl += 1
                    yield ("delay", self.rng.uniform(0.1, 0.6))  # clear the rows
                    self.v_clean[st] = True
                    self.arrive(self.full_v[st])
                else:
                    self.expect_tx(self.full_v[st], 1)
                    self.copy(self.full_v[st], 1, land)
                k += 1
                yield ("delay", self.rng.uniform(0.0, 0.5))
        self.done.add("vp")

    def issue_s(self, i, t, u, kst, b):
        def start():
            if self.q_tile[t] != i:
                self.fail(f"S{t}({i}.{u}) reads the query tile of item {self.q_tile[t]}")
            if self.k_stage[kst] != (i, u // 2):
                self.fail(f"S{t}({i}.{u}) starts on keys {self.k_stage[kst]}")
            self.k_busy[kst] += 1

        def end():
            self.k_busy[kst] -= 1
            if self.k_stage[kst] != (i, u // 2):
                self.fail(f"S{t}({i}.{u}): keys of stage {kst} overwritten while it ran")
            if self.q_tile[t] != i:
                self.fail(f"S{t}({i}.{u}): query tile overwritten while it ran")
            self.s_buf[t][b] = ("S", i, u)

        self.pipe(self.rng.uniform(0.2, 1.0), start, end)

    def issue_pv(self, i, t, u, vst, b):
        def start():
            if self.s_buf[t][b] != ("P", i, u):
                self.fail(f"PV{t}({i}.{u}) reads {self.s_buf[t][b]} instead of P")
            if self.v_stage[vst] != (i, u // 2):
                self.fail(f"PV{t}({i}.{u}) starts on values {self.v_stage[vst]}")
            if not self.v_clean[vst]:
                self.fail(f"PV{t}({i}.{u}) reads rows past the sequence's end before they were cleared")
            if u > 0 and self.o_last[t] != (i, u - 1):
                self.fail(f"PV{t}({i}.{u}) accumulates onto O holding {self.o_last[t]}")
            if u == 0 and self.o_last[t] is not None and self.o_read[t] != self.o_last[t][0]:
                self.fail(f"PV{t}({i}.0) overwrites O of item {self.o_last[t][0]} before the epilogue read it")
            self.o_busy[t] = True
            self.v_busy[vst] += 1

        def end():
            self.v_busy[vst] -= 1
            if self.v_stage[vst] != (i, u // 2) or self.s_buf[t][b] != ("P", i, u):
                self.fail(f"PV{t}({i}.{u}): operands overwritten while it ran")
            self.o_last[t] = (i, u)
            self.o_busy[t] = False

        self.pipe(self.rng.uniform(0.2, 1.0), start, end)

    def mma(self, t):
        """MMA thread of tile t: its S and P·V for every step of every item."""
        kq, spc, it = 0, [0, 0], 0
        for i, item in enumerate(self.items):
            ns = self.steps(item)
            yield ("wait", self.q_full[t], it & 1, it + 1, f"mma{t} q item {i}")
            yield ("wait", self.full_k[kq % K_STAGES], (kq // K_STAGES) & 1, kq // K_STAGES + 1, f"mma{t} k {i}.0")
            self.issue_s(i, t, 0, kq % K_STAGES, 0)
            self.commit(self.s_full[t][0])
            if ns > 1:
                self.issue_s(i, t, 1, kq % K_STAGES, 1)
                self.commit(self.s_full[t][1])
            for u in range(ns):
                b = u & 1
                vc, kc = kq + u // 2, kq + (u + 2) // 2
                more = u + 2 < ns
                if b == 0:
                    yield ("wait", self.full_v[vc % V_STAGES], (vc // V_STAGES) & 1, vc // V_STAGES + 1,
                           f"mma{t} v {i}.{u}")
                if more and b == 0:
                    yield ("wait", self.full_k[kc % K_STAGES], (kc // K_STAGES) & 1, kc // K_STAGES + 1,
                           f"mma{t} k {i}.{u + 2}")
                yield ("wait", self.p_full[t][b], spc[b] & 1, spc[b] + 1, f"mma{t} p {i}.{u}")
                spc[b] += 1
                if self.mutate == "s_before_pv" and more:
                    self.issue_s(i, t, u + 2, kc % K_STAGES, b)
                    self.issue_pv(i, t, u, vc % V_STAGES, b)
                else:
                    self.issue_pv(i, t, u, vc % V_STAGES, b)
                    if more:
                        self.issue_s(i, t, u + 2, kc % K_STAGES, b)
                self.commit(self.s_full[t][b])
                yield ("delay", self.rng.uniform(0.0, 0.3))
            kq += (ns + 1) // 2
            it += 1
        self.done.add(f"mma{t}")

    def rescale(self, i, t, u):
        if self.o_busy[t] or self.o_last[t] != (i, u - 1):
            self.fail(f"softmax{t}({i}.{u}) rescales O holding {self.o_last[t]} (P·V running: {self.o_busy[t]})")
        yield ("delay", self.rng.uniform(0.2, 0.8))
        if self.o_busy[t] or self.o_last[t] != (i, u - 1):
            self.fail(f"softmax{t}({i}.{u}): O changed while it was rescaled")

    def softmax(self, t):
        sfc, ch, done = [0, 0], 0, 0
        one_tile_v = self.mutate == "v_release_one_tile" and t == 0

        def take(i, v, ns):
            """Commit C(v): everything the MMA thread issued before it is done."""
            yield ("wait", self.s_full[t][v & 1], sfc[v & 1] & 1, sfc[v & 1] + 1, f"softmax{t} C({i}.{v})")
            sfc[v & 1] += 1
            pw = v - 2  # P·V(pw) is done
            early = self.mutate == "v_release_early"
            if pw >= 0 and not one_tile_v and ((pw % 2 == 0 and pw != ns - 1) if early else (pw & 1 or pw == ns - 1)):
                self.arrive(self.empty_v[(ch + pw // 2) % V_STAGES])

        for i, item in enumerate(self.items):
            ns = self.steps(item)
            ahead = False
            for u in range(ns):
                b = u & 1
                if not ahead:
                    yield from take(i, u, ns)
                ahead = False
                # S(u) is done: the keys of a chunk are free after its second
                # step (or the item's last), the query tile after the last S
                release_k = b == 0 if self.mutate == "k_release_early" else (b == 1 or u + 1 == ns)
                if release_k:
                    self.arrive(self.empty_k[(ch + u // 2) % K_STAGES])
                if u + 1 == ns:
                    self.arrive(self.q_empty[t])
                if self.s_buf[t][b] != ("S", i, u):
                    self.fail(f"softmax{t}({i}.{u}) reads {self.s_buf[t][b]}")
                yield ("delay", self.rng.uniform(0.1, 0.6))  # tensor-memory loads of S
                if self.s_buf[t][b] != ("S", i, u):
                    self.fail(f"softmax{t}({i}.{u}): S overwritten while it was read")
                yield ("delay", self.rng.uniform(0.3, 2.5))  # the exponentials
                self.s_buf[t][b] = ("P", i, u)
                if u > 0 and self.rng.random() < 0.4:  # the row's max grew: rescale O
                    if self.mutate != "no_early_take":
                        yield from take(i, u + 1, ns)
                        ahead = True
                    yield from self.rescale(i, t, u)
                self.arrive(self.p_full[t][b], 4)
            if self.mutate != "no_final_wait":
                if ns > 1 and not ahead:
                    yield from take(i, ns, ns)
                yield from take(i, ns + 1, ns)
            if self.o_last[t] != (i, ns - 1):
                self.fail(f"epilogue {t} of item {i} reads O holding {self.o_last[t]}")
            yield ("delay", self.rng.uniform(0.2, 1.5))  # tensor-memory loads of O
            if self.o_last[t] != (i, ns - 1):
                self.fail(f"epilogue {t} of item {i}: O changed while it was read")
            self.o_read[t] = i
            ch += (ns + 1) // 2
            # the output staging buffer, the two tiles' in turn
            turn = 2 * done + t
            done += 1
            if turn > 0 and self.mutate != "no_turn_wait":
                yield ("wait", self.out_free, (turn - 1) & 1, turn, f"softmax{t} staging turn {i}")
            if self.out_owner is not None:
                self.fail(f"epilogue {t} of item {i} stages its rows while tile {self.out_owner} uses the buffer")
            self.out_owner = t
            yield ("delay", self.rng.uniform(0.5, 3.0))  # stage the rows, the TMA store reads them
            self.out_owner = None
            self.arrive(self.out_free)
        self.done.add(f"sm{t}")


# Item lists a CTA may get: (steps of tile 0, steps of tile 1), 64 keys a
# step.  The later tile attends as many steps or more; a sequence's last
# pair may have one tile.  Lists mix single-step items, items with an odd
# number of steps (a chunk of keys with one step), items longer than every
# ring and one-tile items.
ITEM_LISTS = [
    [(1, 1)],
    [(1, 0)],
    [(2, 2)],
    [(16, 16)],
    [(1, 1), (1, 1), (1, 1)],
    [(5, 6), (3, 0), (9, 9)],
    [(15, 16), (13, 15), (1, 0), (7, 8), (1, 3)],
    [(1, 0), (2, 0), (3, 4), (1, 0)],
    [(11, 13), (5, 6), (6, 7), (3, 4), (2, 2), (1, 0)],
    [(3, 5)] * 5,
    [(9, 0), (10, 11)],
]


@pytest.mark.parametrize("items", ITEM_LISTS, ids=lambda s: "-".join(f"{a}x{b}" for a, b in s))
def test_prefill_protocol_is_race_free(items):
    for seed in range(80):
        v = Sim(items, seed).run()
        assert not v, f"seed {seed}: {v[:3]}"


@pytest.mark.parametrize("mutate", ["k_count_one", "k_release_early", "v_release_early", "s_before_pv",
                                    "no_early_take", "one_p_barrier", "no_turn_wait", "no_final_wait", "producer_parity",
                                    "no_q_empty_wait", "v_release_one_tile", "no_land_wait"])
def test_planted_protocol_mistakes_are_caught(mutate):
    caught = 0
    for items in ([(5, 6), (9, 11)], [(16, 16), (3, 3), (7, 8)], [(1, 1)] * 4, [(4, 4), (1, 0), (5, 6)]):
        for seed in range(30):
            caught += bool(Sim(items, seed, mutate).run())
    assert caught > 0
