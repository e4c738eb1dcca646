"""The synchronisation protocol of the persistent tcgen05 prefill kernel
(csrc/prefill_tc.cu), checked on the CPU by a randomised discrete-event
model: no deadlock, every mbarrier wait sees exactly the phase it means
(never one two phases later that passes the same parity test), and every
buffer holds the right data whenever a copy, an MMA, the softmax or the
epilogue touches it.

A CTA works through a list of items, each a pair of query tiles attending
the same chunks of keys (nch = the longer tile's count; the shorter tile's
extra keys are masked).  The model follows the kernel's roles and order:
  * a key producer: per item, query tile 0 once tile 0's last S of the
    previous item has completed (q_empty_0), the keys of the first chunk,
    query tile 1 likewise (q_empty_1), then the keys of the other chunks;
    keys of chunk k (counting over the CTA's items) go into ring stage k % 2
    once both tiles have released the stage's previous chunk;
  * a value producer: the values of chunk k into stage k % 3 likewise; for
    a chunk that holds rows past its sequence's end, the copy signals
    v_land, the producer waits for it, clears those rows and then arrives
    on the stage's full barrier itself;
  * one MMA thread per tile: per item S_t(0), then per chunk c, once the
    keys of chunk c + 1 and P_t(c) are in, P·V_t(c) and S_t(c+1); a commit signals S_t(c) (it arrives when
    every MMA the thread issued before it is done, so it also covers
    P·V_t(c-1)) and, after the item's last P·V, o_final.  The first P·V of an
    item overwrites O_t without a barrier of its own: it waits for P_t(0),
    which the warpgroup writes only after it has read the previous item's
    O_t (the model checks that it has);
  * per tile a softmax warpgroup: wait for S_t(c); release the keys of chunk
    c, the values of chunk c - 1 and, after the item's last S, its query
    tile (one arrival per tile); wait for its turn (the two warpgroups take
    strict turns, tile 0's chunk k before tile 1's chunk k before tile 0's
    chunk k + 1); rescale O_t (the commit that signalled S_t(c) covers
    P·V_t(c-1)), write P_t(c) over S_t, arrive (one arrival per warp), pass
    the turn; after the item's last chunk wait for its last P·V, release its
    values, read O_t, then store the rows;
  * the tensor pipe runs the operations in issue order, a commit arriving
    when everything issued before it has completed.
TMA copies, MMAs and the softmax take random times.  Planted mistakes (a
stage of keys released by one tile alone, keys released before their S has
run, S issued before the P·V that reads the buffer it overwrites, an
epilogue without its wait, a producer waiting on the wrong parity, query
tiles reloaded without waiting for q_empty, values never released by one
tile, rows cleared before their copy has landed) show that the checks
catch each kind of failure: stale data, a deadlock."""

import pytest

from tests._event_sim import Bar, EventSim

K_STAGES, V_STAGES = 2, 3


class Sim(EventSim):
    def __init__(self, items, seed, mutate=None):
        super().__init__(seed)
        self.items = [tuple(x) for x in items]  # (nch0, nch1) per item, nch1 <= nch0 only if nch1 == 0
        # the last chunk of every other item holds rows past its sequence's end
        self.clears = [i % 2 == 1 for i in range(len(self.items))]
        self.mutate = mutate
        # the stage and query-tile releases take one arrival from each tile's softmax
        self.full_k = [Bar(f"full_k{i}", 1) for i in range(K_STAGES)]
        self.empty_k = [Bar(f"empty_k{i}", 1 if mutate == "k_count_one" else 2) for i in range(K_STAGES)]
        self.full_v = [Bar(f"full_v{i}", 1) for i in range(V_STAGES)]
        self.empty_v = [Bar(f"empty_v{i}", 2) for i in range(V_STAGES)]
        self.v_land = Bar("v_land", 1)
        self.s_full = [Bar(f"s_full{t}", 1) for t in range(2)]
        self.p_full = [Bar(f"p_full{t}", 4) for t in range(2)]
        self.o_final = [Bar(f"o_final{t}", 1) for t in range(2)]
        self.q_full = [Bar(f"q_full{t}", 1) for t in range(2)]
        self.q_empty = [Bar(f"q_empty{t}", 1) for t in range(2)]
        # softmax turns: tile 0's chunk k, tile 1's chunk k, tile 0's chunk k + 1, ...
        self.turn = [Bar(f"turn{t}", 4) for t in range(2)]
        # buffer contents, tagged (item, chunk)
        self.k_stage = [None] * K_STAGES
        self.v_stage = [None] * V_STAGES
        self.v_clean = [True] * V_STAGES  # rows past the sequence's end hold no stale copy
        self.k_busy = [0] * K_STAGES  # S operations reading the stage right now
        self.q_tile = [None, None]  # item whose query tile has landed
        self.s_buf = [None, None]  # ("S", i, c) or ("P", i, c)
        self.o_last = [None, None]  # (item, last chunk accumulated into O_t)
        self.o_read = [None, None]  # item whose O_t the epilogue has read
        self.pipe_free = 0.0

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
        for i, nch in enumerate(self.items):
            yield from self.load_q(i, 0)
            for c in range(max(nch)):
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
            if max(nch) == 1:
                yield from self.load_q(i, 1)
        self.done.add("kp")

    def value_producer(self):
        k, vl = 0, 0
        for i, nch in enumerate(self.items):
            n = max(nch)
            for c in range(n):
                st = k % V_STAGES
                yield ("wait", self.empty_v[st], ((k // V_STAGES) & 1) ^ 1, k // V_STAGES, f"value producer {i}.{c}")
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

    def issue_s(self, i, t, c, kst):
        def start():
            if self.q_tile[t] != i:
                self.fail(f"S{t}({i}.{c}) reads the query tile of item {self.q_tile[t]}")
            if self.k_stage[kst] != (i, c):
                self.fail(f"S{t}({i}.{c}) starts on keys {self.k_stage[kst]}")
            self.k_busy[kst] += 1

        def end():
            self.k_busy[kst] -= 1
            if self.k_stage[kst] != (i, c):
                self.fail(f"S{t}({i}.{c}): keys of stage {kst} overwritten while it ran")
            if self.q_tile[t] != i:
                self.fail(f"S{t}({i}.{c}): query tile overwritten while it ran")
            self.s_buf[t] = ("S", i, c)

        self.pipe(self.rng.uniform(0.3, 2.0), start, end)
        self.commit(self.s_full[t])

    def issue_pv(self, i, t, c, vst):
        nch_t = max(self.items[i])

        def start():
            if self.s_buf[t] != ("P", i, c):
                self.fail(f"PV{t}({i}.{c}) reads {self.s_buf[t]} instead of P")
            if self.v_stage[vst] != (i, c):
                self.fail(f"PV{t}({i}.{c}) starts on values {self.v_stage[vst]}")
            if not self.v_clean[vst]:
                self.fail(f"PV{t}({i}.{c}) reads rows past the sequence's end before they were cleared")
            if c > 0 and self.o_last[t] != (i, c - 1):
                self.fail(f"PV{t}({i}.{c}) accumulates onto O holding {self.o_last[t]}")
            if c == 0 and self.o_last[t] is not None and self.o_read[t] != self.o_last[t][0]:
                self.fail(f"PV{t}({i}.0) overwrites O of item {self.o_last[t][0]} before the epilogue read it")

        def end():
            if self.v_stage[vst] != (i, c) or self.s_buf[t] != ("P", i, c):
                self.fail(f"PV{t}({i}.{c}): operands overwritten while it ran")
            self.o_last[t] = (i, c)

        self.pipe(self.rng.uniform(0.3, 2.0), start, end)
        if c + 1 == nch_t:
            self.commit(self.o_final[t])

    def mma(self, t):
        """MMA thread of tile t: its S and P·V for every chunk of every item."""
        kq, vq, sp, it = 0, 0, 0, 0
        for i, nch in enumerate(self.items):
            n = max(nch)
            yield ("wait", self.q_full[t], it & 1, it + 1, f"mma{t} q item {i}")
            yield ("wait", self.full_k[kq % K_STAGES], (kq // K_STAGES) & 1, kq // K_STAGES + 1, f"mma{t} k {i}.0")
            self.issue_s(i, t, 0, kq % K_STAGES)
            kq += 1
            for c in range(n):
                vst = vq % V_STAGES
                yield ("wait", self.full_v[vst], (vq // V_STAGES) & 1, vq // V_STAGES + 1, f"mma{t} v {i}.{c}")
                if c + 1 < n:
                    yield ("wait", self.full_k[kq % K_STAGES], (kq // K_STAGES) & 1, kq // K_STAGES + 1,
                           f"mma{t} k {i}.{c + 1}")
                yield ("wait", self.p_full[t], sp & 1, sp + 1, f"mma{t} p {i}.{c}")
                sp += 1
                if self.mutate == "s_before_pv" and c + 1 < n:
                    self.issue_s(i, t, c + 1, kq % K_STAGES)
                    self.issue_pv(i, t, c, vst)
                    kq += 1
                    vq += 1
                    continue
                self.issue_pv(i, t, c, vst)
                vq += 1
                if c + 1 < n:
                    self.issue_s(i, t, c + 1, kq % K_STAGES)
                    kq += 1
                yield ("delay", self.rng.uniform(0.0, 0.3))
            it += 1
        self.done.add(f"mma{t}")

    def softmax(self, t):
        sc, ot = 0, 0
        early_k = self.mutate == "k_release_early" and t == 0
        for i, nch in enumerate(self.items):
            n = max(nch)
            for c in range(n):
                if early_k:  # releases the keys before S has run on them
                    self.arrive(self.empty_k[sc % K_STAGES])
                yield ("wait", self.s_full[t], sc & 1, sc + 1, f"softmax{t} s {i}.{c}")
                # S(c) is done: the keys of chunk c, the values of chunk c - 1
                # (the commit covers P·V(c - 1)) and, after the last S, the
                # query tiles are free as far as this tile is concerned
                if not early_k:
                    self.arrive(self.empty_k[sc % K_STAGES])
                if c > 0 and not (self.mutate == "v_release_one_tile" and t == 0):
                    self.arrive(self.empty_v[(sc - 1) % V_STAGES])
                if c + 1 == n:
                    self.arrive(self.q_empty[t])
                # strict alternation of the two warpgroups' softmax turns
                if t == 0 and sc > 0:
                    yield ("wait", self.turn[0], (sc - 1) & 1, sc, f"softmax0 turn {i}.{c}")
                elif t == 1:
                    yield ("wait", self.turn[1], sc & 1, sc + 1, f"softmax1 turn {i}.{c}")
                sc += 1
                if self.s_buf[t] != ("S", i, c):
                    self.fail(f"softmax{t}({i}.{c}) reads {self.s_buf[t]}")
                if c > 0 and self.o_last[t] != (i, c - 1):
                    self.fail(f"softmax{t}({i}.{c}) rescales O holding {self.o_last[t]}")
                yield ("delay", self.rng.uniform(0.5, 4.0))
                if self.s_buf[t] != ("S", i, c):
                    self.fail(f"softmax{t}({i}.{c}): S overwritten while it was read")
                self.s_buf[t] = ("P", i, c)
                self.arrive(self.p_full[t], 4)
                self.arrive(self.turn[1 - t], 4)
            if self.mutate != "no_final_wait":
                yield ("wait", self.o_final[t], ot & 1, ot + 1, f"softmax{t} epilogue {i}")
            if not (self.mutate == "v_release_one_tile" and t == 0):
                self.arrive(self.empty_v[(sc - 1) % V_STAGES])
            if self.o_last[t] != (i, n - 1):
                self.fail(f"epilogue {t} of item {i} reads O holding {self.o_last[t]}")
            yield ("delay", self.rng.uniform(0.2, 1.5))  # tensor-memory loads of O
            if self.o_last[t] != (i, n - 1):
                self.fail(f"epilogue {t} of item {i}: O changed while it was read")
            self.o_read[t] = i
            ot += 1
            yield ("delay", self.rng.uniform(0.5, 3.0))  # normalise and store the rows
        self.done.add(f"sm{t}")


# Item lists a CTA may get: (chunks of tile 0, chunks of tile 1).  The later
# tile attends as many chunks or one more; a sequence's last pair may have
# one tile.  Lists mix single-chunk items, items longer than every ring and
# one-tile items.
ITEM_LISTS = [
    [(1, 1)],
    [(1, 0)],
    [(8, 8)],
    [(1, 1), (1, 1), (1, 1)],
    [(3, 4), (2, 0), (5, 5)],
    [(8, 8), (7, 8), (1, 0), (4, 4), (1, 2)],
    [(1, 0), (1, 0), (2, 2), (1, 0)],
    [(6, 7), (3, 3), (3, 4), (2, 2), (1, 1), (1, 0)],
    [(2, 3)] * 5,
    [(5, 0), (5, 6)],
]


@pytest.mark.parametrize("items", ITEM_LISTS, ids=lambda s: "-".join(f"{a}x{b}" for a, b in s))
def test_prefill_protocol_is_race_free(items):
    for seed in range(40):
        v = Sim(items, seed).run()
        assert not v, f"seed {seed}: {v[:3]}"


@pytest.mark.parametrize("mutate", ["k_count_one", "k_release_early", "s_before_pv", "no_final_wait",
                                    "producer_parity", "no_q_empty_wait", "v_release_one_tile", "no_land_wait"])
def test_planted_protocol_mistakes_are_caught(mutate):
    caught = 0
    for items in ([(3, 3), (5, 6)], [(8, 8), (2, 2), (4, 4)], [(1, 1)] * 4, [(2, 2), (1, 0), (3, 3)]):
        for seed in range(30):
            caught += bool(Sim(items, seed, mutate).run())
    assert caught > 0
