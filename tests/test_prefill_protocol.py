"""The synchronisation protocol of the tcgen05 prefill kernel
(csrc/prefill_tc.cu), checked on the CPU by a randomised discrete-event
model: no deadlock, every mbarrier wait sees exactly the phase it means
(never one two phases later that passes the same parity test), and every
buffer holds the right data whenever a copy, an MMA, the softmax or the
epilogue touches it.

The model follows the kernel's roles and its order of operations:
  * a key producer: both query tiles, then the keys of chunk c into ring
    stage c % 3 once the stage's previous chunk has been released;
  * a value producer: the values of chunk c into stage c % 2 likewise;
  * one MMA thread: S of both tiles for chunk 0, then per chunk c and tile t
    (if the tile attends chunk c) P·V_t(c) once P_t(c) is in, then S_t(c+1);
    a stage is released by a commit after the last MMA that reads it;
  * per tile a softmax: wait for S_t(c), rescale O_t at once (the commit
    that released S_t(c) covers P·V_t(c-1)), write P_t(c) over S_t, arrive;
    after the last chunk wait for the tile's last P·V and read O_t;
  * the tensor pipe runs the MMA thread's operations in issue order, a
    commit arriving when everything issued before it has completed.
TMA copies and MMAs take random times; planted mistakes (a stage of keys
released after the first of its two readers, S issued before the P·V that
reads the buffer it overwrites, an epilogue without its wait, a producer
waiting on the wrong parity) show that the checks catch each kind of
failure: stale data, a deadlock."""

import pytest

from tests._event_sim import Bar, EventSim

K_STAGES, V_STAGES = 3, 2


class Sim(EventSim):
    def __init__(self, nch, seed, mutate=None):
        super().__init__(seed)
        self.nch = nch  # chunks each tile attends (0: no such tile)
        self.n = max(nch)
        self.mutate = mutate
        self.full_k = [Bar(f"full_k{i}", 1) for i in range(K_STAGES)]
        self.empty_k = [Bar(f"empty_k{i}", 1) for i in range(K_STAGES)]
        self.full_v = [Bar(f"full_v{i}", 1) for i in range(V_STAGES)]
        self.empty_v = [Bar(f"empty_v{i}", 1) for i in range(V_STAGES)]
        self.s_full = [Bar(f"s_full{t}", 1) for t in range(2)]
        self.p_full = [Bar(f"p_full{t}", 128) for t in range(2)]
        self.o_final = [Bar(f"o_final{t}", 1) for t in range(2)]
        self.q_full = [Bar(f"q_full{t}", 1) for t in range(2)]
        # buffer contents
        self.k_stage = [None] * K_STAGES
        self.v_stage = [None] * V_STAGES
        self.q_tile = [False, False]
        self.s_buf = [None, None]  # ("S", c) or ("P", c)
        self.o_last = [-1, -1]  # last chunk accumulated into O_t
        self.pipe_free = 0.0

    def run(self):
        roles = [self.key_producer(), self.value_producer(), self.mma()]
        roles += [self.softmax(t) for t in range(2) if self.nch[t] > 0]
        return self.run_roles(roles, {"kp", "vp", "mma"} | {f"sm{t}" for t in range(2) if self.nch[t] > 0})

    # --- copies and the tensor pipe ---
    def pipe(self, duration, start, end):
        t0 = max(self.now, self.pipe_free)
        self.pipe_free = t0 + duration
        self.at(t0, start)
        self.at(t0 + duration, end)

    def commit(self, bar):
        self.pipe(0.0, lambda: None, lambda: self.arrive(bar))

    # --- roles ---
    def key_producer(self):
        for t in range(2):
            if self.nch[t]:
                self.expect_tx(self.q_full[t], 2)
                self.copy(self.q_full[t], 2, lambda t=t: self.q_tile.__setitem__(t, True))
        for c in range(self.n):
            st = c % K_STAGES
            flip = 0 if self.mutate == "producer_parity" else 1
            yield ("wait", self.empty_k[st], ((c // K_STAGES) & 1) ^ flip, c // K_STAGES, f"key producer c{c}")
            self.expect_tx(self.full_k[st], 1)
            self.copy(self.full_k[st], 1, lambda st=st, c=c: self.k_stage.__setitem__(st, c))
            yield ("delay", self.rng.uniform(0.0, 0.5))
        self.done.add("kp")

    def value_producer(self):
        for c in range(self.n):
            st = c % V_STAGES
            yield ("wait", self.empty_v[st], ((c // V_STAGES) & 1) ^ 1, c // V_STAGES, f"value producer c{c}")
            self.expect_tx(self.full_v[st], 1)
            self.copy(self.full_v[st], 1, lambda st=st, c=c: self.v_stage.__setitem__(st, c))
            yield ("delay", self.rng.uniform(0.0, 0.5))
        self.done.add("vp")

    def issue_s(self, t, c):
        st = c % K_STAGES

        def start():
            if not self.q_tile[t]:
                self.fail(f"S{t}({c}) reads a query tile that has not landed")
            if self.k_stage[st] != c:
                self.fail(f"S{t}({c}) starts on keys of chunk {self.k_stage[st]}")

        def end():
            if self.k_stage[st] != c:
                self.fail(f"S{t}({c}): keys of stage {st} overwritten while it ran")
            self.s_buf[t] = ("S", c)

        self.pipe(self.rng.uniform(0.3, 2.0), start, end)
        self.commit(self.s_full[t])

    def issue_pv(self, t, c):
        st = c % V_STAGES

        def start():
            if self.s_buf[t] != ("P", c):
                self.fail(f"PV{t}({c}) reads {self.s_buf[t]} instead of P({c})")
            if self.v_stage[st] != c:
                self.fail(f"PV{t}({c}) starts on values of chunk {self.v_stage[st]}")
            if self.o_last[t] != c - 1:
                self.fail(f"PV{t}({c}) accumulates onto O holding chunk {self.o_last[t]}")

        def end():
            if self.v_stage[st] != c or self.s_buf[t] != ("P", c):
                self.fail(f"PV{t}({c}): operands overwritten while it ran")
            self.o_last[t] = c

        self.pipe(self.rng.uniform(0.3, 2.0), start, end)
        if c + 1 == self.nch[t]:
            self.commit(self.o_final[t])

    def mma(self):
        nch = self.nch
        for t in range(2):
            if nch[t]:
                yield ("wait", self.q_full[t], 0, 1, f"mma q{t}")
        yield ("wait", self.full_k[0], 0, 1, "mma k0")
        for t in range(2):
            if nch[t]:
                self.issue_s(t, 0)
        self.commit(self.empty_k[0])
        for c in range(self.n):
            yield ("wait", self.full_v[c % V_STAGES], (c // V_STAGES) & 1, c // V_STAGES + 1, f"mma v{c}")
            k_next = False
            tiles = [1, 0] if self.mutate == "release_k_after_first" else [0, 1]
            for t in (0, 1):
                if c >= nch[t]:
                    continue
                yield ("wait", self.p_full[t], c & 1, c + 1, f"mma p{t}({c})")
                if self.mutate == "s_before_pv" and c + 1 < nch[t]:
                    if not k_next:
                        yield ("wait", self.full_k[(c + 1) % K_STAGES], ((c + 1) // K_STAGES) & 1,
                               (c + 1) // K_STAGES + 1, f"mma k{c + 1}")
                        k_next = True
                    self.issue_s(t, c + 1)
                    self.issue_pv(t, c)
                    if t == 1 or c + 1 >= nch[1]:
                        self.commit(self.empty_k[(c + 1) % K_STAGES])
                    continue
                self.issue_pv(t, c)
                if c + 1 < nch[t]:
                    if not k_next:
                        yield ("wait", self.full_k[(c + 1) % K_STAGES], ((c + 1) // K_STAGES) & 1,
                               (c + 1) // K_STAGES + 1, f"mma k{c + 1}")
                        k_next = True
                    self.issue_s(t, c + 1)
                    last = t == tiles[1] or c + 1 >= nch[1]
                    if last:
                        self.commit(self.empty_k[(c + 1) % K_STAGES])
            self.commit(self.empty_v[c % V_STAGES])
            yield ("delay", self.rng.uniform(0.0, 0.3))
        self.done.add("mma")

    def softmax(self, t):
        for c in range(self.nch[t]):
            yield ("wait", self.s_full[t], c & 1, c + 1, f"softmax{t} s({c})")
            if self.s_buf[t] != ("S", c):
                self.fail(f"softmax{t}({c}) reads {self.s_buf[t]} instead of S({c})")
            if c > 0 and self.o_last[t] != c - 1:
                self.fail(f"softmax{t}({c}) rescales O holding chunk {self.o_last[t]}, not {c - 1}")
            yield ("delay", self.rng.uniform(0.5, 4.0))
            if self.s_buf[t] != ("S", c):
                self.fail(f"softmax{t}({c}): S overwritten while it was read")
            self.s_buf[t] = ("P", c)
            self.arrive(self.p_full[t], 128)
        if self.mutate != "no_final_wait":
            yield ("wait", self.o_final[t], 0, 1, f"softmax{t} epilogue")
        if self.o_last[t] != self.nch[t] - 1:
            self.fail(f"epilogue {t} reads O holding chunk {self.o_last[t]}, not {self.nch[t] - 1}")
        self.done.add(f"sm{t}")


# (chunks of tile 0, chunks of tile 1): equal, the later tile one chunk
# longer, a single valid tile, one chunk, longer than every ring
SHAPES = [(1, 1), (1, 0), (1, 2), (2, 2), (3, 3), (3, 4), (4, 0), (5, 6), (7, 7), (8, 8), (6, 7)]


@pytest.mark.parametrize("nch", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
def test_prefill_protocol_is_race_free(nch):
    for seed in range(60):
        v = Sim(nch, seed).run()
        assert not v, f"seed {seed}: {v[:3]}"


@pytest.mark.parametrize("mutate", ["release_k_after_first", "s_before_pv", "no_final_wait", "producer_parity"])
def test_planted_protocol_mistakes_are_caught(mutate):
    caught = 0
    for nch in [(3, 3), (5, 6), (8, 8)]:
        for seed in range(40):
            caught += bool(Sim(nch, seed, mutate).run())
    assert caught > 0
