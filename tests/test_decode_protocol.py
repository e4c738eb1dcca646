"""The synchronisation protocol of the bf16 decode kernel
(csrc/decode_tc.cu), checked on the CPU by a randomised discrete-event
model (tests/_event_sim.py): no deadlock, every mbarrier wait sees exactly
the phase it means, and every buffer holds the right data when it is read.

The model follows the kernel's roles:
  * the producer warp, per work item n: wait until every consumer warp has
    read the query slot n % 2 last used by item n - 2, write the item's
    descriptor, copy its query rows into the slot, then stream its chunks,
    chunk k (counted over all items) into ring stage k % S once that
    stage's previous chunk has been consumed; after the last item it
    signals the end through the next slot;
  * four consumer warps: per item, wait for the slot, read the descriptor
    and the query, release the slot; warp w consumes the item's chunks
    with k % 4 == w and releases each stage; then the item epilogue: wait
    until every warp has finished combining the previous item, store its
    state, wait until all four have, combine, and arrive.
  * shared-prefix items (a tile of query rows on the tensor cores): the
    warps release the query slot, store their query rows and arrive
    (q_ready); warp 0 waits for each chunk's stage, issues S and commits
    s_ready; every warp runs its softmax rows and arrives (p_ready); warp 0
    issues P·V and commits the stage's release, and after the last chunk
    o_done, which every warp waits for; then the item epilogue's handshake.
    The tensor pipe runs warp 0's operations in order; a commit arrives when
    everything before it is done.
With S a multiple of four every stage always belongs to the same warp, so
a warp never tests a stage whose earlier phase is still pending for
another warp.  With S = 5 or 6 a warp running ahead passes the parity test
on a phase two behind, which is why the bf16 kernel asserts the multiple
(and why these checks are shown to fire for 5 and 6).  A ring of any size
is safe when a warp first waits for the release of its stage's previous
chunk (the FP8 kernel's five-stage ring does this)."""

import pytest

from tests._event_sim import Bar, EventSim

WARPS = 4
END = "end"


class DecodeSim(EventSim):
    def __init__(self, items, stages, seed, mutate=None, release_wait=False, warps=WARPS):
        super().__init__(seed)
        self.W = warps
        self.mutate = mutate
        self.release_wait = release_wait
        # chunks of each work item (0 for an empty context); ("g", n) is a
        # shared-prefix item of n chunks
        self.items = items
        self.S = stages
        self.full = [Bar(f"full{i}", 1) for i in range(stages)]
        self.empty = [Bar(f"empty{i}", 1) for i in range(stages)]
        self.qfull = [Bar(f"qfull{i}", 1) for i in range(2)]
        self.qempty = [Bar(f"qempty{i}", self.W) for i in range(2)]
        self.epi_full = Bar("epi_full", self.W)
        self.epi_done = Bar("epi_done", self.W)
        self.stage = [None] * stages  # chunk held by each stage
        self.desc = [None, None]  # item described by each slot
        self.q = [None, None]  # item whose query rows each slot holds
        self.state = [None] * self.W  # item whose partial state each warp has stored
        self.combined = {}  # item -> warps that finished its combine
        self.q_ready = Bar("q_ready", self.W)
        self.s_ready = Bar("s_ready", 1)
        self.p_ready = Bar("p_ready", self.W)
        self.o_done = Bar("o_done", 1)
        self.pipe_free = 0.0
        self.gi = [0] * self.W  # shared-prefix items each warp has finished
        self.gch = [0] * self.W  # their chunks
        self.s_done = -1  # last chunk whose S has completed

    @staticmethod
    def chunks(item):
        return item[1] if isinstance(item, tuple) else item

    def pipe(self, duration, start, end):
        t0 = max(self.now, self.pipe_free)
        self.pipe_free = t0 + duration
        self.at(t0, start)
        self.at(t0 + duration, end)

    def commit(self, bar):
        self.pipe(0.0, lambda: None, lambda: self.arrive(bar))

    def run(self):
        roles = [self.producer()] + [self.consumer(w) for w in range(self.W)]
        return self.run_roles(roles, {"producer"} | {f"w{w}" for w in range(self.W)})

    def producer(self):
        k = 0
        for n in range(len(self.items) + 1):
            slot = n & 1
            yield ("wait", self.qempty[slot], ((n >> 1) & 1) ^ 1, n >> 1, f"producer q slot for item {n}")
            if n == len(self.items):
                self.desc[slot] = END
                self.arrive(self.qfull[slot])
                break
            self.desc[slot] = n
            if isinstance(self.items[n], tuple):  # a shared-prefix item: no query copy
                self.arrive(self.qfull[slot])
            else:
                self.expect_tx(self.qfull[slot], 1)
                self.copy(self.qfull[slot], 1, lambda slot=slot, n=n: self.q.__setitem__(slot, n))
            for _ in range(self.chunks(self.items[n])):
                st = k % self.S
                yield ("wait", self.empty[st], ((k // self.S) & 1) ^ 1, k // self.S, f"producer chunk {k}")
                self.expect_tx(self.full[st], 1)
                self.copy(self.full[st], 1, lambda st=st, k=k: self.stage.__setitem__(st, k))
                k += 1
                yield ("delay", self.rng.uniform(0.0, 0.4))
        self.done.add("producer")

    def consumer(self, w):
        k = 0
        n = 0
        while True:
            slot = n & 1
            yield ("wait", self.qfull[slot], (n >> 1) & 1, (n >> 1) + 1, f"warp {w} q slot for item {n}")
            if self.desc[slot] == END:
                self.done.add(f"w{w}")
                return
            if isinstance(self.items[n], tuple):
                if self.desc[slot] != n:
                    self.fail(f"warp {w} item {n}: slot holds descriptor {self.desc[slot]}")
                self.arrive(self.qempty[slot])
                k = yield from self.group(w, n, k)
                yield from self.epilogue(w, n)
                n += 1
                continue
            if self.desc[slot] != n or self.q[slot] != n:
                self.fail(f"warp {w} item {n}: slot holds descriptor {self.desc[slot]}, query {self.q[slot]}")
            yield ("delay", self.rng.uniform(0.0, 0.5))
            if self.q[slot] != n:
                self.fail(f"warp {w} item {n}: query overwritten while read")
            self.arrive(self.qempty[slot])
            for _ in range(self.items[n]):
                if k % self.W == w:
                    st = k % self.S
                    if self.release_wait and k >= self.S:
                        # the stage's previous chunk (another warp's) has been released
                        yield ("wait", self.empty[st], ((k - self.S) // self.S) & 1, (k - self.S) // self.S + 1,
                               f"warp {w} release of chunk {k - self.S}")
                    yield ("wait", self.full[st], (k // self.S) & 1, k // self.S + 1, f"warp {w} chunk {k}")
                    if self.stage[st] != k:
                        self.fail(f"warp {w} reads chunk {self.stage[st]} from stage {st}, wanted {k}")
                    yield ("delay", self.rng.uniform(0.2, 3.0))
                    if self.stage[st] != k:
                        self.fail(f"warp {w}: stage {st} overwritten while chunk {k} was read")
                    self.arrive(self.empty[st])
                k += 1
            yield from self.epilogue(w, n)
            n += 1

    def group(self, w, n, k):
        """A shared-prefix item; returns the chunk count after it."""
        gi = self.gi[w]
        yield ("delay", self.rng.uniform(0.1, 1.0))  # query rows into tensor memory
        self.arrive(self.q_ready)
        for _ in range(self.items[n][1]):
            st = k % self.S
            gch = self.gch[w]
            if w == 0:
                yield ("wait", self.full[st], (k // self.S) & 1, k // self.S + 1, f"issuer chunk {k}")
                if self.gch[0] == self.gch_start(n):
                    yield ("wait", self.q_ready, gi & 1, gi + 1, f"issuer q_ready item {n}")

                def s_start(st=st, k=k):
                    if self.stage[st] != k:
                        self.fail(f"S of chunk {k} reads chunk {self.stage[st]}")

                def s_end(k=k):
                    self.s_done = k
                self.pipe(self.rng.uniform(0.2, 1.5), s_start, s_end)
                self.commit(self.s_ready)
            if self.mutate != "no_s_wait":
                yield ("wait", self.s_ready, gch & 1, gch + 1, f"warp {w} s_ready chunk {k}")
            if self.s_done != k:
                self.fail(f"warp {w} reads S of chunk {k} before it is done (S done up to {self.s_done})")
            yield ("delay", self.rng.uniform(0.2, 2.0))  # softmax of the warp's rows
            self.arrive(self.p_ready)
            if w == 0:
                yield ("wait", self.p_ready, gch & 1, gch + 1, f"issuer p_ready chunk {k}")

                def pv_end(st=st, k=k):
                    if self.stage[st] != k:
                        self.fail(f"P·V of chunk {k} read a stage overwritten with {self.stage[st]}")
                if self.mutate == "release_before_pv":
                    self.commit(self.empty[st])
                    self.pipe(self.rng.uniform(0.2, 1.5), lambda: None, pv_end)
                else:
                    self.pipe(self.rng.uniform(0.2, 1.5), lambda: None, pv_end)
                    self.commit(self.empty[st])
                if _ + 1 == self.items[n][1]:
                    self.commit(self.o_done)
            self.gch[w] += 1
            k += 1
        yield ("wait", self.o_done, gi & 1, gi + 1, f"warp {w} o_done item {n}")
        self.gi[w] += 1
        return k

    def gch_start(self, n):
        return sum(self.items[i][1] for i in range(n) if isinstance(self.items[i], tuple))

    def epilogue(self, w, n):
        if True:
            if n > 0:
                yield ("wait", self.epi_done, (n - 1) & 1, n, f"warp {w} epilogue {n} (previous combine)")
                if len(self.combined.get(n - 1, ())) != self.W:
                    self.fail(f"warp {w} stores item {n} before item {n - 1} is combined")
            self.state[w] = n
            self.arrive(self.epi_full)
            yield ("wait", self.epi_full, n & 1, n + 1, f"warp {w} epilogue {n} (states)")
            if any(s != n for s in self.state):
                self.fail(f"warp {w} combines item {n} from states {self.state}")
            yield ("delay", self.rng.uniform(0.1, 1.0))
            if any(s != n for s in self.state):
                self.fail(f"warp {w}: a state was overwritten during the combine of item {n}")
            self.combined.setdefault(n, set()).add(w)
            self.arrive(self.epi_done)


def _items(rng, group=False):
    items = [rng.choice([0, 1, 2, 3, 5, 8, 13]) for _ in range(rng.randint(1, 9))]
    if group:  # shared-prefix items at the head of the list, as the planner puts them, and one more anywhere
        items = [("g", rng.choice([1, 2, 4, 16])) for _ in range(rng.randint(1, 3))] + items
        items.insert(rng.randint(0, len(items)), ("g", rng.choice([1, 3, 8])))
    return items


@pytest.mark.parametrize("stages", [4, 8, 12])
def test_decode_protocol_is_race_free(stages):
    import random

    for seed in range(150):
        items = _items(random.Random(1000 + seed))
        v = DecodeSim(items, stages, seed).run()
        assert not v, f"seed {seed}, items {items}: {v[:3]}"


@pytest.mark.parametrize("stages", [5, 6])
def test_stage_counts_not_a_multiple_of_the_warps_are_caught(stages):
    import random

    caught = sum(bool(DecodeSim(_items(random.Random(1000 + seed)), stages, seed).run()) for seed in range(150))
    assert caught > 0


@pytest.mark.parametrize("stages", [4, 8])
def test_decode_protocol_with_shared_prefix_items_is_race_free(stages):
    import random

    for seed in range(150):
        items = _items(random.Random(2000 + seed), group=True)
        v = DecodeSim(items, stages, seed).run()
        assert not v, f"seed {seed}, items {items}: {v[:3]}"


@pytest.mark.parametrize("mutate", ["release_before_pv", "no_s_wait"])
def test_planted_shared_item_mistakes_are_caught(mutate):
    import random

    caught = sum(bool(DecodeSim(_items(random.Random(3000 + seed), group=True), 4, seed, mutate).run())
                 for seed in range(100))
    assert caught > 0


@pytest.mark.parametrize("stages", [5, 6, 7])
def test_any_stage_count_is_race_free_when_a_warp_waits_for_the_previous_release(stages):
    """With S not a multiple of four a stage passes between warps; a warp
    that first waits for the release of the stage's previous chunk can
    never test a full barrier two phases behind (the FP8 kernel's ring)."""
    import random

    for seed in range(150):
        for group in (False, True):
            items = _items(random.Random(4000 + seed), group=group)
            v = DecodeSim(items, stages, seed, release_wait=True).run()
            assert not v, f"seed {seed}, items {items}: {v[:3]}"


@pytest.mark.parametrize("warps,stages,race_free", [(6, 5, False), (6, 6, True), (6, 7, True), (4, 5, True)])
def test_stage_passing_needs_no_more_warps_than_stages(warps, stages, race_free):
    """A warp that waits for its stage's previous release (the FP8 kernel's
    protocol) can still pass that wait, and the full one after it, two
    phases early when the consumer warps outnumber the stages: a warp at
    chunk k knows only that chunks up to k - W - S were released (its own
    previous chunk k - W was filled), while its parity waits are exact only
    if chunk k - 2S was.  With W <= S that always holds."""
    import random

    caught = 0
    for seed in range(150):
        items = _items(random.Random(3000 + seed))
        caught += bool(DecodeSim(items, stages, seed, release_wait=True, warps=warps).run())
    if race_free:
        assert caught == 0
    else:
        assert caught > 0

