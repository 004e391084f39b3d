"""A model of the streaming kernel's copy ring, checked under random schedules on the CPU (the
kernel's race check: no tool runs on the GPU for it).

The ring (stream_tma.cu): R slots; the producer of slot j loads the block's chunks
k = j, j + R, j + 2R, ... into it, each load completing a phase of the slot's `full` barrier when
its bytes land, and before reloading the slot waits until the previous chunk's consumer has
arrived on the slot's `empty` barrier. Consumers take chunk numbers k = 0, 1, 2, ... from a shared
counter and read slot k mod R. Barrier waits test a phase *parity*: a wait for the phase of round r
passes whenever the number of completed phases c has parity different from r, so it cannot tell
c = r + 1 (the chunk landed) from c = r - 1 (the chunk before it has not). The kernel therefore has
the producer publish a tag {k} on the slot when it issues the load of chunk k, and a consumer of
chunk k waits for its tag before the parity wait. The tag is written only after the chunk k - R was
consumed, so c >= r when it is seen, and c <= r + 1 because the slot cannot be reloaded before
chunk k is consumed: the parity wait is then exact.

The model runs producers, in-flight copies and consumers as separate actors, picks the next actor at
random, and records every read of a slot whose chunk has not landed. Without the tag such reads
occur; with it none does, every chunk is consumed exactly once, and every schedule terminates."""
import random

import pytest

DONE = -2


class Ring:
    def __init__(self, R, n_chunks, n_consumers, tagged, rng):
        self.R, self.n, self.tagged, self.rng = R, n_chunks, tagged, rng
        self.full_c = [0] * R        # completed phases of each slot's full barrier
        self.empty_c = [0] * R       # completed phases of each slot's empty barrier
        self.tag = [None] * R        # chunk number published on the slot (None: never loaded)
        self.data = [None] * R       # chunk whose bytes are in the slot
        self.prod_round = [0] * R    # next round of each slot's producer
        self.prod_done = [False] * R
        self.inflight = []           # (slot, chunk) copies issued but not landed
        self.next_k = 0
        self.cons = [dict(k=None, stage="take") for _ in range(n_consumers)]
        self.consumed = []
        self.bad_reads = 0

    @staticmethod
    def parity_passed(completed, rnd):
        """A wait for the phase of round `rnd` on a barrier with `completed` phases."""
        return (completed & 1) != (rnd & 1)

    def producer_step(self, j):
        r = self.prod_round[j]
        k = j + r * self.R
        if r > 0 and not self.parity_passed(self.empty_c[j], r - 1):
            return False  # the previous chunk of this slot is still in use
        if k >= self.n:
            self.tag[j] = DONE
            self.prod_done[j] = True
            return True
        self.tag[j] = k
        self.inflight.append((j, k))
        self.prod_round[j] = r + 1
        return True

    def land(self, idx):
        j, k = self.inflight.pop(idx)
        self.data[j] = k
        self.full_c[j] += 1

    def consumer_step(self, c):
        st = self.cons[c]
        if st["stage"] == "take":
            if self.next_k >= self.n + self.R * 4:  # past every chunk: stop taking
                st["stage"] = "stopped"
                return True
            st["k"] = self.next_k
            self.next_k += 1
            st["stage"] = "tag" if self.tagged else "full"
            return True
        k = st["k"]
        j, r = k % self.R, k // self.R
        if st["stage"] == "tag":
            if self.tag[j] == DONE:
                st["stage"] = "take"  # this slot has no more chunks
                return True
            if self.tag[j] != k:
                return False
            st["stage"] = "full"
            return True
        if st["stage"] == "full":
            if k >= self.n:  # (untagged model: a number past the last chunk)
                st["stage"] = "take"
                return True
            if not self.parity_passed(self.full_c[j], r):
                return False
            if self.data[j] != k:
                self.bad_reads += 1  # read a slot whose chunk has not landed
            self.consumed.append(k)
            self.empty_c[j] += 1
            st["stage"] = "take"
            return True
        return False

    def run(self, max_steps=200000):
        for _ in range(max_steps):
            actors = [("p", j) for j in range(self.R) if not self.prod_done[j]]
            actors += [("l", i) for i in range(len(self.inflight))]
            actors += [("c", c) for c in range(len(self.cons)) if self.cons[c]["stage"] != "stopped"]
            if not actors:
                return True
            self.rng.shuffle(actors)
            for kind, x in actors:
                moved = (self.producer_step(x) if kind == "p" else
                         self.land(x) or True if kind == "l" else self.consumer_step(x))
                if moved:
                    break
            else:
                return False  # nothing can move: a deadlock
        return False


@pytest.mark.parametrize("R,n,consumers", [(4, 37, 3), (8, 64, 6), (32, 200, 18)])
def test_tagged_ring_is_exact(R, n, consumers):
    for seed in range(60):
        ring = Ring(R, n, consumers, tagged=True, rng=random.Random(seed))
        assert ring.run(), f"schedule {seed} did not terminate"
        assert ring.bad_reads == 0, f"schedule {seed}: {ring.bad_reads} reads before landing"
        assert sorted(ring.consumed) == list(range(n))  # every chunk exactly once
        assert not ring.inflight


def test_parity_only_ring_reads_before_landing():
    """The same ring without the tags: some schedules pass a parity wait one phase early."""
    bad = 0
    for seed in range(200):
        ring = Ring(4, 37, 3, tagged=False, rng=random.Random(seed))
        ring.run()
        bad += ring.bad_reads
    assert bad > 0
