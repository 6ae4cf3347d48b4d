"""Host model of the decode attention's synchronisation (sparse_attend_kernel).

The producer warp and the consumer warps are generators that wait on and
arrive at mbarriers with the kernel's counts and wait parities: a 2-slot
segment ring (key counts and the Q tile of a (request, KV head) segment) and a
6-stage ring of 64-key chunks, stage s always taken by consumer warp s mod 3;
the consumers meet at the end of every segment (the kernel's named barrier)
to merge their states.  TMA copies land in any order at random moments.
Random segment lists (blocks of 1..128 keys, empty entries) are run under
random schedules, and every run must finish, never poll a barrier two phases
away from the phase it waits for, never copy into a slot or stage that is
still being read, and read in every use the segment or chunk it expects.

A warp that took chunks round-robin (chunk c to warp c mod C) with a stage
count that is not a multiple of C could wait on a stage two phases ahead and
read a stale chunk; a test plants that assignment and checks that the model
reports it.  Without the segment ring the same model is the decode scorer's
page ring (decode_select_kernel: page i to warp i mod 6 through 6 or 12
stages), checked as it is and in the eight-warp form that once faulted.  No
GPU is involved.
"""
import random

import pytest

from _kernel_consts import kconst, mbar_count

# the kernels' own values (sparse_attend.cu, decode_select.cu)
SEG_SLOTS = kconst("kSegSlots", "sparse_attend.cu")
CHUNK_KEYS = kconst("kChunkKeys", "sparse_attend.cu")
STAGES = kconst("kAttStages", "sparse_attend.cu")
CONSUMERS = kconst("kConsumerWarps", "sparse_attend.cu")
SEG_EMPTY = mbar_count("seg_empty", "sparse_attend.cu")  # every consumer warp releases a segment slot
SEL_CONSUMERS = kconst("kSelConsumers", "decode_select.cu")
SEL_STAGES = (kconst("kSelRingBytes", "decode_select.cu") // (128 * 256),  # bf16 pages
              kconst("kSelRingBytes", "decode_select.cu") // (128 * 128))  # E4M3 pages


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.done = name, count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, self.name
        if self.pending == 0:
            self.done += 1
            self.pending = self.count


class Sim:
    def __init__(self, segments, rng, stages=STAGES, consumers=CONSUMERS, by_chunk=False, segment_ring=True,
                 seg_slots=SEG_SLOTS):
        # segments: list of lists of key counts (0 = an empty / padded entry).
        # Without the segment ring (and its end-of-segment meetings) this is the
        # decode scorer's page ring: one stage per item, item i to a warp.
        self.segs, self.rng = segments, rng
        self.S, self.C, self.by_chunk, self.seg_ring = stages, consumers, by_chunk, segment_ring
        self.Q = seg_slots
        self.bars = {}
        for i in range(seg_slots):
            self.bars[f"seg_full{i}"] = Bar(f"seg_full{i}", 1)
            self.bars[f"seg_empty{i}"] = Bar(f"seg_empty{i}", SEG_EMPTY if consumers == CONSUMERS else consumers)
        for s in range(stages):
            self.bars[f"full{s}"] = Bar(f"full{s}", 1)
            self.bars[f"empty{s}"] = Bar(f"empty{s}", 1)
        self.tag, self.reading, self.landing = {}, {}, set()
        self.loads = []
        self.meet = [0, 0]  # segment-end rendezvous: arrivals, generation

    def wait(self, name, parity, need):
        bar = self.bars[name]

        def ok():
            c = bar.done
            assert need - 1 <= c <= need, f"{name}: {c} phases done, waiting for phase {need - 1}"
            return (c & 1) != parity
        return ok

    def load(self, buf, tag, name):
        assert not self.reading.get(buf), f"copy into {buf} while it is read"
        assert buf not in self.landing, f"two copies into {buf}"
        self.landing.add(buf)
        self.loads.append((buf, tag, name))

    def read(self, buf, tag):
        assert buf not in self.landing, f"read of {buf} while a copy lands"
        assert self.tag.get(buf) == tag, f"{buf} holds {self.tag.get(buf)}, expected {tag}"

    def owner(self, sc):
        return (sc % self.C) if self.by_chunk else (sc % self.S) % self.C

    def chunks(self, keys):
        return [(k + CHUNK_KEYS - 1) // CHUNK_KEYS for k in keys]

    def producer(self):
        sc = 0
        for nseg, keys in enumerate(self.segs):
            ss = nseg % self.Q
            if self.seg_ring:
                yield self.wait(f"seg_empty{ss}", ((nseg // self.Q) & 1) ^ 1, nseg // self.Q)
                self.load(f"seg{ss}", ("seg", nseg), f"seg_full{ss}")
            for nch in self.chunks(keys):
                for _ in range(nch):
                    s = sc % self.S
                    yield self.wait(f"empty{s}", ((sc // self.S) & 1) ^ 1, sc // self.S)
                    self.load(f"stage{s}", ("chunk", sc), f"full{s}")
                    sc += 1

    def consumer(self, w):
        sc = 0
        for nseg, keys in enumerate(self.segs):
            ss = nseg % self.Q
            if self.seg_ring:
                yield self.wait(f"seg_full{ss}", (nseg // self.Q) & 1, nseg // self.Q + 1)
                self.read(f"seg{ss}", ("seg", nseg))
                self.reading[f"seg{ss}"] = self.reading.get(f"seg{ss}", 0) + 1
                yield None  # the Q fragments are loaded
                self.reading[f"seg{ss}"] -= 1
                self.bars[f"seg_empty{ss}"].arrive()
            for nch in self.chunks(keys):
                for _ in range(nch):
                    if self.owner(sc) == w:
                        s = sc % self.S
                        yield self.wait(f"full{s}", (sc // self.S) & 1, sc // self.S + 1)
                        self.read(f"stage{s}", ("chunk", sc))
                        self.reading[f"stage{s}"] = self.reading.get(f"stage{s}", 0) + 1
                        yield None  # S, softmax, O on the chunk
                        self.reading[f"stage{s}"] -= 1
                        self.bars[f"empty{s}"].arrive()
                    sc += 1
            # the consumers meet twice at the end of the segment (merge through
            # shared memory); warp 0 then writes while the others go on
            for _ in range(2 if self.seg_ring else 0):
                gen = self.meet[1]
                self.meet[0] += 1
                if self.meet[0] == self.C:
                    self.meet = [0, gen + 1]
                yield lambda gen=gen: self.meet[1] != gen

    def run(self):
        roles = [self.producer()] + [self.consumer(w) for w in range(self.C)]
        blocked = [None] * len(roles)
        live = set(range(len(roles)))
        steps = 0
        while live or self.loads:
            steps += 1
            assert steps < 500000, "no progress"
            ready = [r for r in live if blocked[r] is None or blocked[r]()]
            moves = [("role", r) for r in ready] + [("land", k) for k in range(len(self.loads))]
            assert moves, "deadlock"
            kind, x = self.rng.choice(moves)
            if kind == "land":
                buf, tag, name = self.loads.pop(x)
                self.landing.discard(buf)
                self.tag[buf] = tag
                self.bars[name].arrive()
                continue
            try:
                blocked[x] = next(roles[x])
            except StopIteration:
                live.discard(x)
                blocked[x] = None


def segment_list(rng, n):
    segs = []
    for _ in range(n):
        segs.append([rng.choice([0, 1, 37, 64, 65, 100, 128, 128, 128]) for _ in range(rng.randint(1, 16))])
    return segs


@pytest.mark.parametrize("seed", range(30))
def test_decode_attend_protocol_random_schedules(seed):
    rng = random.Random(seed)
    Sim(segment_list(rng, rng.randint(1, 6)), rng).run()


@pytest.mark.parametrize("seed", range(10))
def test_decode_attend_protocol_one_q_slot(seed):
    # the FP8 cache's form: one Q tile in the segment ring (two CTAs per SM)
    rng = random.Random(300 + seed)
    Sim(segment_list(rng, rng.randint(1, 6)), rng, seg_slots=1).run()


def test_decode_attend_protocol_twice_the_stages():
    # the stage count only has to be a multiple of the consumer warps
    assert STAGES % CONSUMERS == 0
    for seed in range(5):
        rng = random.Random(100 + seed)
        Sim(segment_list(rng, 4), rng, stages=2 * STAGES).run()


def test_model_catches_round_robin_chunks():
    # chunks handed out round-robin over 4 warps through 6 stages: a warp can
    # wait on a stage two phases ahead; the model must report it
    failed = 0
    for seed in range(30):
        rng = random.Random(seed)
        try:
            Sim(segment_list(rng, 4), rng, stages=6, consumers=4, by_chunk=True).run()
        except AssertionError:
            failed += 1
    assert failed > 0


@pytest.mark.parametrize("stages", SEL_STAGES)
def test_decode_scorer_page_ring(stages):
    # the decode scorer: item (page) i to warp i mod kSelConsumers through the
    # bf16 or the E4M3 ring (6 or 12 stages as compiled) -- round-robin, safe
    # because the stage count is a multiple of the warps
    assert stages % SEL_CONSUMERS == 0
    for seed in range(10):
        rng = random.Random(200 + seed)
        Sim(segment_list(rng, 4), rng, stages=stages, consumers=SEL_CONSUMERS, by_chunk=True,
            segment_ring=False).run()


def test_model_reports_the_eight_warp_scorer_ring():
    # the scorer's first form: eight warps round-robin over six stages (the
    # Xid 31 recorded for it); the model must report a parity aliasing
    failed = 0
    for seed in range(30):
        rng = random.Random(seed)
        try:
            Sim(segment_list(rng, 4), rng, stages=6, consumers=8, by_chunk=True, segment_ring=False).run()
        except AssertionError:
            failed += 1
    assert failed > 0
