"""Host model of the prefill scorer's synchronisation (prefill_select_kernel).

Roles as in the kernel: a TMA thread (the unit's index-Q tiles of two heads
once, then the unit's causal key blocks through a 3-stage ring), an MMA
thread (per key block, both heads into one of two tensor-memory buffers) and
four epilogue warps (block max of their token rows from that buffer).  Units
whose block count does not exceed topk are written by the epilogue alone and
skipped by the other two roles, so the block counters of the MMA thread and
the epilogue must agree.  TMA copies land in any order and the MMA groups
execute in issue order.  Random unit lists under random schedules must
finish, never poll a barrier two phases away from the phase they wait for,
never write under a pending access, and read in every use the content they
expect.  A planted mistake (the MMA thread taking every other key block from
the neighbouring stage) must be reported.  No GPU is involved.
"""
import random

import pytest

from _kernel_consts import kconst, mbar_count

# the kernel's own values (prefill_select.cu): epilogue warps = arrivals that free a tensor-memory buffer
EPI = mbar_count("t_empty", "prefill_select.cu")
STAGES = kconst("kPsStages", "prefill_select.cu")


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
    def __init__(self, units, topk, rng, stages=STAGES, skew=False):
        # units: block counts nb (qb + 1) of this CTA's units, in order
        self.units, self.topk, self.rng, self.S, self.skew = units, topk, rng, stages, skew
        self.bars = {"a_full": Bar("a_full", 1), "a_empty": Bar("a_empty", 1)}
        for s in range(stages):
            self.bars[f"b_full{s}"] = Bar(f"b_full{s}", 1)
            self.bars[f"b_empty{s}"] = Bar(f"b_empty{s}", 1)
        for b in range(2):
            self.bars[f"t_full{b}"] = Bar(f"t_full{b}", 1)
            self.bars[f"t_empty{b}"] = Bar(f"t_empty{b}", EPI)
        self.tag, self.pend_r, self.pend_w, self.warp_r = {}, {}, {}, {}
        self.pipe, self.loads = [], []

    def wait(self, name, parity, need):
        bar = self.bars[name]

        def ok():
            c = bar.done
            assert need - 1 <= c <= need, f"{name}: {c} phases done, waiting for phase {need - 1}"
            return (c & 1) != parity
        return ok

    def _add(self, d, k, v):
        d[k] = d.get(k, 0) + v
        assert d[k] >= 0

    def load(self, buf, tag, name):
        assert not self.pend_r.get(buf) and not self.pend_w.get(buf), f"copy into {buf} under a pending access"
        self._add(self.pend_w, buf, 1)
        self.loads.append((buf, tag, name))

    def mma(self, reads, writes):
        for w, _ in writes:
            assert not self.warp_r.get(w), f"MMA writes {w} while a warp reads it"
        for r, tag in reads:
            assert not self.pend_w.get(r), f"MMA reads {r} while it is being written"
            assert self.tag.get(r) == tag, f"MMA reads {r} holding {self.tag.get(r)}, expected {tag}"
            self._add(self.pend_r, r, 1)
        for w, _ in writes:
            self._add(self.pend_w, w, 1)
        self.pipe.append(("mma", [r for r, _ in reads], writes))

    def scored(self):
        return [(u, nb) for u, nb in enumerate(self.units) if nb > self.topk]

    def stage_of(self, bc):
        s = bc % self.S
        if self.skew and bc % 2:  # the planted mistake: odd blocks read the other stage
            s = (s + 1) % self.S
        return s

    def tma(self):
        nunit = bc = 0
        for u, nb in self.scored():
            yield self.wait("a_empty", (nunit & 1) ^ 1, nunit)
            self.load("A", ("A", u), "a_full")
            for b in range(nb):
                s = bc % self.S
                yield self.wait(f"b_empty{s}", ((bc // self.S) & 1) ^ 1, bc // self.S)
                self.load(f"B{s}", ("B", u, b), f"b_full{s}")
                bc += 1
            nunit += 1

    def mma_thread(self):
        nunit = bc = kc = 0
        for u, nb in self.scored():
            yield self.wait("a_full", nunit & 1, nunit + 1)
            for b in range(nb):
                s, buf = self.stage_of(bc), kc & 1
                yield self.wait(f"b_full{s}", (bc // self.S) & 1, bc // self.S + 1)
                yield self.wait(f"t_empty{buf}", ((kc >> 1) & 1) ^ 1, kc >> 1)
                self.mma([("A", ("A", u)), (f"B{s}", ("B", u, b))], [(f"T{buf}_{w}", ("T", u, b)) for w in range(EPI)])
                self.pipe.append(("commit", f"b_empty{s}"))
                self.pipe.append(("commit", f"t_full{buf}"))
                bc += 1
                kc += 1
            self.pipe.append(("commit", "a_empty"))
            nunit += 1

    def epilogue(self, w):
        kc = 0
        for u, nb in enumerate(self.units):
            if nb <= self.topk:
                yield None  # the rows are written without scores
                continue
            for b in range(nb):
                buf = kc & 1
                yield self.wait(f"t_full{buf}", (kc >> 1) & 1, (kc >> 1) + 1)
                t = f"T{buf}_{w}"
                assert not self.pend_w.get(t), f"read of {t} under a pending write"
                assert self.tag.get(t) == ("T", u, b), f"{t} holds {self.tag.get(t)}, expected {('T', u, b)}"
                self._add(self.warp_r, t, 1)
                yield None  # the block max of both heads
                self._add(self.warp_r, t, -1)
                self.bars[f"t_empty{buf}"].arrive()
                kc += 1

    def run(self):
        roles = [self.tma(), self.mma_thread()] + [self.epilogue(w) for w in range(EPI)]
        blocked = [None] * len(roles)
        live = set(range(len(roles)))
        steps = 0
        while live or self.pipe or self.loads:
            steps += 1
            assert steps < 500000, "no progress"
            ready = [r for r in live if blocked[r] is None or blocked[r]()]
            moves = [("role", r) for r in ready]
            if self.pipe:
                moves.append(("pipe", 0))
            moves += [("land", k) for k in range(len(self.loads))]
            assert moves, "deadlock"
            kind, x = self.rng.choice(moves)
            if kind == "pipe":
                op = self.pipe.pop(0)
                if op[0] == "mma":
                    for r in op[1]:
                        self._add(self.pend_r, r, -1)
                    for b, tag in op[2]:
                        self._add(self.pend_w, b, -1)
                        self.tag[b] = tag
                else:
                    self.bars[op[1]].arrive()
            elif kind == "land":
                buf, tag, name = self.loads.pop(x)
                self._add(self.pend_w, buf, -1)
                self.tag[buf] = tag
                self.bars[name].arrive()
            else:
                try:
                    blocked[x] = next(roles[x])
                except StopIteration:
                    live.discard(x)
                    blocked[x] = None


def unit_list(rng):
    return [rng.randint(1, 24) for _ in range(rng.randint(1, 8))]


@pytest.mark.parametrize("seed", range(30))
def test_prefill_select_protocol_random_schedules(seed):
    rng = random.Random(seed)
    Sim(unit_list(rng), rng.choice([1, 3, 16]), rng).run()


def test_model_catches_a_skewed_stage():
    failed = 0
    for seed in range(30):
        rng = random.Random(seed)
        try:
            Sim(unit_list(rng), 3, rng, skew=True).run()
        except AssertionError:
            failed += 1
    assert failed > 0
