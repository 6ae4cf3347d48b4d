"""Host model of the attention backward's synchronisation (bw_attend_kernel).

The kernel's roles -- the scheduler / Q copy warp, the dO copy warp, the MMA
thread and the eight math warps -- are written here as generators that wait
on and arrive at mbarriers with the kernel's counts and wait parities, and the
asynchronous engines (TMA copies landing in any order, the tensor pipe
executing MMA groups and commits in issue order, the bulk reductions reading
their staging) complete at random moments.  Random tile sequences (runs of
tiles over one key block) are run under random schedules, and every run must:

* finish (no deadlock);
* never poll a barrier that is two phases away from the one it waits for
  (a parity wait would then pass on the wrong phase);
* never write a buffer -- a Q / dO ring slot, a tensor-memory quarter (S,
  dP / dQ, dV, dK), a warp's bytes of the P / dS tiles -- while a reader or
  writer of its previous content is still pending, and never read one that a
  pending writer has not finished;
* read, at every use, the content that use expects (this tile's Q and dO,
  this run's K / V and dK / dV, this tile's S, dP, P, dS and dQ): each buffer
  carries a tag of what was last written to it.

No GPU is involved; this checks the protocol's design, not the device code.
"""
import random

import pytest

from _kernel_consts import kconst, mbar_count

# the kernel's own values (prefill_attend.cu, bw_attend_kernel)
INFO, SLOTS, MATH = (kconst(n, "prefill_attend.cu") for n in ("kBwInfo", "kBwSlots", "kBwMath"))
INFO_EMPTY, P_FULL, DQ_FREE, ACC_FREE = (mbar_count(b, "prefill_attend.cu", after="bw_attend_kernel(")
                                         for b in ("info_empty", "p_full", "dq_free", "acc_free"))


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
    def __init__(self, tiles, rng, early_q_release=False):
        self.rng = rng
        self.tiles = tiles  # list of (fresh, last)
        self.early_q_release = early_q_release  # a planted mistake, for the last test
        self.tag = {}  # buffer -> what it holds
        b = self.bars = {}

        def bar(name, count=1):
            b[name] = Bar(name, count)
        for i in range(INFO):
            bar(f"info_full{i}")
            bar(f"info_empty{i}", INFO_EMPTY)
        bar("kv_full")
        bar("kv_empty")
        for i in range(SLOTS):
            bar(f"qd_full{i}")
            bar(f"qd_empty{i}")
        bar("s_full")
        bar("p_full", P_FULL)
        bar("dq_full")
        bar("dq_free", DQ_FREE)
        bar("acc_full")
        bar("acc_free", ACC_FREE)
        # buffer state: pending asynchronous readers / writers, and active
        # readers in the math warps (tensor memory)
        self.pend_r = {}  # buffer -> count of pending async readers
        self.pend_w = {}  # buffer -> count of pending async writers
        self.math_r = {}  # tensor-memory quarter -> active math readers
        self.pipe = []  # in-order tensor pipe: ("mma", reads, writes) or ("commit", bar)
        self.loads = []  # TMA copies in flight: (buffer, tag, barrier)
        self.bulk = {w: [] for w in range(MATH)}  # per math warp: staging reads in flight

    # ---- helpers ----
    def wait(self, name, parity, need):
        bar = self.bars[name]

        def ok():
            c = bar.done
            assert need - 1 <= c <= need, f"{name}: {c} phases done, waiting for phase {need - 1}"
            return (c & 1) != parity
        return ok

    def _inc(self, d, k):
        d[k] = d.get(k, 0) + 1

    def _dec(self, d, k):
        d[k] -= 1
        assert d[k] >= 0

    def write_now(self, buf, tag):  # a synchronous write by a warp (shared or tensor memory)
        assert not self.pend_r.get(buf) and not self.pend_w.get(buf), f"write of {buf} under a pending access"
        assert not self.math_r.get(buf), f"write of {buf} while a warp reads it"
        self.tag[buf] = tag

    def read_start(self, buf, tag):
        assert not self.pend_w.get(buf), f"read of {buf} under a pending write"
        assert self.tag.get(buf) == tag, f"{buf} holds {self.tag.get(buf)}, expected {tag}"
        self._inc(self.math_r, buf)

    def read_end(self, buf):
        self._dec(self.math_r, buf)

    def mma(self, reads, writes):
        # reads: [(buffer, expected tag)]; writes: [(buffer, tag written)]
        for w, _ in writes:
            assert not self.math_r.get(w), f"MMA writes {w} while a warp reads it"
        for r, tag in reads:
            assert not self.pend_w.get(r), f"MMA reads {r} while it is being written"
            assert self.tag.get(r) == tag, f"MMA reads {r} holding {self.tag.get(r)}, expected {tag}"
            self._inc(self.pend_r, r)
        for w, _ in writes:
            self._inc(self.pend_w, w)
        self.pipe.append(("mma", [r for r, _ in reads], writes))

    def commit(self, name):
        self.pipe.append(("commit", name))

    def load(self, buf, tag, name):
        assert not self.pend_r.get(buf) and not self.math_r.get(buf), f"copy into {buf} while it is read"
        assert not self.pend_w.get(buf), f"two copies into {buf}"
        self._inc(self.pend_w, buf)
        self.loads.append((buf, tag, name))

    # ---- roles ----
    def scheduler(self):  # warp 8: tile info, K / V, the tiles' Q
        nkv = 0
        for i, (fresh, last) in enumerate(self.tiles):
            s, u = i % INFO, i // INFO
            yield self.wait(f"info_empty{s}", (u & 1) ^ 1, u)
            self.bars[f"info_full{s}"].arrive()
            if fresh:
                yield self.wait("kv_empty", (nkv & 1) ^ 1, nkv)
                self.load("KV", ("KV", nkv), "kv_full")
                nkv += 1
            ld = 2 * i
            slot = ld % SLOTS
            yield self.wait(f"qd_empty{slot}", ((ld // SLOTS) & 1) ^ 1, ld // SLOTS)
            self.load(f"slot{slot}", ("Q", i), f"qd_full{slot}")

    def dout_warp(self):  # warp 10: the tiles' dO
        for i in range(len(self.tiles)):
            s, u = i % INFO, i // INFO
            yield self.wait(f"info_full{s}", u & 1, u + 1)
            self.bars[f"info_empty{s}"].arrive()
            ld = 2 * i + 1
            slot = ld % SLOTS
            yield self.wait(f"qd_empty{slot}", ((ld // SLOTS) & 1) ^ 1, ld // SLOTS)
            self.load(f"slot{slot}", ("dO", i), f"qd_full{slot}")

    def mma_thread(self):  # warp 9
        nkv = 0
        P = [f"P{w}" for w in range(MATH)]
        DS = [f"DS{w}" for w in range(MATH)]
        for i, (fresh, last) in enumerate(self.tiles):
            s, u = i % INFO, i // INFO
            yield self.wait(f"info_full{s}", u & 1, u + 1)
            self.bars[f"info_empty{s}"].arrive()
            run = nkv
            if fresh:
                yield self.wait("kv_full", nkv & 1, nkv + 1)
                nkv += 1
            r = nkv - 1  # this tile's run
            kv = ("KV", r)
            lq, lo = 2 * i, 2 * i + 1
            sq, so = f"slot{lq % SLOTS}", f"slot{lo % SLOTS}"
            yield self.wait(f"qd_full{lq % SLOTS}", (lq // SLOTS) & 1, lq // SLOTS + 1)
            self.mma([(sq, ("Q", i)), ("KV", kv)], [("S", ("S", i))])
            if self.early_q_release:
                self.commit(f"qd_empty{lq % SLOTS}")
            yield self.wait(f"qd_full{lo % SLOTS}", (lo // SLOTS) & 1, lo // SLOTS + 1)
            if i > 0:
                yield self.wait("dq_free", (i - 1) & 1, i)
            self.mma([(so, ("dO", i)), ("KV", kv)], [("DPQ", ("dP", i))])
            self.commit("s_full")
            yield self.wait("p_full", i & 1, i + 1)
            if fresh and run > 0:
                yield self.wait("acc_free", (run - 1) & 1, run)
            self.mma([(b, ("DS", i)) for b in DS] + [(sq, ("Q", i))], [("DK", ("DK", r))])
            if not self.early_q_release:
                self.commit(f"qd_empty{lq % SLOTS}")
            self.mma([(b, ("P", i)) for b in P] + [(so, ("dO", i))], [("DV", ("DV", r))])
            self.commit(f"qd_empty{lo % SLOTS}")
            self.mma([(b, ("DS", i)) for b in DS] + [("KV", kv)], [("DPQ", ("dQ", i))])
            self.commit("dq_full")
            if last:
                self.commit("acc_full")
                self.commit("kv_empty")

    def math_warp(self, w):
        nacc = 0
        mine = [f"P{w}", f"DS{w}"]
        for i, (fresh, last) in enumerate(self.tiles):
            s, u = i % INFO, i // INFO
            yield self.wait(f"info_full{s}", u & 1, u + 1)
            self.bars[f"info_empty{s}"].arrive()
            yield self.wait("s_full", i & 1, i + 1)
            # the previous tile's staging reads of this warp's bytes are done
            yield lambda: not self.bulk[w]
            self.read_start("S", ("S", i))
            self.read_start("DPQ", ("dP", i))
            yield None  # the tensor-memory loads and the arithmetic take time
            self.write_now(f"P{w}", ("P", i))
            self.write_now(f"DS{w}", ("DS", i))
            self.read_end("S")
            self.read_end("DPQ")
            self.bars["p_full"].arrive()
            yield self.wait("dq_full", i & 1, i + 1)
            self.read_start("DPQ", ("dQ", i))
            yield None
            self.write_now(f"P{w}", ("dQ staged", i))  # in this warp's P bytes
            self.read_end("DPQ")
            self.bars["dq_free"].arrive()
            self.stage_read(w, [f"P{w}"])
            if last:
                yield self.wait("acc_full", nacc & 1, nacc + 1)
                for acc in ("DV", "DK"):
                    yield lambda: not self.bulk[w]
                    self.read_start(acc, (acc, nacc))
                    yield None
                    for b in mine:
                        self.write_now(b, (acc + " staged", nacc))
                    self.read_end(acc)
                    self.stage_read(w, mine)
                nacc += 1
                self.bars["acc_free"].arrive()

    def stage_read(self, w, bufs):
        for b in bufs:
            self._inc(self.pend_r, b)
        self.bulk[w].append(bufs)

    # ---- engines ----
    def engines(self):
        """Asynchronous completions that may happen now."""
        out = []
        if self.pipe:
            out.append(self.step_pipe)
        for k in range(len(self.loads)):
            out.append(lambda k=k: self.land(k))
        for w in range(MATH):
            if self.bulk[w]:
                out.append(lambda w=w: self.bulk_done(w))
        return out

    def step_pipe(self):
        op = self.pipe.pop(0)
        if op[0] == "mma":
            for r in op[1]:
                self._dec(self.pend_r, r)
            for x, tag in op[2]:
                self._dec(self.pend_w, x)
                self.tag[x] = tag
        else:
            self.bars[op[1]].arrive()

    def land(self, k):
        buf, tag, name = self.loads.pop(k)
        self._dec(self.pend_w, buf)
        self.tag[buf] = tag
        self.bars[name].arrive()

    def bulk_done(self, w):
        for b in self.bulk[w].pop(0):
            self._dec(self.pend_r, b)

    def run(self):
        roles = [self.scheduler(), self.dout_warp(), self.mma_thread()] + [self.math_warp(w) for w in range(MATH)]
        blocked = [None] * len(roles)
        live = set(range(len(roles)))
        steps = 0
        while live or self.pipe or self.loads or any(self.bulk.values()):
            steps += 1
            assert steps < 200000, "no progress"
            ready = [r for r in live if blocked[r] is None or blocked[r]()]
            moves = [("role", r) for r in ready] + [("engine", e) for e in self.engines()]
            assert moves, "deadlock: " + ", ".join(str(r) for r in sorted(live))
            kind, x = self.rng.choice(moves)
            if kind == "engine":
                x()
                continue
            try:
                blocked[x] = next(roles[x])
            except StopIteration:
                live.discard(x)
                blocked[x] = None
        # every barrier ends between phases
        for b in self.bars.values():
            assert b.pending == b.count, b.name


def tile_sequence(rng, n_runs):
    tiles = []
    for _ in range(n_runs):
        n = rng.randint(1, 5)
        tiles += [(j == 0, j == n - 1) for j in range(n)]
    return tiles


@pytest.mark.parametrize("seed", range(40))
def test_backward_protocol_random_schedules(seed):
    rng = random.Random(seed)
    Sim(tile_sequence(rng, rng.randint(1, 8)), rng).run()


def test_backward_protocol_single_tile_and_long_run():
    Sim([(True, True)], random.Random(1)).run()
    Sim([(j == 0, j == 23) for j in range(24)], random.Random(2)).run()


def test_model_catches_an_early_slot_release():
    # a planted mistake: the Q slot released right after S, although dK reads
    # Q again; the next dO may then land over it before dK is issued, and the
    # model must see that (so it is able to see such mistakes at all)
    failed = 0
    for seed in range(30):
        rng = random.Random(seed)
        try:
            Sim(tile_sequence(rng, 4), rng, early_q_release=True).run()
        except AssertionError:
            failed += 1
    assert failed > 0
