"""Host model of the prefill attention's synchronisation (bm_attend_kernel).

Roles as in the kernel: the scheduler / TMA warp (K of a new block, the
tile's Q rows, V of a new block), the S-MMA thread, the O-MMA thread, two
softmax warpgroups taking the even and the odd tiles and two epilogue
warpgroups taking every tile, half of its O columns each (four warps each).
Tensor memory holds S twice, P (bf16) twice in columns of its own, and O
once: a softmax warpgroup frees its S buffer as soon as it has read it, and
both epilogue warpgroups have read a tile's O before the next O product may
overwrite it;
shared memory holds Q twice, K twice, V once, and per epilogue warp two 4 KB
staging halves: per 32-column quarter of its rows the warp waits until the
bulk group of two quarters ago has read the half it is about to fill
(cp.async.bulk.wait_group.read 1), writes it, and issues that quarter's
tensor-engine store / add as a new bulk group.  The TMA copies land in any
order, each MMA thread's groups and commits execute in that thread's issue
order (no order is assumed between the two threads: what one reads the other
writes only behind a barrier), and the bulk groups read their staging at
random moments, in any order.  Random tile sequences (runs of tiles over one
key block) under random schedules must finish, never poll a barrier two
phases away from the phase they wait for, never write anything under a
pending access, and read in every use the content it expects.  Planted
mistakes (the O MMA not waiting for the epilogue to free its O buffer; the
epilogue refilling a staging half without the bulk read wait) must be
reported.  No GPU is involved.
"""
import random

import pytest

from _kernel_consts import kconst, mbar_count

# the kernel's own values (prefill_attend.cu, bm_attend_kernel)
INFO, QST, KST, VST = (kconst(n, "prefill_attend.cu") for n in ("kBmInfo", "kBmQStages", "kBmKStages", "kBmVStages"))
O_FREE, P_FULL, S_FREE, INFO_EMPTY = (mbar_count(b, "prefill_attend.cu", after="bm_attend_kernel(")
                                      for b in ("o_free", "p_full", "s_free", "info_empty"))
assert O_FREE == 8 and INFO_EMPTY == 14


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
    def __init__(self, tiles, rng, skip_o_free=False, skip_bulk_wait=False):
        self.tiles, self.rng, self.skip_o_free = tiles, rng, skip_o_free  # tiles: list of block ids
        self.skip_bulk_wait = skip_bulk_wait
        self.bars = {}

        def bar(name, count=1):
            self.bars[name] = Bar(name, count)
        for i in range(QST):
            bar(f"q_full{i}")
            bar(f"q_empty{i}")
        for i in range(KST):
            bar(f"k_full{i}")
            bar(f"k_empty{i}")
        for i in range(VST):
            bar(f"v_full{i}")
            bar(f"v_empty{i}")
        for b in range(2):
            bar(f"s_full{b}")
            bar(f"s_free{b}", S_FREE)
            bar(f"p_full{b}", P_FULL)
            bar(f"p_free{b}")
        bar("o_full")
        bar("o_free", O_FREE)
        for i in range(INFO):
            bar(f"info_full{i}")
            bar(f"info_empty{i}", INFO_EMPTY)
        self.tag, self.pend_r, self.pend_w, self.warp_r = {}, {}, {}, {}
        self.pipe = {"S": [], "O": []}  # per MMA thread, in issue order
        self.loads = []
        # per epilogue warp: its bulk groups not yet done reading their staging half, (group id, half)
        self.groups = {(wg, q): [] for wg in (0, 1) for q in range(4)}
        self.issued = {(wg, q): 0 for wg in (0, 1) for q in range(4)}

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

    # accesses -------------------------------------------------------------
    def warp_read(self, buf, tag):
        assert not self.pend_w.get(buf), f"read of {buf} under a pending write"
        assert self.tag.get(buf) == tag, f"{buf} holds {self.tag.get(buf)}, expected {tag}"
        self._add(self.warp_r, buf, 1)

    def warp_read_end(self, buf):
        self._add(self.warp_r, buf, -1)

    def warp_write(self, buf, tag):
        assert not self.pend_r.get(buf) and not self.pend_w.get(buf), f"write of {buf} under a pending access"
        self.tag[buf] = tag

    def mma(self, pipe, reads, writes):
        for w, _ in writes:
            assert not self.warp_r.get(w), f"MMA writes {w} while a warp reads it"
            assert not self.pend_r.get(w), f"MMA writes {w} while an earlier MMA may still read it"
        for r, tag in reads:
            assert not self.pend_w.get(r), f"MMA reads {r} while it is being written"
            assert self.tag.get(r) == tag, f"MMA reads {r} holding {self.tag.get(r)}, expected {tag}"
            self._add(self.pend_r, r, 1)
        for w, _ in writes:
            self._add(self.pend_w, w, 1)
        self.pipe[pipe].append(("mma", [r for r, _ in reads], writes))

    def commit(self, pipe, name):
        self.pipe[pipe].append(("commit", name))

    def load(self, buf, tag, name):
        assert not self.pend_r.get(buf) and not self.pend_w.get(buf), f"copy into {buf} under a pending access"
        self._add(self.pend_w, buf, 1)
        self.loads.append((buf, tag, name))

    # roles ------------------------------------------------------------------
    def fresh(self, i):
        return i == 0 or self.tiles[i] != self.tiles[i - 1]

    def producer(self):
        nkf = nvf = 0
        for i, blk in enumerate(self.tiles):
            s, u = i % INFO, i // INFO
            yield self.wait(f"info_empty{s}", (u & 1) ^ 1, u)
            self.bars[f"info_full{s}"].arrive()
            if self.fresh(i):
                ks = nkf % KST
                yield self.wait(f"k_empty{ks}", ((nkf // KST) & 1) ^ 1, nkf // KST)
                self.load(f"K{ks}", ("K", i), f"k_full{ks}")
                nkf += 1
            qs = i % QST
            yield self.wait(f"q_empty{qs}", ((i // QST) & 1) ^ 1, i // QST)
            self.load(f"Q{qs}", ("Q", i), f"q_full{qs}")
            if self.fresh(i):
                vs = nvf % VST
                yield self.wait(f"v_empty{vs}", ((nvf // VST) & 1) ^ 1, nvf // VST)
                self.load(f"V{vs}", ("V", i), f"v_full{vs}")
                nvf += 1

    def s_mma(self):
        nk = ks = 0
        first = 0  # first tile of the current block (its K / V carry that tile's tag)
        for i in range(len(self.tiles)):
            s, u = i % INFO, i // INFO
            yield self.wait(f"info_full{s}", u & 1, u + 1)
            self.bars[f"info_empty{s}"].arrive()
            if self.fresh(i):
                if nk > 0:
                    self.commit("S", f"k_empty{ks}")
                ks = nk % KST
                yield self.wait(f"k_full{ks}", (nk // KST) & 1, nk // KST + 1)
                nk += 1
                first = i
            b, qs = i & 1, i % QST
            yield self.wait(f"q_full{qs}", (i // QST) & 1, i // QST + 1)
            yield self.wait(f"s_free{b}", ((i >> 1) & 1) ^ 1, i >> 1)
            self.mma("S", [(f"Q{qs}", ("Q", i)), (f"K{ks}", ("K", first))],
                     [(f"S{b}_{q}", ("S", i)) for q in range(4)])
            self.commit("S", f"s_full{b}")
            self.commit("S", f"q_empty{qs}")

    def o_mma(self):
        nv = vs = 0
        first = 0
        for i in range(len(self.tiles)):
            s, u = i % INFO, i // INFO
            yield self.wait(f"info_full{s}", u & 1, u + 1)
            self.bars[f"info_empty{s}"].arrive()
            if self.fresh(i):
                if nv > 0:
                    self.commit("O", f"v_empty{vs}")
                vs = nv % VST
                yield self.wait(f"v_full{vs}", (nv // VST) & 1, nv // VST + 1)
                nv += 1
                first = i
            b = i & 1
            yield self.wait(f"p_full{b}", (i >> 1) & 1, (i >> 1) + 1)
            if not self.skip_o_free:
                # the one O buffer: both epilogue warpgroups have read tile i - 1's
                yield self.wait("o_free", (i & 1) ^ 1, i)
            self.mma("O", [(f"P{b}_{q}", ("P", i)) for q in range(4)] + [(f"V{vs}", ("V", first))],
                     [(f"O_{q}_{h}", ("O", i)) for q in range(4) for h in range(2)])
            self.commit("O", "o_full")
            self.commit("O", f"p_free{b}")

    def softmax(self, wg, q):
        for i in range(wg, len(self.tiles), 2):
            s, u, k = i % INFO, i // INFO, i >> 1
            yield self.wait(f"info_full{s}", u & 1, u + 1)
            self.bars[f"info_empty{s}"].arrive()
            yield self.wait(f"s_full{wg}", k & 1, k + 1)
            yield self.wait(f"p_free{wg}", (k & 1) ^ 1, k)  # the O MMA of its previous tile has read P
            buf = f"S{wg}_{q}"
            self.warp_read(buf, ("S", i))
            yield None  # the passes over the row, P written as it goes
            self.warp_write(f"P{wg}_{q}", ("P", i))
            self.warp_read_end(buf)
            self.bars[f"s_free{wg}"].arrive()
            yield None
            self.bars[f"p_full{wg}"].arrive()

    def epilogue(self, wg, q):
        w = (wg, q)
        buf = f"O_{q}_{wg}"  # the warp's rows, the warpgroup's half of the columns
        for i in range(len(self.tiles)):
            s, u = i % INFO, i // INFO
            yield self.wait(f"info_full{s}", u & 1, u + 1)
            self.bars[f"info_empty{s}"].arrive()
            yield self.wait("o_full", i & 1, i + 1)
            self.warp_read(buf, ("O", i))  # both of its 32-column quarters into registers
            yield None
            assert self.tag.get(buf) == ("O", i), f"{buf} changed under the epilogue's reads"
            self.warp_read_end(buf)
            self.bars["o_free"].arrive()
            for qq in range(2):
                if not self.skip_bulk_wait:
                    # cp.async.bulk.wait_group.read 1: every group but the newest has read its half
                    newest = self.issued[w] - 1
                    yield lambda: all(g == newest for g, _ in self.groups[w])
                half = f"stage{wg}_{q}_{qq & 1}"
                self.warp_write(half, ("stage", i, qq))
                yield None
                assert self.tag.get(half) == ("stage", i, qq)
                self._add(self.pend_r, half, 1)
                self.groups[w].append((self.issued[w], half))
                self.issued[w] += 1

    # engines ----------------------------------------------------------------
    def engines(self):
        out = [lambda p=p: self.step_pipe(p) for p in ("S", "O") if self.pipe[p]]
        out += [lambda k=k: self.land(k) for k in range(len(self.loads))]
        out += [lambda w=w, j=j: self.group_read(w, j) for w, gs in self.groups.items() for j in range(len(gs))]
        return out

    def step_pipe(self, pipe):
        op = self.pipe[pipe].pop(0)
        if op[0] == "mma":
            for r in op[1]:
                self._add(self.pend_r, r, -1)
            for w, tag in op[2]:
                self._add(self.pend_w, w, -1)
                self.tag[w] = tag
        else:
            self.bars[op[1]].arrive()

    def land(self, k):
        buf, tag, name = self.loads.pop(k)
        self._add(self.pend_w, buf, -1)
        self.tag[buf] = tag
        self.bars[name].arrive()

    def group_read(self, w, j):
        _, half = self.groups[w].pop(j)
        self._add(self.pend_r, half, -1)

    def run(self):
        roles = [self.producer(), self.s_mma(), self.o_mma()]
        roles += [self.softmax(wg, q) for wg in (0, 1) for q in range(4)]
        roles += [self.epilogue(wg, q) for wg in (0, 1) for q in range(4)]
        blocked = [None] * len(roles)
        live = set(range(len(roles)))
        steps = 0
        while live or any(self.pipe.values()) or self.loads or any(self.groups.values()):
            steps += 1
            assert steps < 500000, "no progress"
            ready = [r for r in live if blocked[r] is None or blocked[r]()]
            moves = [("role", r) for r in ready] + [("engine", e) for e in self.engines()]
            assert moves, "deadlock"
            kind, x = self.rng.choice(moves)
            if kind == "engine":
                x()
                continue
            try:
                blocked[x] = next(roles[x])
            except StopIteration:
                live.discard(x)
                blocked[x] = None


def tile_sequence(rng, n_blocks):
    tiles = []
    for blk in range(n_blocks):
        tiles += [blk] * rng.randint(1, 5)
    return tiles


@pytest.mark.parametrize("seed", range(30))
def test_prefill_attend_protocol_random_schedules(seed):
    rng = random.Random(seed)
    Sim(tile_sequence(rng, rng.randint(1, 8)), rng).run()


def test_prefill_attend_protocol_single_tiles():
    # every tile a new block: K, V and the info ring turn over on every tile
    for seed in range(5):
        rng = random.Random(50 + seed)
        Sim(list(range(20)), rng).run()


def test_model_catches_a_missing_o_free_wait():
    failed = 0
    for seed in range(30):
        rng = random.Random(seed)
        try:
            Sim(tile_sequence(rng, 5), rng, skip_o_free=True).run()
        except AssertionError:
            failed += 1
    assert failed > 0


def test_model_catches_a_missing_bulk_read_wait():
    failed = 0
    for seed in range(30):
        rng = random.Random(seed)
        try:
            Sim(tile_sequence(rng, 5), rng, skip_bulk_wait=True).run()
        except AssertionError:
            failed += 1
    assert failed > 0
