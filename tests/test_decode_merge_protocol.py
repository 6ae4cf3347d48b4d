"""Host model of the decode attention's stream-K merge (sparse_attend_kernel,
the form without clusters).

The units (query, KV head, selected block) are split evenly over the grid, so
a (query, KV head) segment of topk units can be cut between consecutive CTAs.
Each contributor of a cut segment, when it has finished its units:

  1. loads the segment's counter with acquire semantics; if the other
     contributors' counts are all in it, it completes the segment and merges
     at once, from its own state and their published partials;
  2. otherwise publishes its partial (max, sum, O) in its slot, fences, adds
     its unit count to the counter, and merges if that add completed it.

The merger resets the counter to zero.  The model runs the contributors of
every cut segment under random interleavings of these steps and checks that
exactly one contributor merges, that it reads only partials already
published, that it combines every contributor once, and that the counter ends
at zero.  It also checks the slot arithmetic: the slot a contributor writes is
the slot the merger reads for it, and no two cut segments share a slot or a
counter.  A contributor that adds before it publishes (a planted mistake) must
be reported.  No GPU is involved.
"""
import random

import pytest

from _kernel_consts import kconst

MAX_TOPK = kconst("kMaxTopk", "launch.h")


# the kernel's stream-K partition (seg_begin / cta_of) and partial slots
def seg_begin(c, N, G):
    return c * N // G


def cta_of(i, N, G):
    c = i * G // N
    while c + 1 < G and seg_begin(c + 1, N, G) <= i:
        c += 1
    while c > 0 and seg_begin(c, N, G) > i:
        c -= 1
    return c


def writer_slot(c, range0, N, G):
    """Slot a CTA writes a cut segment's partial into: its first segment -> 2c, its last -> 2c+1."""
    return 2 * c + (0 if range0 <= seg_begin(c, N, G) else 1)


def merger_slot(x, c_first, range0, N, G):
    """Slot the merger reads contributor x (0 = c_first) from."""
    if x == 0:
        return 2 * c_first + (1 if seg_begin(c_first, N, G) < range0 else 0)
    return 2 * (c_first + x)


def cut_segments(N, G, topk):
    """(range0, [(cta, units)]) for every segment split over more than one CTA."""
    out = []
    for seg in range(N // topk):
        range0 = seg * topk
        c0, c1 = cta_of(range0, N, G), cta_of(range0 + topk - 1, N, G)
        if c0 == c1:
            continue
        parts = []
        for c in range(c0, c1 + 1):
            lo, hi = max(range0, seg_begin(c, N, G)), min(range0 + topk, seg_begin(c + 1, N, G))
            assert hi > lo
            parts.append((c, hi - lo))
        out.append((range0, parts))
    return out


@pytest.mark.parametrize("batch,G,topk", [(64, 152, 16), (4, 152, 16), (16, 152, 16), (1000, 152, 16),
                                          (7, 40, 5), (33, 304, 16), (3, 17, 3), (2, 152, 1)])
def test_slots_and_counters(batch, G, topk):
    N = batch * 4 * topk
    G = min(G, N)
    slots, counters = {}, {}
    for range0, parts in cut_segments(N, G, topk):
        assert len(parts) <= topk and len(parts) <= MAX_TOPK
        c_first = parts[0][0]
        assert c_first not in counters, "two cut segments share a counter"
        counters[c_first] = range0
        for x, (c, _) in enumerate(parts):
            w = writer_slot(c, range0, N, G)
            assert w == merger_slot(x, c_first, range0, N, G), (range0, x, c)
            assert w not in slots, "two cut segments share a partial slot"
            slots[w] = range0
            assert 0 <= w < 2 * G


def run_segment(parts, topk, rng, add_before_publish=False):
    """One cut segment's contributors under a random interleaving of their steps."""
    state = {"ticket": 0, "published": set(), "mergers": [], "combined": None}
    n = len(parts)

    def contributor(x, cnt):
        yield  # finished its units, at a random moment
        v = state["ticket"]  # acquire load
        yield
        if v + cnt == topk:
            merge(x)
            return
        if add_before_publish:
            old = state["ticket"]
            state["ticket"] += cnt
            yield
            state["published"].add(x)
        else:
            state["published"].add(x)  # partial written and fenced
            yield
            old = state["ticket"]
            state["ticket"] += cnt  # atomic add
        yield
        if old + cnt == topk:
            merge(x)

    def merge(x):
        state["mergers"].append(x)
        for y in range(n):
            if y != x:
                assert y in state["published"], f"contributor {x} merged before {y} published its partial"
        state["combined"] = sorted(range(n))
        state["ticket"] = 0

    live = [contributor(x, cnt) for x, (_, cnt) in enumerate(parts)]
    while live:
        g = rng.choice(live)
        try:
            next(g)
        except StopIteration:
            live.remove(g)
    assert len(state["mergers"]) == 1, f"{len(state['mergers'])} contributors merged"
    assert state["combined"] == list(range(n))
    assert state["ticket"] == 0


@pytest.mark.parametrize("seed", range(4))
def test_merge_protocol_random_schedules(seed):
    rng = random.Random(seed)
    for batch, G, topk in [(64, 152, 16), (5, 152, 16), (7, 40, 5), (1, 64, 16)]:
        N = batch * 4 * topk
        for _, parts in cut_segments(N, min(G, N), topk):
            for _ in range(50):
                run_segment(parts, topk, rng)


def test_model_reports_add_before_publish():
    rng = random.Random(0)
    parts = [(0, 5), (1, 6), (2, 5)]
    caught = 0
    for _ in range(300):
        try:
            run_segment(parts, 16, rng, add_before_publish=True)
        except AssertionError:
            caught += 1
    assert caught > 0
