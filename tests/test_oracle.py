"""Pins for the CPU oracle (no GPU).

Each test ties the oracle to something other than itself: values worked by hand
from the pages' definitions (tests/golden), the OCP E4M3 encoding, closed forms,
invariants of the selection rule, exhaustive enumeration on tiny inputs, and a
library routine (dense causal attention) in the regime where the sparse method
reduces to it.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import msa_synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SCALE = 1.0 / math.sqrt(128.0)


def _bf16(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


# ---- E4M3 decoding (OCP 8-bit FP, E4M3 "fn") --------------------------------

def test_e4m3_special_values():
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
             0x38: 1.0, 0x3C: 1.5, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0, 0x80: -0.0}
    for b, v in cases.items():
        assert oracle.e4m3_value(b) == v, hex(b)
    assert math.isnan(oracle.e4m3_value(0x7F))
    assert math.isnan(oracle.e4m3_value(0xFF))


def test_e4m3_matches_torch_for_every_byte():
    allb = torch.arange(256, dtype=torch.uint8)
    ref = allb.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for b in range(256):
        mine = oracle.e4m3_value(b)
        if math.isnan(ref[b]):
            assert math.isnan(mine)
        else:
            assert mine == ref[b], b


# ---- the hand-worked three-block example -------------------------------------

def _three_block_inputs(index_k_vals):
    T = 384
    iq = np.zeros((T, 4, 128), np.float32)
    iq[:, :, 0] = 1.0
    ik = np.zeros((T, 1, 128), np.float32)
    for row, val in index_k_vals.items():
        ik[int(row), 0, 0] = val
    q = np.zeros((T, 64, 128), np.float32)
    k = np.zeros((T, 4, 128), np.float32)
    v = np.zeros((T, 4, 128), np.float32)
    v[:] = (np.arange(T) // 128 + 1).astype(np.float32)[:, None, None]
    return _bf16(iq), _bf16(ik), _bf16(q), _bf16(k), _bf16(v)


def _golden_cases():
    with open(os.path.join(GOLDEN, "hand_worked_3block.json")) as f:
        g = json.load(f)
    return g["cases"], g["setup"]["topk"]


@pytest.mark.parametrize("case", _golden_cases()[0], ids=lambda c: c["name"])
def test_hand_worked_three_blocks(case):
    topk = case.get("topk_override", _golden_cases()[1])
    iq, ik, q, k, v = _three_block_inputs(case["index_k"])
    cu = np.array([0, 384], np.int32)
    toks = np.array([int(t) for t in case["expect"]], np.int64)
    q2k, gap, scores = oracle.select_prefill(iq, ik, cu, toks, topk=topk, init=case["init"],
                                             local=case["local"], return_scores=True)
    out = oracle.attend_prefill(q, k, v, cu, toks, q2k, SCALE)
    for i, (t, exp) in enumerate(case["expect"].items()):
        for g in range(4):
            assert list(q2k[g, i]) == exp["q2k"], (t, g)
        np.testing.assert_allclose(out[i], exp["out"], rtol=0, atol=1e-12)
        if "scores" in exp:
            for g in range(4):
                np.testing.assert_array_equal(scores[i, g, :3], exp["scores"])


# ---- document locality -------------------------------------------------------

def test_blocks_restart_at_each_document():
    # two documents of 200 and 300 tokens; doc 2's block ids restart at 0
    T = 500
    iq = np.zeros((T, 4, 128), np.float32)
    iq[:, :, 0] = 1.0
    ik = np.zeros((T, 1, 128), np.float32)
    ik[10, 0, 0] = 0.9      # doc 1, block 0: must not leak into doc 2
    ik[200 + 5, 0, 0] = 0.25   # doc 2, local block 0
    ik[200 + 130, 0, 0] = 0.5  # doc 2, local block 1
    cu = np.array([0, 200, 500], np.int32)
    toks = np.array([499, 199], np.int64)  # doc 2 pos 299 (nb=3); doc 1 pos 199 (nb=2)
    q2k, _, scores = oracle.select_prefill(_bf16(iq), _bf16(ik), cu, toks, topk=2, init=0, local=1,
                                           return_scores=True)
    assert list(q2k[0, 0]) == [1, 2]
    np.testing.assert_array_equal(scores[0, 0, :3], [0.25, 0.5, 0.0])
    assert list(q2k[0, 1]) == [0, 1]


# ---- selection: invariants and exhaustive enumeration ------------------------

def _random_prefill(T, seed, topk=4, init=0, local=1):
    p = msa_synth.prefill_inputs([T], seed=seed, topk=topk, init_blocks=init, local_blocks=local)
    toks = np.arange(T, dtype=np.int64)
    q2k, gap, scores = oracle.select_prefill(p.index_q, p.index_k, p.cu_seqlens, toks, topk=topk,
                                             init=init, local=local, return_scores=True)
    return p, toks, q2k, gap, scores


@pytest.mark.parametrize("init,local", [(0, 1), (1, 1), (2, 0), (0, 0), (1, 2)])
def test_selection_invariants(init, local):
    topk = 4
    _, toks, q2k, gap, scores = _random_prefill(1100, seed=3, topk=topk, init=init, local=local)
    for i, t in enumerate(toks):
        nb = t // 128 + 1
        forced = {b for b in range(nb) if b < init or b >= nb - local}
        for g in range(4):
            row = list(q2k[g, i])
            sel = [b for b in row if b >= 0]
            assert row == sel + [-1] * (topk - len(sel))
            assert sel == sorted(set(sel))
            assert all(0 <= b < nb for b in sel)
            assert len(sel) == min(topk, nb)
            if nb > topk:
                assert forced <= set(sel)
                s32 = scores[i, g, :nb].astype(np.float32)
                free_sel = [s32[b] for b in sel if b not in forced]
                free_rej = [s32[b] for b in range(nb) if b not in forced and b not in sel]
                if free_sel and free_rej:
                    assert min(free_sel) >= max(free_rej)


def test_selection_exhaustive_subsets():
    """For nb <= 10, the kept non-forced set is the unique size-need subset with
    the largest score sum (scores are distinct in fp32 here)."""
    topk, init, local = 4, 1, 1
    _, toks, q2k, _, scores = _random_prefill(1280, seed=5, topk=topk, init=init, local=local)
    checked = 0
    for i, t in enumerate(toks[::7]):
        i = i * 7
        nb = int(t // 128 + 1)
        if nb <= topk:
            continue
        forced = {b for b in range(nb) if b < init or b >= nb - local}
        free = [b for b in range(nb) if b not in forced]
        need = topk - len(forced)
        for g in range(4):
            s32 = scores[i, g, :nb].astype(np.float32).astype(np.float64)
            if len(set(s32[free])) != len(free):
                continue
            best = max(itertools.combinations(free, need), key=lambda c: sum(s32[list(c)]))
            assert sorted(forced | set(best)) == [b for b in q2k[g, i] if b >= 0]
            checked += 1
    assert checked > 100


def test_power_of_two_scaling_keeps_selection():
    p, toks, q2k, _, _ = _random_prefill(900, seed=11)
    iq2 = (p.index_q.float() * 2).to(torch.bfloat16)
    q2k2, _ = oracle.select_prefill(iq2, p.index_k, p.cu_seqlens, toks, topk=4)
    np.testing.assert_array_equal(q2k, q2k2)


def test_exempt_rows_are_rare_and_reported():
    _, _, _, gap, _ = _random_prefill(1500, seed=2)
    ex = oracle.exempt_rows(gap)
    assert ex.sum() < 0.02 * ex.size


# ---- the near-tie gap (the exemption's only input) ---------------------------
#
# One 640-token document; the query at position 639 has nb = 5 candidate blocks,
# block 4 is forced (local 1) and topk 3 leaves need = 2 of blocks 0..3 to the
# scores.  Every key of block b holds the same index key (a_b, c_b, 0, ...) and
# every index query is (1, 1, 0, ...), so block b scores exactly a_b + c_b (both
# bf16, the sum exact in fp32).  The gap is |s_k - s_k+1| / max(|s_k|, |s_k+1|)
# between the k-th kept and the first rejected non-forced score, in the
# (score desc, id asc) order.

def _gap_case(block_scores):
    T = 640
    iq = np.zeros((T, 4, 128), np.float32)
    iq[:, :, 0] = 1.0
    iq[:, :, 1] = 1.0
    ik = np.zeros((T, 1, 128), np.float32)
    for b, (a, c) in enumerate(block_scores):
        ik[128 * b: 128 * (b + 1), 0, 0] = a
        ik[128 * b: 128 * (b + 1), 0, 1] = c
    cu = np.array([0, T], np.int32)
    toks = np.array([639, 200], np.int64)
    q2k, gap, scores = oracle.select_prefill(_bf16(iq), _bf16(ik), cu, toks, topk=3, init=0, local=1,
                                             return_scores=True)
    return q2k, gap, scores


E18, E16 = 2.0 ** -18, 2.0 ** -16


@pytest.mark.parametrize("name,blocks,keep,gap,exempt", [
    # k-th 1, next 1 - 2^-18: a near tie (3.8e-6 < 1e-5)
    ("near_tie", [(2.0, 0.0), (1.0, 0.0), (1.0, -E18), (0.25, 0.0), (0.0, 0.0)], [0, 1, 4], E18, True),
    # k-th 1, next 1 - 2^-16: 1.5e-5, decided by score
    ("decided", [(2.0, 0.0), (1.0, 0.0), (1.0, -E16), (0.25, 0.0), (0.0, 0.0)], [0, 1, 4], E16, False),
    # the near tie sits above the boundary (1st and 2nd); the boundary (2nd 1 - 2^-18,
    # 3rd 0.5) is decided: a gap taken between the wrong pair would call it exempt
    ("tie_above_boundary", [(1.0, 0.0), (1.0, -E18), (0.5, 0.0), (0.25, 0.0), (0.0, 0.0)], [0, 1, 4],
     (0.5 - E18) / (1.0 - E18), False),
    # the near tie sits below the boundary (3rd and 4th), the boundary gap is 0.5
    ("tie_below_boundary", [(2.0, 0.0), (1.0, 0.0), (0.5, 0.0), (0.5, -E18), (0.0, 0.0)], [0, 1, 4], 0.5, False),
    # negative scores: k-th -0.5, next -(0.5 + 2^-18); relative to the larger magnitude
    ("negative", [(1.0, 0.0), (-0.5, 0.0), (-0.5, -E18), (-1.0, 0.0), (0.0, 0.0)], [0, 1, 4],
     E18 / (0.5 + E18), True),
    # an exact tie at the boundary: the lower id is kept, the gap is 0 (exempt)
    ("exact_tie", [(2.0, 0.0), (1.0, 0.0), (1.0, 0.0), (0.25, 0.0), (0.0, 0.0)], [0, 1, 4], 0.0, True),
    # the forced block's score plays no part, however close it is to the boundary
    ("forced_not_counted", [(2.0, 0.0), (1.0, 0.0), (0.5, 0.0), (0.25, 0.0), (1.0, -E18)], [0, 1, 4], 0.5,
     False),
])
def test_near_tie_gap(name, blocks, keep, gap, exempt):
    q2k, g, scores = _gap_case(blocks)
    for h in range(4):
        assert list(q2k[h, 0]) == keep, name
        np.testing.assert_array_equal(scores[0, h, :5], [a + c for a, c in blocks])
        assert g[h, 0] == gap, (name, g[h, 0], gap)
        assert bool(oracle.exempt_rows(g)[h, 0]) == exempt, name
        # position 200: nb = 2 <= topk, nothing is decided by score
        assert g[h, 1] == np.inf and not oracle.exempt_rows(g)[h, 1]
        assert list(q2k[h, 1]) == [0, 1, -1]


def test_near_tie_gap_decode_matches_prefill():
    # the decode select reports the same gap for the same context (query at position 639)
    q2k_p, g_p, _ = _gap_case([(2.0, 0.0), (1.0, 0.0), (1.0, -E18), (0.25, 0.0), (0.0, 0.0)])
    T = 640
    iq = np.zeros((1, 4, 128), np.float32)
    iq[:, :, :2] = 1.0
    ik = np.zeros((T, 1, 128), np.float32)
    for b, (a, c) in enumerate([(2.0, 0.0), (1.0, 0.0), (1.0, -E18), (0.25, 0.0), (0.0, 0.0)]):
        ik[128 * b: 128 * (b + 1), 0, 0] = a
        ik[128 * b: 128 * (b + 1), 0, 1] = c
    q2k_d, g_d, s_d = oracle.select_decode(_bf16(iq), _bf16(ik), np.array([T], np.int32),
                                           cu_seqlens_k=np.array([0, T], np.int64), topk=3, init=0, local=1,
                                           return_scores=True)
    np.testing.assert_array_equal(q2k_d[:, 0], q2k_p[:, 0])
    np.testing.assert_array_equal(g_d[:, 0], g_p[:, 0])
    np.testing.assert_array_equal(s_d[0, :, :5], np.tile([2.0, 1.0, 1.0 - E18, 0.25, 0.0], (4, 1)))
