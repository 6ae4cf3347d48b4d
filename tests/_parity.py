"""Comparison helpers shared by the GPU parity tests."""
import math

import numpy as np
import torch

SCALE = 1.0 / math.sqrt(128.0)
ATOL_MAX = 1e-2    # max-abs error of the bf16 output against the fp64 oracle
ATOL_MEAN = 1e-3   # mean-abs error
GAP_REL = 1e-5     # near-tie exemption of the k-th / (k+1)-th score
BF16_HALF_ULP_REL = 2.0 ** -8  # rounding of an exact value to the bf16 output

# One entry per parity comparison made in this process: printed in the pytest
# terminal summary (tests/conftest.py), so every run reports its differing and
# exempt q2k rows and how many output elements needed the bf16-rounding allowance.
REPORT = []


def check_q2k(gpu_q2k, ref_q2k, gap, nb, topk, init, local, label="", scores=None):
    """Bit-exact q2k except rows whose top-k boundary is a near tie (gap < 1e-5
    relative); those rows are reported and must still be valid selections.
    gpu_q2k / ref_q2k: [G, n, topk]; nb: [n] candidate blocks per query;
    scores: the oracle's block scores [n, G, max_nb] (fp64; the decision is taken
    on their fp32 rounding).  With scores, every block on which a differing
    exempt row disagrees with the oracle must score within 1e-5 relative of the
    oracle's k-th kept score (the last kept non-forced block): the GPU may swap
    only near-tied blocks.  Returns (rows that differ, exempt rows)."""
    gpu = np.asarray(gpu_q2k)
    ref = np.asarray(ref_q2k)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    diff = (gpu != ref).any(axis=2)
    exempt = np.asarray(gap) < GAP_REL
    bad = diff & ~exempt
    if bad.any():
        g, i = np.argwhere(bad)[0]
        raise AssertionError(f"{label}: q2k mismatch at head {g} row {i}: gpu {gpu[g, i]} ref {ref[g, i]} "
                             f"(nb={nb[i]}, gap={gap[g, i]:.3g}); {bad.sum()} bad rows")
    for g, i in np.argwhere(diff):
        row = gpu[g, i]
        sel = [b for b in row if b >= 0]
        n = int(nb[i])
        assert row.tolist() == sel + [-1] * (topk - len(sel))
        assert sel == sorted(set(sel)) and len(sel) == min(topk, n)
        forced = {b for b in range(n) if b < init or b >= n - local} if n > topk else set()
        assert forced <= set(sel)
        if scores is not None:
            s32 = np.asarray(scores[i, g, :n], dtype=np.float64).astype(np.float32).astype(np.float64)
            kept = [b for b in ref[g, i] if b >= 0 and b not in forced]
            s_k = min(s32[b] for b in kept)
            for b in set(sel) ^ {int(x) for x in ref[g, i] if x >= 0}:
                den = max(abs(s32[b]), abs(s_k))
                assert abs(s32[b] - s_k) <= GAP_REL * den, \
                    f"{label}: head {g} row {i} swaps block {b} (score {s32[b]!r}) outside the tie band of " \
                    f"the k-th score {s_k!r}"
    nd, ne = int(diff.sum()), int(exempt.sum())
    REPORT.append(f"{label}: q2k {gpu.shape[0] * gpu.shape[1]} rows, {nd} differ, {ne} exempt (near tie)")
    return nd, ne


def check_out(gpu_out, ref_out, label=""):
    """max-abs <= 1e-2 beyond the rounding of each element to the bf16 output
    (half an ulp, at most 2^-8 |ref|), mean-abs <= 1e-3."""
    g = gpu_out.float().cpu().double().numpy() if isinstance(gpu_out, torch.Tensor) else np.asarray(gpu_out)
    r = np.asarray(ref_out)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.isfinite(g).all(), f"{label}: non-finite output"
    err = np.abs(g - r)
    excess = float((err - BF16_HALF_ULP_REL * np.abs(r)).max())
    mx, mean = float(err.max()), float(err.mean())
    assert excess <= ATOL_MAX and mean <= ATOL_MEAN, \
        f"{label}: max-abs {mx:.3g} (beyond bf16 rounding {excess:.3g}) mean-abs {mean:.3g}"
    allowance = int((err > ATOL_MAX).sum())
    REPORT.append(f"{label}: out {err.size} elements, max-abs {mx:.3g}, mean-abs {mean:.3g}, "
                  f"{allowance} above 1e-2 (within the bf16-rounding allowance)")
    return mx, mean


def decode_nb(seq_lens, max_blocks=None):
    L = np.asarray(seq_lens.cpu() if isinstance(seq_lens, torch.Tensor) else seq_lens, dtype=np.int64)
    nb = (L + 127) // 128
    return nb if max_blocks is None else np.minimum(nb, max_blocks)


def prefill_nb(cu_seqlens, tokens):
    cu = np.asarray(cu_seqlens.cpu() if isinstance(cu_seqlens, torch.Tensor) else cu_seqlens, dtype=np.int64)
    tokens = np.asarray(tokens, dtype=np.int64)
    d = np.searchsorted(cu, tokens, side="right") - 1
    return (tokens - cu[d]) // 128 + 1
