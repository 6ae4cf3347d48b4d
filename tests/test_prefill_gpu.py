"""Packed-document prefill path on the GPU (through the C ABI) against the CPU oracle."""
import json
import os

import numpy as np
import pytest
import torch

import block_sparse_attention_08_gb300 as msa
import msa_synth
import oracle
from _parity import SCALE, check_out, check_q2k, prefill_nb

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _check(p, tokens=None, topk=16, init=0, local=1, attend=True, label="prefill"):
    """q2k of every token against the oracle (bit-exact but for reported near
    ties); the attention, on the oracle's selection, on `tokens` (all when None)."""
    q2k = msa.msa_select_blocks_prefill(p.index_q, p.index_k, p.cu_seqlens, p.max_seqlen, topk=topk,
                                        init_blocks=init, local_blocks=local)
    torch.cuda.synchronize()
    T = p.total_tokens
    every = np.arange(T, dtype=np.int64)
    ref_q2k, gap, scores = oracle.select_prefill(p.index_q, p.index_k, p.cu_seqlens, every, topk=topk, init=init,
                                                 local=local, return_scores=True)
    check_q2k(q2k.cpu().numpy(), ref_q2k, gap, prefill_nb(p.cu_seqlens, every), topk, init, local,
              f"{label} (topk {topk}, init {init}, local {local})", scores=scores)
    if not attend:
        return
    # attention on the oracle's selection
    tok = every if tokens is None else np.asarray(tokens, dtype=np.int64)
    full = torch.from_numpy(ref_q2k).cuda()
    out = msa.msa_sparse_attend_prefill(p.q, p.k, p.v, full, p.cu_seqlens, p.max_seqlen, scale=SCALE)
    torch.cuda.synchronize()
    ref_out = oracle.attend_prefill(p.q, p.k, p.v, p.cu_seqlens, tok, ref_q2k[:, tok], SCALE)
    check_out(out[torch.from_numpy(tok).cuda()], ref_out, f"{label} out ({len(tok)} of {T} tokens)")


DOCS = [1, 127, 128, 129, 700, 2047, 2048, 2049, 3000, 5000]


@pytest.mark.parametrize("topk,init,local", [(16, 0, 1), (16, 1, 1), (4, 1, 1), (3, 0, 0), (2, 0, 2), (1, 1, 0)])
def test_prefill_small(topk, init, local):
    p = msa_synth.prefill_inputs(DOCS, seed=11 + topk + init, device="cuda")
    _check(p, topk=topk, init=init, local=local, label="prefill small documents")


@pytest.mark.parametrize("topk,init,local", [(16, 0, 1), (16, 1, 1), (3, 0, 0)])
def test_prefill_e4m3_small(topk, init, local):
    # unscaled E4M3 index (the decoded values' dot products, fp32 accumulate)
    p = msa_synth.prefill_inputs(DOCS, seed=21 + topk + init, device="cuda", index_dtype="e4m3")
    assert p.index_q.dtype == torch.float8_e4m3fn
    _check(p, topk=topk, init=init, local=local, attend=(topk == 16 and init == 0),
           label="prefill small documents, E4M3 index")


@pytest.mark.parametrize("pattern", ["all equal", "two levels"])
def test_prefill_tied_scores(pattern):
    # Exact ties: every index key of a document the same vector a ("all
    # equal": every block of a query scores the same), or blocks alternating
    # between a and -a ("two levels": the scores of a query are +s and -s).
    # Ties are broken by the lower block id on both sides, so q2k must match
    # the oracle bit for bit, near-tie exemption or not.
    p = msa_synth.prefill_inputs([3000, 700, 2049], seed=41, device="cuda")
    cu = p.cu_seqlens.cpu().tolist()
    ik = p.index_k
    for d in range(len(cu) - 1):
        rows = ik[cu[d]:cu[d + 1]]
        a = rows[0].clone()
        rows[:] = a
        if pattern == "two levels":
            blk = torch.arange(cu[d + 1] - cu[d], device="cuda") // 128
            rows[blk % 2 == 1] = -a
    T = p.total_tokens
    every = np.arange(T, dtype=np.int64)
    for topk, init, local in [(16, 0, 1), (16, 2, 3), (5, 1, 0)]:
        q2k = msa.msa_select_blocks_prefill(p.index_q, ik, p.cu_seqlens, p.max_seqlen, topk=topk, init_blocks=init,
                                            local_blocks=local)
        torch.cuda.synchronize()
        ref, _, _ = oracle.select_prefill(p.index_q, ik, p.cu_seqlens, every, topk=topk, init=init, local=local,
                                          return_scores=True)
        assert np.array_equal(q2k.cpu().numpy(), ref), (pattern, topk, init, local)


def test_prefill_many_tiny_documents():
    # 400 documents of 1..40 tokens around two longer ones: many documents per
    # bucketing window, most of them a single partial block
    lens = np.random.default_rng(8).integers(1, 41, size=400).tolist()
    p = msa_synth.prefill_inputs(lens[:200] + [2500] + lens[200:] + [700], seed=9, device="cuda")
    _check(p, label="prefill, 402 documents")


def test_prefill_e4m3_repeated_calls_are_identical():
    p = msa_synth.prefill_inputs([2500, 300], seed=6, device="cuda", index_dtype="e4m3")
    a = msa.msa_select_blocks_prefill(p.index_q, p.index_k, p.cu_seqlens, p.max_seqlen)
    for _ in range(2):
        assert torch.equal(a, msa.msa_select_blocks_prefill(p.index_q, p.index_k, p.cu_seqlens, p.max_seqlen))


def test_prefill_single_short_document():
    p = msa_synth.prefill_inputs([37], seed=1, device="cuda")
    _check(p)


def _three_block(index_k_vals):
    T = 384
    iq = torch.zeros(T, 4, 128)
    iq[:, :, 0] = 1.0
    ik = torch.zeros(T, 1, 128)
    for row, val in index_k_vals.items():
        ik[int(row), 0, 0] = val
    v = (torch.arange(T) // 128 + 1).float()[:, None, None].expand(T, 4, 128).contiguous()

    def bf(x):
        return x.to(torch.bfloat16).cuda()
    return bf(iq), bf(ik), bf(torch.zeros(T, 64, 128)), bf(torch.zeros(T, 4, 128)), bf(v)


def test_hand_worked_three_blocks_on_gpu():
    with open(os.path.join(GOLDEN, "hand_worked_3block.json")) as f:
        g = json.load(f)
    cu = torch.tensor([0, 384], dtype=torch.int32, device="cuda")
    for case in g["cases"]:
        topk = case.get("topk_override", g["setup"]["topk"])
        iq, ik, q, k, v = _three_block(case["index_k"])
        q2k = msa.msa_select_blocks_prefill(iq, ik, cu, 384, topk=topk, init_blocks=case["init"],
                                            local_blocks=case["local"])
        out = msa.msa_sparse_attend_prefill(q, k, v, q2k, cu, 384, scale=SCALE)
        for t, exp in case["expect"].items():
            for gg in range(4):
                assert q2k[gg, int(t)].tolist() == exp["q2k"], (case["name"], t, gg)
            np.testing.assert_allclose(out[int(t)].float().cpu().numpy(), exp["out"], atol=1e-2)


def test_prefill_repeated_calls_agree():
    """One workspace serves calls of different sizes: the selection repeats bit
    for bit; the attention's fp32 row sums are added by the tensor engine in an
    order that varies, so its bf16 output repeats to within one bf16 ulp."""
    p = msa_synth.prefill_inputs([3000, 400, 2500], seed=4, device="cuda")
    o = msa_synth.prefill_inputs([9000], seed=5, device="cuda")
    a = msa.msa_select_blocks_prefill(p.index_q, p.index_k, p.cu_seqlens, p.max_seqlen)
    oa = msa.msa_sparse_attend_prefill(p.q, p.k, p.v, a, p.cu_seqlens, p.max_seqlen)
    for _ in range(3):
        x = msa.msa_select_blocks_prefill(o.index_q, o.index_k, o.cu_seqlens, o.max_seqlen)
        msa.msa_sparse_attend_prefill(o.q, o.k, o.v, x, o.cu_seqlens, o.max_seqlen)
        b = msa.msa_select_blocks_prefill(p.index_q, p.index_k, p.cu_seqlens, p.max_seqlen)
        ob = msa.msa_sparse_attend_prefill(p.q, p.k, p.v, b, p.cu_seqlens, p.max_seqlen)
        assert torch.equal(a, b)
        d = (oa.float() - ob.float()).abs()
        assert (d <= 2.0 ** -7 * oa.float().abs() + 1e-6).all(), float(d.max())  # one bf16 ulp


def _sample_tokens(cu, n, seed):
    cu = np.asarray(cu.cpu(), dtype=np.int64)
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(cu[-1], size=n, replace=False).tolist())
    for d in range(len(cu) - 1):  # document edges and block edges
        for off in (0, 1, 127, 128, 129, 2047, 2048):
            if cu[d] + off < cu[d + 1]:
                pick.add(int(cu[d] + off))
        pick.add(int(cu[d + 1] - 1))
    return np.array(sorted(pick), dtype=np.int64)


# The full-size workloads: q2k of every token against the oracle; the attention
# on a sample of tokens (random ones plus document and block edges).

@pytest.mark.slow
def test_prefill_workload_1doc_16k():
    p = msa_synth.workload("prefill_1doc_16k", device="cuda")
    _check(p, tokens=_sample_tokens(p.cu_seqlens, 384, 0), label="prefill_1doc_16k")


@pytest.mark.slow
def test_prefill_workload_1doc_16k_e4m3():
    p = msa_synth.workload("prefill_1doc_16k_e4m3", device="cuda")
    _check(p, attend=False, label="prefill_1doc_16k_e4m3")


@pytest.mark.slow
def test_prefill_workload_packed_2x32k():
    p = msa_synth.workload("prefill_packed_2x32k", device="cuda")
    _check(p, tokens=_sample_tokens(p.cu_seqlens, 384, 1), init=1, local=1, label="prefill_packed_2x32k")


def test_prefill_attend_empty_rows_and_bad_ids():
    """A (query, KV head) row with no block outputs zeros; an id at or past the
    query's block count is skipped and reported in the device error word
    (MSA_DEVERR_BLOCK = 2, detail = the flat q2k index), the rest of the row is
    attended as usual."""
    from block_sparse_attention_08_gb300 import binding
    p = msa_synth.prefill_inputs([300, 700], seed=6, device="cuda")
    T = p.total_tokens
    tok = np.arange(T, dtype=np.int64)
    topk = 4
    ref_q2k, _ = oracle.select_prefill(p.index_q, p.index_k, p.cu_seqlens, tok, topk=topk, init=1, local=1)
    q2k = ref_q2k.copy()
    q2k[1, 5, :] = -1                # token 5, KV head 1: nothing to attend
    t_bad = 300 + 600                # document 1, position 600: blocks 0..4
    j_bad = int(np.argmax(q2k[2, t_bad] >= 0))
    q2k[2, t_bad, j_bad] = 5         # one past its last causal block
    ws_q2k = torch.from_numpy(q2k).cuda()
    msa.msa_select_blocks_prefill(p.index_q, p.index_k, p.cu_seqlens, p.max_seqlen, topk=topk, init_blocks=1,
                                  local_blocks=1)  # sizes the shared workspace
    ws = binding._WS[("prefill", "cuda:0")]
    ws.read_device_error()           # clear the error word
    out = msa.msa_sparse_attend_prefill(p.q, p.k, p.v, ws_q2k, p.cu_seqlens, p.max_seqlen, scale=SCALE)
    torch.cuda.synchronize()
    code, detail = ws.read_device_error()
    assert code == 2 and detail == (2 * T + t_bad) * topk + j_bad, (code, detail)
    ref = q2k.copy()
    ref[2, t_bad, j_bad] = -1        # the skipped id
    ref_out = oracle.attend_prefill(p.q, p.k, p.v, p.cu_seqlens, tok, ref, SCALE)
    o = out.float().cpu().numpy()
    assert not o[5, 16:32].any()
    check_out(out, ref_out, "prefill out with empty and bad rows")


def test_prefill_far_block_within_the_reference_range():
    """Keys of block 0 scored far above the local block (exponents up to about 2^40
    over each row's reference) are summed exactly against the fixed reference."""
    p = msa_synth.prefill_inputs([900, 400], seed=13, device="cuda")
    k = p.k.clone()
    k[:128] = (k[:128].float() * 8).to(torch.bfloat16)      # document 0, block 0
    k[900:1028] = (k[900:1028].float() * 8).to(torch.bfloat16)  # document 1, block 0
    T = p.total_tokens
    tok = np.arange(T, dtype=np.int64)
    ref_q2k, _ = oracle.select_prefill(p.index_q, p.index_k, p.cu_seqlens, tok, topk=4, init=1, local=1)
    ws = msa.Workspace(msa.workspace_size(msa.make_config(4, 1, 1), 1, T, (p.max_seqlen + 127) // 128))
    out = msa.msa_sparse_attend_prefill(p.q, k, p.v, torch.from_numpy(ref_q2k).cuda(), p.cu_seqlens, p.max_seqlen,
                                        scale=SCALE, workspace=ws)
    torch.cuda.synchronize()
    assert ws.read_device_error() == (0, 0)
    ref = oracle.attend_prefill(p.q, k, p.v, p.cu_seqlens, tok, ref_q2k, SCALE)
    check_out(out, ref, "prefill, block 0 scored up to 2^40 above the reference")


def test_prefill_score_past_the_reference_range_is_reported():
    """One key of block 0 scores 2^115 above the local block's max for KV head 1:
    MSA_DEVERR_RANGE is recorded; the other KV heads' rows are exact."""
    T = 300
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    q = torch.zeros(T, 64, 128)
    q[:, :, 0] = 30.0
    k = torch.zeros(T, 4, 128)
    k[10, 1, 0] = 30.0          # s = 900 for head group 1 against key 10; every other score is 0
    v = torch.randn(T, 4, 128, generator=torch.Generator().manual_seed(3))
    q, k, v = (x.to(torch.bfloat16).cuda() for x in (q, k, v))
    q2k = torch.full((4, T, 2), -1, dtype=torch.int32)
    pos = torch.arange(T)
    q2k[:, :, 0] = 0
    q2k[:, :, 1] = torch.where(pos >= 128, pos // 128, torch.tensor(-1))
    q2k = q2k.cuda()
    ws = msa.Workspace(msa.workspace_size(msa.make_config(2, 0, 1), 1, T, 3))
    out = msa.msa_sparse_attend_prefill(q, k, v, q2k, cu, T, scale=SCALE, workspace=ws)
    torch.cuda.synchronize()
    code, detail = ws.read_device_error()
    assert code == 5 and (detail // 2) // T == 1, (code, detail)   # an entry of KV head 1
    ref = oracle.attend_prefill(q, k, v, cu, np.arange(T, dtype=np.int64), q2k.cpu().numpy(), SCALE)
    for g in (0, 2, 3):
        check_out(out[:, 16 * g:16 * g + 16], ref[:, 16 * g:16 * g + 16], f"prefill out of range: KV head {g}")
