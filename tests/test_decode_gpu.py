"""Decode path on the GPU (through the C ABI) against the CPU oracle."""
import numpy as np
import pytest
import torch

import block_sparse_attention_08_gb300 as msa
import msa_synth
import oracle
from _parity import SCALE, check_out, check_q2k, decode_nb

pytestmark = pytest.mark.gpu

SMALL_LENS = [1, 2, 127, 128, 129, 300, 1000, 2048, 2049, 2050, 4095, 5000, 8191]


def _run(d, topk, init, local, label="decode", workspace=None):
    kw = dict(page_table=d.page_table, cu_seqlens_k=d.cu_seqlens_k, max_blocks=d.max_blocks, workspace=workspace)
    q2k = msa.msa_select_blocks_decode(d.index_q, d.index_k_cache, d.seq_lens, topk=topk, init_blocks=init,
                                       local_blocks=local, **kw)
    torch.cuda.synchronize()
    ref_q2k, gap, scores = oracle.select_decode(d.index_q, d.index_k_cache, d.seq_lens, page_table=d.page_table,
                                                cu_seqlens_k=d.cu_seqlens_k, topk=topk, init=init, local=local,
                                                return_scores=True)
    nb = decode_nb(d.seq_lens, d.max_blocks)
    check_q2k(q2k.cpu().numpy(), ref_q2k, gap, nb, topk, init, local, f"{label} (topk {topk}, init {init}, "
              f"local {local})", scores=scores)
    # attention on the oracle's selection (identical q2k on both sides)
    out = msa.msa_sparse_attend_decode(d.q, d.k_cache, d.v_cache, torch.from_numpy(ref_q2k).cuda(), d.seq_lens,
                                       scale=SCALE, **kw)
    torch.cuda.synchronize()
    ref_out = oracle.attend_decode(d.q, d.k_cache, d.v_cache, d.seq_lens, ref_q2k, SCALE,
                                   page_table=d.page_table, cu_seqlens_k=d.cu_seqlens_k)
    check_out(out, ref_out, f"{label} out")
    return q2k, out


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("topk,init,local", [(16, 0, 1), (4, 1, 1), (3, 0, 0), (16, 2, 3), (1, 0, 1)])
def test_decode_small(paged, topk, init, local):
    d = msa_synth.decode_inputs(SMALL_LENS, paged=paged, seed=topk * 7 + init, device="cuda")
    _run(d, topk, init, local)


def test_decode_many_requests():
    # more (request, KV head) segments than SMs several times over: every CTA
    # walks many segments and the stream-K cuts land inside short ones
    lens = np.random.default_rng(71).integers(1, 3000, size=200).tolist()
    d = msa_synth.decode_inputs(lens, paged=True, seed=71, device="cuda")
    _run(d, 16, 1, 1)


@pytest.mark.parametrize("n_req,topk", [(1, 16), (3, 16), (4, 16), (2, 3), (4, 5), (6, 16), (9, 16), (12, 16),
                                        (19, 16), (20, 16), (40, 16), (5, 1)])
def test_decode_request_counts(n_req, topk):
    """Small batches run the attention as one cluster of CTAs per (request, KV
    head) segment, merged through distributed shared memory: clusters of 8 for
    up to 4 requests, of 4 up to 9, of 2 up to 19, never more CTAs per cluster
    than topk (so topk 3 takes clusters of 2, topk 5 of 4 with shares 1, 1, 1, 2,
    topk 1 none).  From 20 requests on, stream-K with merges through global
    memory.  Every size against the oracle."""
    lens = np.random.default_rng(100 + n_req).integers(1, 20000, size=n_req).tolist()
    d = msa_synth.decode_inputs(lens, paged=True, seed=100 + n_req, device="cuda")
    _run(d, topk, 0, 1 if topk > 1 else 0, f"decode {n_req} requests")


def test_decode_no_request_needs_scoring():
    # every context within topk blocks: the scorer has no page to score (its
    # claims and groups are all empty) and the top-k writes every row itself
    lens = [1, 2, 127, 128, 129, 1000, 2047, 2048, 300, 5]
    d = msa_synth.decode_inputs(lens, paged=True, seed=19, device="cuda")
    _run(d, 16, 0, 1, "decode, no request above topk blocks")


def test_decode_rows_longer_than_the_topk_stage():
    # a context of 1200 blocks: its score rows are longer than the 1024 the
    # top-k stages in shared memory, so they are read from global memory as
    # they go; the others are staged
    lens = [1200 * 128 - 5, 3000, 70000]
    d = msa_synth.decode_inputs(lens, paged=True, seed=23, device="cuda")
    _run(d, 16, 1, 1, "decode, a 153 k-token context")


@pytest.mark.parametrize("pattern", ["all equal", "two levels"])
def test_decode_tied_scores(pattern):
    # Exact ties: every key of a context the same vector ("all equal": every
    # block scores the same), or blocks alternating between two vectors ("two
    # levels": half the blocks tie at the higher score).  Ties are broken by the
    # lower block id on both sides, so q2k must match the oracle bit for bit,
    # near-tie exemption or not.  Rows of 301 and 547 blocks put more than 64
    # candidates at the top-k's threshold (its exact fallback path).
    lens = [300 * 128 + 7, 5000, 70000]
    d = msa_synth.decode_inputs(lens, paged=False, seed=31, device="cuda")
    ik = d.index_k_cache
    cu = d.cu_seqlens_k.cpu().tolist()
    for r, L in enumerate(lens):
        a, b = ik[cu[r]].clone(), ik[cu[r] + 1].clone()
        rows = ik[cu[r]:cu[r] + L]
        rows[:] = a
        if pattern == "two levels":
            blk = torch.arange(L, device="cuda") // 128
            rows[blk % 2 == 1] = b
    for topk, init, local in [(16, 0, 1), (16, 2, 3), (5, 1, 0)]:
        kw = dict(page_table=d.page_table, cu_seqlens_k=d.cu_seqlens_k, max_blocks=d.max_blocks)
        q2k = msa.msa_select_blocks_decode(d.index_q, ik, d.seq_lens, topk=topk, init_blocks=init,
                                           local_blocks=local, **kw)
        torch.cuda.synchronize()
        ref, _, _ = oracle.select_decode(d.index_q, ik, d.seq_lens, page_table=d.page_table,
                                         cu_seqlens_k=d.cu_seqlens_k, topk=topk, init=init, local=local,
                                         return_scores=True)
        assert np.array_equal(q2k.cpu().numpy(), ref), (pattern, topk, init, local)


@pytest.mark.parametrize("paged", [False, True])
def test_decode_small_batch_mxfp8_and_fp8_kv(paged):
    # the cluster-merged attention (3 requests: clusters of 8) with both output
    # and cache variants: MXFP8 equal to the quantised bf16 output, FP8 K/V against the oracle
    d = msa_synth.decode_inputs([9000, 300, 20000], paged=paged, seed=13, device="cuda")
    kw = dict(page_table=d.page_table, cu_seqlens_k=d.cu_seqlens_k, max_blocks=d.max_blocks)
    q2k, out = _run(d, 16, 0, 1, "decode 3 requests")
    oq, osc = msa.msa_sparse_attend_decode_mxfp8(d.q, d.k_cache, d.v_cache, q2k, d.seq_lens, scale=SCALE, **kw)
    torch.cuda.synchronize()
    rq, rs = oracle.mxfp8_quantize(out.reshape(out.shape[0], -1))
    assert np.array_equal(oq.cpu().numpy(), rq) and np.array_equal(osc.cpu().numpy(), rs)
    k8, v8 = _fp8_caches(d, 0.25, 0.5)
    out8 = msa.msa_sparse_attend_decode_fp8kv(d.q, k8, v8, q2k, d.seq_lens, k_scale=0.25, v_scale=0.5, scale=SCALE,
                                              **kw)
    torch.cuda.synchronize()
    ref = oracle.attend_decode_fp8(d.q, k8, v8, d.seq_lens, q2k.cpu().numpy(), SCALE, k_scale=0.25, v_scale=0.5,
                                   page_table=d.page_table, cu_seqlens_k=d.cu_seqlens_k)
    check_out(out8, ref, f"decode attention, FP8 K/V, 3 requests ({'paged' if paged else 'contiguous'})")


def test_decode_e4m3_small():
    d = msa_synth.decode_inputs(SMALL_LENS, paged=True, index_dtype="e4m3", seed=3, device="cuda")
    _run(d, 16, 0, 1)


def test_decode_paged_equals_contiguous():
    lens = [700, 4097, 129, 9000]
    a = msa_synth.decode_inputs(lens, paged=True, seed=5, device="cuda")
    pt = a.page_table.cpu().numpy()
    rows = np.concatenate([pt[r, np.arange(L) // 128] * 128 + np.arange(L) % 128 for r, L in enumerate(lens)])
    rows = torch.from_numpy(rows).cuda()
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int64, device="cuda")
    q2k_a = msa.msa_select_blocks_decode(a.index_q, a.index_k_cache, a.seq_lens, page_table=a.page_table)
    q2k_b = msa.msa_select_blocks_decode(a.index_q, a.index_k_cache[rows].contiguous(), a.seq_lens,
                                         cu_seqlens_k=cu, max_blocks=a.max_blocks)
    assert torch.equal(q2k_a, q2k_b)
    oa = msa.msa_sparse_attend_decode(a.q, a.k_cache, a.v_cache, q2k_a, a.seq_lens, page_table=a.page_table)
    ob = msa.msa_sparse_attend_decode(a.q, a.k_cache[rows].contiguous(), a.v_cache[rows].contiguous(), q2k_a,
                                      a.seq_lens, cu_seqlens_k=cu, max_blocks=a.max_blocks)
    assert torch.equal(oa, ob)


def test_decode_repeated_calls_reuse_workspace():
    """Each call clears its own counters, so one workspace serves repeated calls
    of different sizes with identical results."""
    d = msa_synth.decode_inputs([3000, 70, 9000, 128 * 20 + 1], paged=True, seed=9, device="cuda")
    e = msa_synth.decode_inputs([50000, 20000], paged=True, seed=10, device="cuda")
    kw = dict(page_table=d.page_table)
    first = msa.msa_select_blocks_decode(d.index_q, d.index_k_cache, d.seq_lens, **kw)
    o1 = msa.msa_sparse_attend_decode(d.q, d.k_cache, d.v_cache, first, d.seq_lens, **kw)
    for _ in range(3):
        other = msa.msa_select_blocks_decode(e.index_q, e.index_k_cache, e.seq_lens, page_table=e.page_table)
        msa.msa_sparse_attend_decode(e.q, e.k_cache, e.v_cache, other, e.seq_lens, page_table=e.page_table)
        again = msa.msa_select_blocks_decode(d.index_q, d.index_k_cache, d.seq_lens, **kw)
        o2 = msa.msa_sparse_attend_decode(d.q, d.k_cache, d.v_cache, again, d.seq_lens, **kw)
        assert torch.equal(first, again) and torch.equal(o1, o2)


def test_decode_workspace_shared_across_batch_sizes():
    """One workspace serves decode calls of different sizes in any order: a
    64-request call, a 4-request call over long contexts (its block scores
    reach far into the workspace), then the 64-request call again.  The
    attention's merge counters sit at a fixed place that no call's scores or
    partials cover, so every call matches the oracle and the repeated call its
    first result bit for bit."""
    big = msa_synth.decode_inputs(np.random.default_rng(81).integers(1, 6000, size=64).tolist(), paged=True,
                                  seed=81, device="cuda")
    small = msa_synth.decode_inputs([60000, 40000, 30000, 20000], paged=True, seed=82, device="cuda")
    cfg = msa.make_config()
    need = max(msa.workspace_size(cfg, 0, big.batch, big.max_blocks),
               msa.workspace_size(cfg, 0, small.batch, small.max_blocks))
    ws = msa.Workspace(need)
    q2k_a, out_a = _run(big, 16, 0, 1, "decode 64 requests, first call", workspace=ws)
    _run(small, 16, 0, 1, "decode 4 long requests, same workspace", workspace=ws)
    q2k_b, out_b = _run(big, 16, 0, 1, "decode 64 requests, after the 4-request call", workspace=ws)
    assert torch.equal(q2k_a, q2k_b) and torch.equal(out_a, out_b)
    assert ws.read_device_error() == (0, 0)
    # the scorer's page-claim counter (header bytes 128-131) is back at zero
    assert not ws.buf[128:132].any().item()


def test_decode_select_walks_past_unscored_requests():
    """Scored requests (more than topk blocks) between long runs of short
    requests that need no scoring: the scorer's page claims walk past 150
    requests at a time, and a claim's pages cross from one request to the next."""
    lens = [100] * 150 + [40000] + [90] * 170 + [30000, 5000, 2100, 2200, 2177]
    d = msa_synth.decode_inputs(lens, paged=True, seed=91, device="cuda")
    _run(d, 16, 1, 1, "decode, long runs of unscored requests")


def test_decode_bad_page_is_reported_not_faulted():
    d = msa_synth.decode_inputs([3000, 4000], paged=True, seed=2, device="cuda")
    pt = d.page_table.clone()
    pt[1, 3] = 10 ** 6  # outside the pool: the kernel's bounds check skips it
    ws = msa.Workspace(msa.workspace_size(msa.make_config(), 0, 2, pt.shape[1]))
    msa.msa_select_blocks_decode(d.index_q, d.index_k_cache, d.seq_lens, page_table=pt, workspace=ws)
    code, detail = ws.read_device_error()
    assert code == 1 and detail == 1 * pt.shape[1] + 3
    assert ws.read_device_error() == (0, 0)


def test_decode_workload_b4_ctx8k_contig():
    d = msa_synth.workload("decode_b4_ctx8k_contig", device="cuda")
    _run(d, 16, 0, 1, "decode_b4_ctx8k_contig")


@pytest.mark.slow
def test_decode_workload_b64_paged():
    d = msa_synth.workload("decode_b64_ctx4k_64k_paged", device="cuda")
    _run(d, 16, 0, 1, "decode_b64_ctx4k_64k_paged")


@pytest.mark.slow
def test_decode_workload_b16_128k_e4m3():
    d = msa_synth.workload("decode_b16_ctx128k_paged_e4m3", device="cuda")
    _run(d, 16, 0, 1, "decode_b16_ctx128k_paged_e4m3")


@pytest.mark.parametrize("paged", [False, True])
def test_decode_mxfp8_output(paged):
    # the MXFP8 emission equals the MX quantisation of the same call's bf16 output, bit for bit,
    # and that bf16 output matches the oracle
    d = msa_synth.decode_inputs(SMALL_LENS, paged=paged, seed=12, device="cuda")
    kw = dict(page_table=d.page_table, cu_seqlens_k=d.cu_seqlens_k, max_blocks=d.max_blocks)
    q2k, out = _run(d, 16, 0, 1)
    ref_q2k = q2k  # the same q2k for both emissions
    out = msa.msa_sparse_attend_decode(d.q, d.k_cache, d.v_cache, ref_q2k, d.seq_lens, scale=SCALE, **kw)
    oq, osc = msa.msa_sparse_attend_decode_mxfp8(d.q, d.k_cache, d.v_cache, ref_q2k, d.seq_lens, scale=SCALE, **kw)
    torch.cuda.synchronize()
    rq, rs = oracle.mxfp8_quantize(out.reshape(out.shape[0], -1))
    assert np.array_equal(oq.cpu().numpy(), rq)
    assert np.array_equal(osc.cpu().numpy(), rs)


def test_decode_mxfp8_workload_sample():
    d = msa_synth.workload("decode_b64_ctx4k_64k_paged", device="cuda", max_requests=8)
    q2k = msa.msa_select_blocks_decode(d.index_q, d.index_k_cache, d.seq_lens, page_table=d.page_table)
    out = msa.msa_sparse_attend_decode(d.q, d.k_cache, d.v_cache, q2k, d.seq_lens, page_table=d.page_table,
                                       scale=SCALE)
    oq, osc = msa.msa_sparse_attend_decode_mxfp8(d.q, d.k_cache, d.v_cache, q2k, d.seq_lens,
                                                 page_table=d.page_table, scale=SCALE)
    torch.cuda.synchronize()
    rq, rs = oracle.mxfp8_quantize(out.reshape(out.shape[0], -1))
    assert np.array_equal(oq.cpu().numpy(), rq) and np.array_equal(osc.cpu().numpy(), rs)


def _fp8_caches(d, k_scale, v_scale):
    k8 = (d.k_cache.float() / k_scale).to(torch.float8_e4m3fn)
    v8 = (d.v_cache.float() / v_scale).to(torch.float8_e4m3fn)
    return k8, v8


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (0.0625, 0.5), (3.0, 0.2)])
def test_decode_fp8_kv_cache(paged, k_scale, v_scale):
    """The decode attention over an FP8 (E4M3) main K/V cache against the fp64 oracle on the
    same bytes and scales, on the oracle's selection."""
    d = msa_synth.decode_inputs(SMALL_LENS, paged=paged, seed=41, device="cuda")
    k8, v8 = _fp8_caches(d, k_scale, v_scale)
    kw = dict(page_table=d.page_table, cu_seqlens_k=d.cu_seqlens_k)
    ref_q2k, _ = oracle.select_decode(d.index_q, d.index_k_cache, d.seq_lens, **kw)
    q2k = torch.from_numpy(ref_q2k).cuda()
    out = msa.msa_sparse_attend_decode_fp8kv(d.q, k8, v8, q2k, d.seq_lens, k_scale=k_scale, v_scale=v_scale,
                                             max_blocks=d.max_blocks, scale=SCALE, **kw)
    torch.cuda.synchronize()
    ref = oracle.attend_decode_fp8(d.q, k8, v8, d.seq_lens, ref_q2k, SCALE, k_scale=k_scale, v_scale=v_scale, **kw)
    check_out(out, ref, f"decode attention, FP8 K/V ({'paged' if paged else 'contiguous'}, "
                        f"k_scale {k_scale}, v_scale {v_scale})")


def test_decode_fp8_kv_cache_many_requests():
    # many segments per CTA and stream-K cuts inside them, as for the bf16 cache
    lens = np.random.default_rng(72).integers(1, 3000, size=200).tolist()
    d = msa_synth.decode_inputs(lens, paged=True, seed=72, device="cuda")
    k8, v8 = _fp8_caches(d, 1.0, 1.0)
    ref_q2k, _ = oracle.select_decode(d.index_q, d.index_k_cache, d.seq_lens, page_table=d.page_table, topk=16,
                                      init=1, local=1)
    q2k = torch.from_numpy(ref_q2k).cuda()
    out = msa.msa_sparse_attend_decode_fp8kv(d.q, k8, v8, q2k, d.seq_lens, page_table=d.page_table, scale=SCALE)
    torch.cuda.synchronize()
    ref = oracle.attend_decode_fp8(d.q, k8, v8, d.seq_lens, ref_q2k, SCALE, page_table=d.page_table)
    check_out(out, ref, "decode attention, FP8 K/V, 200 requests")


@pytest.mark.slow
def test_decode_fp8_kv_workload_b64_paged():
    d = msa_synth.workload("decode_b64_ctx4k_64k_paged", device="cuda")
    k8, v8 = _fp8_caches(d, 1.0, 1.0)
    q2k = msa.msa_select_blocks_decode(d.index_q, d.index_k_cache, d.seq_lens, page_table=d.page_table)
    out = msa.msa_sparse_attend_decode_fp8kv(d.q, k8, v8, q2k, d.seq_lens, page_table=d.page_table, scale=SCALE)
    torch.cuda.synchronize()
    ref = oracle.attend_decode_fp8(d.q, k8, v8, d.seq_lens, q2k, SCALE, page_table=d.page_table)
    check_out(out, ref, "decode_b64_ctx4k_64k_paged attention, FP8 K/V")
