"""The index producer on the GPU (through the C ABI) against the CPU oracle:
normalised index queries and keys, and the index-K cache after insertion, bit
for bit; then the produced tensors fed straight into the select calls, whose
q2k must match the oracle's selection on the oracle's produced tensors."""
import numpy as np
import pytest
import torch

import block_sparse_attention_08_gb300 as msa
import msa_synth
import oracle
from _parity import check_q2k, decode_nb, prefill_nb

pytestmark = pytest.mark.gpu


def _raw(t):
    t = t.cpu().contiguous()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.view(torch.uint8).numpy()


def _pre_norm(shape, seed, edge=False):
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = (torch.randn(shape, generator=g, device="cuda") * 3.0).to(torch.bfloat16)
    if edge:  # rows the reading singles out: zero, underflowing, -0 elements, overflowing squares
        flat = x.view(-1, 128)
        flat[0] = 0.0
        flat[1] = 2.0 ** -100
        flat[2, :64] = -0.0
        flat[3] = 2.0 ** 70
    return x


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("paged", [True, False])
def test_decode_produce_then_select(dtype, paged):
    lens = [1, 127, 128, 129, 3000, 8191, 20000, 257]
    d = msa_synth.decode_inputs(lens, paged=paged, index_dtype=dtype, seed=31, device="cuda")
    B = d.batch
    iq = _pre_norm((B, 4, 128), 1, edge=True)
    ik = _pre_norm((B, 1, 128), 2)
    cache_before = d.index_k_cache.clone()
    kw = dict(page_table=d.page_table, cu_seqlens_k=d.cu_seqlens_k)
    q_out = msa.msa_index_produce_decode(iq, ik, d.index_k_cache, d.seq_lens, max_blocks=d.max_blocks, **kw)
    torch.cuda.synchronize()
    rq, rcache = oracle.index_produce_decode(iq, ik, cache_before, d.seq_lens, **kw, dtype=dtype)
    assert np.array_equal(_raw(q_out), rq)
    assert np.array_equal(_raw(d.index_k_cache), rcache)
    # the produced index feeds the decode select unchanged
    q2k = msa.msa_select_blocks_decode(q_out, d.index_k_cache, d.seq_lens, max_blocks=d.max_blocks, **kw)
    torch.cuda.synchronize()
    to_t = (lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)) if dtype == "bf16" else \
        (lambda a: torch.from_numpy(a).view(torch.float8_e4m3fn))
    ref_q2k, gap, scores = oracle.select_decode(to_t(rq), to_t(rcache), d.seq_lens, **kw, return_scores=True)
    check_q2k(q2k.cpu().numpy(), ref_q2k, gap, decode_nb(d.seq_lens, d.max_blocks), 16, 0, 1,
              f"decode select on the produced {dtype} index ({'paged' if paged else 'contiguous'})", scores=scores)


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_prefill_produce_then_select(dtype):
    docs = [1, 127, 128, 129, 700, 2049, 3000]
    T = sum(docs)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(docs)]), dtype=torch.int32, device="cuda")
    iq = _pre_norm((T, 4, 128), 3, edge=True)
    ik = _pre_norm((T, 1, 128), 4, edge=True)
    # a paged cache: each document's pages at a random permutation of a pool with two spare pages
    nbs = [(n + 127) // 128 for n in docs]
    pool = sum(nbs) + 2
    perm = np.random.default_rng(5).permutation(pool).astype(np.int32)
    mb = max(nbs)
    pt = np.full((len(docs), mb), -1, np.int32)
    o = 0
    for i, nb in enumerate(nbs):
        pt[i, :nb] = perm[o: o + nb]
        o += nb
    pt = torch.from_numpy(pt).cuda()
    dt = torch.bfloat16 if dtype == "bf16" else torch.float8_e4m3fn
    g = torch.Generator(device="cuda").manual_seed(6)
    cache = torch.randn((pool * 128, 1, 128), generator=g, device="cuda").to(dt)
    cache_before = cache.clone()
    q_out, k_out = msa.msa_index_produce_prefill(iq, ik, cu, index_dtype=dtype, index_k_cache=cache, page_table=pt)
    torch.cuda.synchronize()
    rq, rk, rcache = oracle.index_produce_prefill(iq, ik, cu, dtype=dtype, index_k_cache=cache_before,
                                                  page_table=pt)
    assert np.array_equal(_raw(q_out), rq)
    assert np.array_equal(_raw(k_out), rk)
    assert np.array_equal(_raw(cache), rcache)
    q2k = msa.msa_select_blocks_prefill(q_out, k_out, cu, max(docs))
    torch.cuda.synchronize()
    tok = np.arange(T, dtype=np.int64)
    ref_q2k, gap, scores = oracle.select_prefill(q_out, k_out, cu, tok, return_scores=True)
    check_q2k(q2k.cpu().numpy(), ref_q2k, gap, prefill_nb(cu, tok), 16, 0, 1,
              f"prefill select on the produced {dtype} index", scores=scores)


def test_produce_bad_page_is_reported_not_written():
    d = msa_synth.decode_inputs([300, 5000], paged=True, seed=8, device="cuda")
    pt = d.page_table.clone()
    pt[1, (5000 - 1) // 128] = 10 ** 6          # the new key's page is outside the pool
    ws = msa.Workspace(256)
    before = d.index_k_cache.clone()
    iq, ik = _pre_norm((2, 4, 128), 9), _pre_norm((2, 1, 128), 10)
    msa.msa_index_produce_decode(iq, ik, d.index_k_cache, d.seq_lens, page_table=pt, workspace=ws)
    code, detail = ws.read_device_error()
    assert code == 1 and detail == 1              # MSA_DEVERR_PAGE, request 1
    _, want = oracle.index_produce_decode(iq[:1], ik[:1], before, d.seq_lens[:1], page_table=pt[:1])
    assert np.array_equal(_raw(d.index_k_cache), want)   # only request 0's row was written
