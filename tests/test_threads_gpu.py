"""Calls from a thread other than the one that allocated the data.

PyTorch's autograd worker and any fresh thread may reach the library with no
CUDA context current; every entry point must still run there (the tensor-map
encoder, a driver call, needs one)."""
import threading

import pytest
import torch

import block_sparse_attention_08_gb300 as msa
import msa_synth
from _parity import SCALE

pytestmark = pytest.mark.gpu


def _on_fresh_thread(fn):
    box = {}

    def run():
        try:
            box["out"] = fn()
            torch.cuda.synchronize()
        except BaseException as e:  # re-raised on the caller's thread
            box["err"] = e

    t = threading.Thread(target=run)
    t.start()
    t.join()
    if "err" in box:
        raise box["err"]
    return box["out"]


def test_prefill_path_on_a_fresh_thread():
    p = msa_synth.prefill_inputs([200, 130], seed=21, device="cuda")
    q2k = msa.msa_select_blocks_prefill(p.index_q, p.index_k, p.cu_seqlens, p.max_seqlen)
    T = p.total_tokens
    lse = torch.empty((T, 64), dtype=torch.float32, device="cuda")
    out = msa.msa_sparse_attend_prefill(p.q, p.k, p.v, q2k, p.cu_seqlens, p.max_seqlen, scale=SCALE, lse=lse)
    dout = torch.randn(out.shape, generator=torch.Generator().manual_seed(22)).to(torch.bfloat16).cuda()
    grads = msa.msa_sparse_attend_prefill_backward(p.q, p.k, p.v, q2k, p.cu_seqlens, p.max_seqlen, out, lse, dout,
                                                   scale=SCALE)
    torch.cuda.synchronize()
    # the same calls on a fresh thread give the same integers, and the forward within one bf16
    # rounding (its fp32 row sums are added in an order that varies)
    q2k_t = _on_fresh_thread(lambda: msa.msa_select_blocks_prefill(p.index_q, p.index_k, p.cu_seqlens,
                                                                   p.max_seqlen))
    assert torch.equal(q2k_t, q2k)
    out_t = _on_fresh_thread(lambda: msa.msa_sparse_attend_prefill(p.q, p.k, p.v, q2k, p.cu_seqlens, p.max_seqlen,
                                                                   scale=SCALE))
    assert ((out_t.float() - out.float()).abs() <= 2.0 ** -7 * out.float().abs() + 1e-6).all()  # one bf16 ulp
    g_t = _on_fresh_thread(lambda: msa.msa_sparse_attend_prefill_backward(
        p.q, p.k, p.v, q2k, p.cu_seqlens, p.max_seqlen, out, lse, dout, scale=SCALE))
    # the gradients are summed with atomics (order varies): compare within bf16 rounding
    for a, b in zip(g_t, grads):
        assert (a.float() - b.float()).abs().max() <= 2e-2 * b.float().abs().max()


def test_decode_path_on_a_fresh_thread():
    d = msa_synth.decode_inputs([300, 4096, 129], paged=True, seed=23, device="cuda")
    q2k = msa.msa_select_blocks_decode(d.index_q, d.index_k_cache, d.seq_lens, page_table=d.page_table)
    out = msa.msa_sparse_attend_decode(d.q, d.k_cache, d.v_cache, q2k, d.seq_lens, d.page_table, scale=SCALE)
    torch.cuda.synchronize()
    q2k_t = _on_fresh_thread(lambda: msa.msa_select_blocks_decode(d.index_q, d.index_k_cache, d.seq_lens,
                                                                  page_table=d.page_table))
    assert torch.equal(q2k_t, q2k)
    out_t = _on_fresh_thread(lambda: msa.msa_sparse_attend_decode(d.q, d.k_cache, d.v_cache, q2k, d.seq_lens,
                                                                  d.page_table, scale=SCALE))
    assert torch.equal(out_t, out)
