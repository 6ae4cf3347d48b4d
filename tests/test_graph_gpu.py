"""The C-ABI calls captured in a CUDA graph and replayed, as a serving engine
replays its step (and as the bench times it), give the results of the same
calls run eagerly: the decode step bit for bit (its merges add in a fixed
order), the prefill selection bit for bit and its attention within one bf16
ulp (its fp32 row sums are added by the tensor engine in an order that
varies).  The eager results are themselves checked against the oracle by the
other GPU tests."""
import numpy as np
import pytest
import torch

import block_sparse_attention_08_gb300 as msa
import msa_synth
from _parity import SCALE

pytestmark = pytest.mark.gpu


def _capture(step):
    stream = torch.cuda.current_stream()
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            step()
    stream.wait_stream(cap)
    return g


# 4 requests: the attention's cluster form; 40: its stream-K form
@pytest.mark.parametrize("lens", [[3000, 70, 9000, 128 * 20 + 1],
                                  np.random.default_rng(5).integers(1, 20000, size=40).tolist()])
def test_decode_step_in_a_graph(lens):
    d = msa_synth.decode_inputs(lens, paged=True, seed=77, device="cuda")
    kw = dict(page_table=d.page_table, max_blocks=d.max_blocks)
    ws = msa.Workspace(msa.workspace_size(msa.make_config(), 0, d.batch, d.max_blocks))
    q2k = torch.empty((4, d.batch, 16), dtype=torch.int32, device="cuda")
    out = torch.empty((d.batch, 64, 128), dtype=torch.bfloat16, device="cuda")

    def step():
        msa.msa_select_blocks_decode(d.index_q, d.index_k_cache, d.seq_lens, q2k=q2k, workspace=ws, **kw)
        msa.msa_sparse_attend_decode(d.q, d.k_cache, d.v_cache, q2k, d.seq_lens, scale=SCALE, out=out,
                                     workspace=ws, **kw)

    step()
    torch.cuda.synchronize()
    q_ref, o_ref = q2k.clone(), out.clone()
    g = _capture(step)
    for _ in range(3):
        q2k.zero_()
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(q2k, q_ref) and torch.equal(out, o_ref)
    assert ws.read_device_error() == (0, 0)


def test_prefill_step_in_a_graph():
    p = msa_synth.prefill_inputs([3000, 400, 2500], seed=4, device="cuda")
    T = p.total_tokens
    q2k = torch.empty((4, T, 16), dtype=torch.int32, device="cuda")
    out = torch.empty((T, 64, 128), dtype=torch.bfloat16, device="cuda")

    def step():
        msa.msa_select_blocks_prefill(p.index_q, p.index_k, p.cu_seqlens, p.max_seqlen, q2k=q2k)
        msa.msa_sparse_attend_prefill(p.q, p.k, p.v, q2k, p.cu_seqlens, p.max_seqlen, scale=SCALE, out=out)

    step()
    torch.cuda.synchronize()
    q_ref, o_ref = q2k.clone(), out.float()
    g = _capture(step)
    for _ in range(3):
        q2k.zero_()
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(q2k, q_ref)
        d = (out.float() - o_ref).abs()
        assert (d <= 2.0 ** -7 * o_ref.abs() + 1e-6).all(), float(d.max())  # one bf16 ulp
