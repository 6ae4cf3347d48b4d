"""The bounded on-chip wait on the GPU: a wait that can never complete gives
up, reports MSA_DEVERR_TIMEOUT through the device error word, and leaves the
CUDA context usable.  No fault, trap or endless loop is involved: the waits
poll a shared-memory mbarrier against the GPU's global timer."""
import pytest
import torch

import block_sparse_attention_08_gb300 as msa
import msa_synth
import oracle
from _parity import check_q2k, decode_nb

pytestmark = pytest.mark.gpu

TIMEOUT = 4


def test_wait_gives_up_and_reports():
    (w0, w1), (code, detail) = msa.msa_check_bounded_wait()
    assert code == TIMEOUT and detail == 900          # the first wait's record; the second leaves it
    assert 200e6 <= w0 < 2e9 and 200e6 <= w1 < 2e9    # each ran to the 200 ms limit, then returned


def test_context_usable_after_a_timeout():
    msa.msa_check_bounded_wait()
    d = msa_synth.decode_inputs([300, 5000], paged=True, seed=11, device="cuda")
    q2k = msa.msa_select_blocks_decode(d.index_q, d.index_k_cache, d.seq_lens, page_table=d.page_table,
                                       topk=16, init_blocks=0, local_blocks=1)
    torch.cuda.synchronize()
    ref, gap = oracle.select_decode(d.index_q, d.index_k_cache, d.seq_lens, page_table=d.page_table, topk=16,
                                    init=0, local=1)
    check_q2k(q2k.cpu().numpy(), ref, gap, decode_nb(d.seq_lens, d.max_blocks), 16, 0, 1, "q2k after timeout")
