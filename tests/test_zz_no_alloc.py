"""The allocation-free decode select, called through the C ABI.

Callers that cannot allocate device memory (a runtime without an allocator of
its own, a plugin handed only its input and output buffers) use
msa_select_blocks_decode_noalloc, which keeps its scratch in a fixed array
inside the library.  Its q2k must equal the workspace version's, bit for bit
(the tolerance of every q2k test here), on two calls in a row.  This file is
collected last so that a run stopping at the first failure has run every other
test first.
"""
import ctypes

import pytest
import torch

import block_sparse_attention_08_gb300 as msa
import msa_synth
from block_sparse_attention_08_gb300.binding import msa_config

pytestmark = pytest.mark.gpu


def _fn():
    lib = msa.load()
    f = lib.msa_select_blocks_decode_noalloc
    P = ctypes.c_void_p
    f.argtypes = [ctypes.POINTER(msa_config), P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int64, P, P]
    f.restype = ctypes.c_int
    return f


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(d, q2k, dtype):
    cfg = msa.make_config(d.topk, d.init_blocks, d.local_blocks, dtype)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return _fn()(ctypes.byref(cfg), _ptr(d.index_q), _ptr(d.index_k_cache), _ptr(d.seq_lens), _ptr(d.page_table),
                 _ptr(d.cu_seqlens_k), d.batch, d.max_blocks, d.index_k_cache.shape[0], _ptr(q2k), stream)


@pytest.mark.parametrize("paged,dtype", [(True, "bf16"), (False, "bf16"), (True, "e4m3")])
def test_noalloc_select_matches_workspace_select_twice(paged, dtype):
    d = msa_synth.decode_inputs([1, 300, 2049, 5000, 9000, 20000], paged=paged, index_dtype=dtype, seed=21,
                                device="cuda")
    ref = msa.msa_select_blocks_decode(d.index_q, d.index_k_cache, d.seq_lens, page_table=d.page_table,
                                       cu_seqlens_k=d.cu_seqlens_k, max_blocks=d.max_blocks)
    for _ in range(2):
        q2k = torch.full((4, d.batch, d.topk), -7, dtype=torch.int32, device="cuda")
        assert _noalloc(d, q2k, dtype) == 0
        torch.cuda.synchronize()
        assert torch.equal(q2k, ref)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    d = msa_synth.decode_inputs([3000], paged=True, seed=1, device="cuda")
    q2k = torch.empty((4, 1, 16), dtype=torch.int32, device="cuda")
    cfg = msa.make_config()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # 1 request x 300000 blocks needs 4.8 MB of scores: more than the 4 MiB array
    st = _fn()(ctypes.byref(cfg), _ptr(d.index_q), _ptr(d.index_k_cache), _ptr(d.seq_lens), _ptr(d.page_table),
               None, 1, 300000, d.index_k_cache.shape[0], _ptr(q2k), stream)
    assert st == 4  # MSA_ERR_WORKSPACE
