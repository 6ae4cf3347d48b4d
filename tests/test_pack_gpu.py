"""Packed layout, pack and unpack on the GPU against the CPU oracle."""
import numpy as np
import pytest
import torch

import block_sparse_attention_08_gb300 as msa
import msa_synth
import oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("ids", [
    [[1, 1, 2, 2, 2, 0, 0], [5, 0, 0, 7, 7, 7, 7]],
    [[4, 4, 4], [4, 4, 0]],
    [[0, 3, 3, 0, 9, 9, 0, 2]],
])
def test_pack_metadata_small(ids):
    ids = np.asarray(ids, np.int64)
    cu, rows, mx = msa.msa_pack_metadata(torch.from_numpy(ids).cuda())
    rcu, rrows, rmx = oracle.pack_metadata(ids)
    assert cu.cpu().tolist() == rcu.tolist()
    assert rows.cpu().tolist() == rrows.tolist()
    assert mx == rmx


def test_pack_metadata_workload_map():
    ids = msa_synth.packed_doc_map(2, 32768, seed=0)
    cu, rows, mx = msa.msa_pack_metadata(torch.from_numpy(ids).cuda())
    rcu, rrows, rmx = oracle.pack_metadata(ids)
    np.testing.assert_array_equal(cu.cpu().numpy(), rcu)
    np.testing.assert_array_equal(rows.cpu().numpy(), rrows)
    assert mx == rmx


@pytest.mark.parametrize("ids", [
    [[1, 1, -2, 3]],
    [[1, 2, 1]],
    [[3, 3, 0, 3], [1, 1, 1, 1]],
    [[0, 0, 0]],
    [[1, 2, 3], [5, 6, 5]],
])
def test_pack_metadata_rejects_like_oracle(ids):
    ids = np.asarray(ids, np.int64)
    with pytest.raises(ValueError) as ref:
        oracle.pack_metadata(ids)
    with pytest.raises(msa.MsaError) as got:
        msa.msa_pack_metadata(torch.from_numpy(ids).cuda())
    assert got.value.status == 7
    assert got.value.bad_index == ref.value.bad_row


def test_pack_unpack_roundtrip():
    ids = msa_synth.packed_doc_map(2, 4096, max_len=1024, max_pad=300, seed=3)
    cu, rows, mx = msa.msa_pack_metadata(torch.from_numpy(ids).cuda())
    x = torch.randn(2, 4096, 4, 128, device="cuda").to(torch.bfloat16)
    packed = msa.msa_pack(x, rows)
    ref = oracle.pack(x.float().cpu().numpy(), rows.cpu().numpy())
    np.testing.assert_array_equal(packed.float().cpu().numpy(), ref)
    back = msa.msa_unpack(packed, rows, 2, 4096)
    ref_back = oracle.unpack(ref, rows.cpu().numpy(), 2, 4096)
    np.testing.assert_array_equal(back.float().cpu().numpy(), ref_back)
