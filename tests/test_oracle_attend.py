"""Pins for the oracle's attention, decode geometry and packing (no GPU)."""
import math

import numpy as np
import pytest
import torch

import oracle
import msa_synth

SCALE = 1.0 / math.sqrt(128.0)


def _bits64(x):
    return x.float().double()


def test_zero_query_gives_mean_of_selected_values():
    p = msa_synth.prefill_inputs([700], seed=7, topk=3)
    q0 = torch.zeros_like(p.q)
    toks = np.arange(0, 700, 13, dtype=np.int64)
    q2k, _ = oracle.select_prefill(p.index_q, p.index_k, p.cu_seqlens, toks, topk=3)
    out = oracle.attend_prefill(q0, p.k, p.v, p.cu_seqlens, toks, q2k, SCALE)
    v = _bits64(p.v).numpy()
    for i, t in enumerate(toks):
        for h in (0, 17, 63):
            g = h // 16
            keys = [j for b in q2k[g, i] if b >= 0 for j in range(b * 128, b * 128 + 128) if j <= t]
            np.testing.assert_allclose(out[i, h], v[keys, g].mean(axis=0), rtol=0, atol=1e-12)


def test_two_key_closed_form():
    # document of 2 tokens: query 1 sees keys 0 and 1
    T = 2
    q = torch.zeros(T, 64, 128)
    k = torch.zeros(T, 4, 128)
    v = torch.zeros(T, 4, 128)
    q[1, :, 0] = 2.0
    k[0, :, 0] = 1.0
    k[1, :, 0] = -0.5
    v[0, :, :] = 3.0
    v[1, :, :] = -1.0
    cu = np.array([0, 2], np.int32)
    q2k = np.full((4, 1, 16), -1, np.int32)
    q2k[:, 0, 0] = 0
    out = oracle.attend_prefill(q.bfloat16(), k.bfloat16(), v.bfloat16(), cu, np.array([1]), q2k, SCALE)
    z1, z2 = 2.0 * SCALE, -1.0 * SCALE
    w1 = math.exp(z1) / (math.exp(z1) + math.exp(z2))
    np.testing.assert_allclose(out[0], 3.0 * w1 - (1 - w1), rtol=0, atol=1e-14)


def test_dense_regime_equals_causal_attention():
    """nb <= topk for every token: the method is dense causal attention (checked
    against torch's scaled_dot_product_attention in fp64, a library routine)."""
    lens = [300, 517, 64]
    p = msa_synth.prefill_inputs(lens, seed=9, topk=16)
    toks = np.arange(sum(lens), dtype=np.int64)
    q2k, _ = oracle.select_prefill(p.index_q, p.index_k, p.cu_seqlens, toks, topk=16)
    out = oracle.attend_prefill(p.q, p.k, p.v, p.cu_seqlens, toks, q2k, SCALE)
    cu = p.cu_seqlens.numpy()
    for d in range(len(lens)):
        a, b = cu[d], cu[d + 1]
        qd = _bits64(p.q[a:b]).permute(1, 0, 2)             # [64, n, 128]
        kd = _bits64(p.k[a:b]).repeat_interleave(16, dim=1).permute(1, 0, 2)
        vd = _bits64(p.v[a:b]).repeat_interleave(16, dim=1).permute(1, 0, 2)
        ref = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, is_causal=True, scale=SCALE)
        np.testing.assert_allclose(out[a:b], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_sparse_equals_dense_with_block_mask():
    """A dense [T, T] formulation with a causal & selected-block mask (matrix
    ops, a different code path from the per-block loop) gives the same output."""
    T = 900
    p = msa_synth.prefill_inputs([T], seed=4, topk=3)
    toks = np.arange(T, dtype=np.int64)
    q2k, _ = oracle.select_prefill(p.index_q, p.index_k, p.cu_seqlens, toks, topk=3)
    sample = np.arange(0, T, 37)
    out = oracle.attend_prefill(p.q, p.k, p.v, p.cu_seqlens, sample, q2k[:, sample], SCALE)
    q = _bits64(p.q).numpy()
    k = _bits64(p.k).numpy()
    v = _bits64(p.v).numpy()
    blk = np.arange(T) // 128
    for g in range(4):
        sel = np.zeros((T, T // 128 + 1), bool)
        for t in range(T):
            for b in q2k[g, t]:
                if b >= 0:
                    sel[t, b] = True
        mask = sel[:, blk] & (np.arange(T)[None, :] <= np.arange(T)[:, None])
        for h in range(16 * g, 16 * g + 16, 5):
            z = SCALE * q[:, h] @ k[:, g].T
            z = np.where(mask, z, -np.inf)
            z = z - z.max(axis=1, keepdims=True)
            w = np.exp(z)
            w /= w.sum(axis=1, keepdims=True)
            ref = w @ v[:, g]
            np.testing.assert_allclose(out[:, h], ref[sample], rtol=0, atol=1e-12)


# ---- decode geometry ---------------------------------------------------------

def test_decode_paged_equals_contiguous():
    lens = [1000, 129, 128, 1, 4100]
    a = msa_synth.decode_inputs(lens, paged=True, seed=1, topk=4)
    b = msa_synth.decode_inputs(lens, paged=False, seed=1, topk=4)
    # same values, laid out differently: rebuild b's caches from a's pages
    pt = a.page_table.numpy()
    rows = np.concatenate([pt[r, np.arange(L) // 128] * 128 + np.arange(L) % 128
                           for r, L in enumerate(lens)])
    kc, vc, ikc = a.k_cache[rows], a.v_cache[rows], a.index_k_cache[rows]
    q2k_a, _ = oracle.select_decode(a.index_q, a.index_k_cache, a.seq_lens, page_table=a.page_table, topk=4)
    q2k_b, _ = oracle.select_decode(a.index_q, ikc, b.seq_lens, cu_seqlens_k=b.cu_seqlens_k, topk=4)
    np.testing.assert_array_equal(q2k_a, q2k_b)
    oa = oracle.attend_decode(a.q, a.k_cache, a.v_cache, a.seq_lens, q2k_a, SCALE, page_table=a.page_table)
    ob = oracle.attend_decode(a.q, kc, vc, b.seq_lens, q2k_a, SCALE, cu_seqlens_k=b.cu_seqlens_k)
    np.testing.assert_array_equal(oa, ob)


def test_decode_equals_prefill_last_token():
    """A decode query at position L-1 over a context of L keys is the prefill
    computation of the last token of an L-token document."""
    L = 777
    p = msa_synth.prefill_inputs([L], seed=8, topk=4)
    toks = np.array([L - 1], np.int64)
    q2k_p, _ = oracle.select_prefill(p.index_q, p.index_k, p.cu_seqlens, toks, topk=4)
    out_p = oracle.attend_prefill(p.q, p.k, p.v, p.cu_seqlens, toks, q2k_p, SCALE)
    cuk = np.array([0, L], np.int64)
    q2k_d, _ = oracle.select_decode(p.index_q[L - 1:], p.index_k, np.array([L], np.int32),
                                    cu_seqlens_k=cuk, topk=4)
    out_d = oracle.attend_decode(p.q[L - 1:], p.k, p.v, np.array([L], np.int32), q2k_d, SCALE,
                                 cu_seqlens_k=cuk)
    np.testing.assert_array_equal(q2k_p, q2k_d)
    np.testing.assert_array_equal(out_p, out_d)


def test_decode_e4m3_scores_are_exact_products():
    """E4M3 operands: a one-hot query against keys holding known E4M3 bytes
    selects the block holding the largest decoded value."""
    lens = [512]
    d = msa_synth.decode_inputs(lens, paged=False, index_dtype="e4m3", seed=0, topk=2)
    iq = torch.zeros(1, 4, 128, dtype=torch.uint8)
    iq[0, :, 3] = 0x38  # 1.0
    ik = torch.zeros(512, 1, 128, dtype=torch.uint8)
    ik[10, 0, 3] = 0x30   # 0.5   block 0
    ik[300, 0, 3] = 0x34  # 0.75  block 2
    ik[130, 0, 3] = 0x2C  # 0.375 block 1
    q2k, gap = oracle.select_decode(iq.view(torch.float8_e4m3fn), ik.view(torch.float8_e4m3fn),
                                    d.seq_lens, cu_seqlens_k=d.cu_seqlens_k, topk=2)
    assert list(q2k[0, 0]) == [2, 3]


# ---- packing -----------------------------------------------------------------

def test_pack_metadata_small_map():
    ids = np.array([[1, 1, 2, 2, 2, 0, 0],
                    [5, 0, 0, 7, 7, 7, 7]], np.int64)
    cu, rows, mx = oracle.pack_metadata(ids)
    assert list(cu) == [0, 2, 5, 6, 10]
    assert list(rows) == [0, 1, 2, 3, 4, 7, 10, 11, 12, 13]
    assert mx == 4
    x = np.arange(14 * 3).reshape(2, 7, 3)
    packed = oracle.pack(x, rows)
    back = oracle.unpack(packed, rows, 2, 7)
    assert (back[ids > 0] == x[ids > 0]).all() and (back[ids == 0] == 0).all()


@pytest.mark.parametrize("ids,code", [
    ([[1, 1, -2]], 1),
    ([[1, 2, 1]], 2),
    ([[3, 3, 0, 3]], 2),
    ([[0, 0, 0]], 3),
    (np.zeros((0, 4), np.int64), 4),
])
def test_pack_metadata_rejects(ids, code):
    with pytest.raises(ValueError) as e:
        oracle.pack_metadata(np.asarray(ids, np.int64).reshape(-1, np.asarray(ids).shape[-1]))
    assert e.value.code == code


def test_same_id_in_two_rows_is_two_documents():
    ids = np.array([[4, 4, 4], [4, 4, 0]], np.int64)
    cu, rows, mx = oracle.pack_metadata(ids)
    assert list(cu) == [0, 3, 5] and mx == 3


def test_packed_doc_map_recipe():
    ids = msa_synth.packed_doc_map(2, 32768, seed=0)
    cu, rows, mx = oracle.pack_metadata(ids)
    lens = np.diff(cu)
    assert lens.min() >= 1 and mx <= 16384
    assert 32768 * 2 - 2048 <= cu[-1] <= 32768 * 2
    assert list(lens) == msa_synth.doc_lengths_from_map(ids)


# ---- decode attention over an FP8 (E4M3) main K/V cache ----------------------

def _fp8_case(seed=4, lens=(300, 1000, 129)):
    d = msa_synth.decode_inputs(list(lens), paged=True, seed=seed)
    k8 = (d.k_cache.float() * 0.5).to(torch.float8_e4m3fn)
    v8 = (d.v_cache.float() * 0.5).to(torch.float8_e4m3fn)
    q2k, _ = oracle.select_decode(d.index_q, d.index_k_cache, d.seq_lens, page_table=d.page_table, topk=4)
    return d, k8, v8, q2k


def test_fp8_cache_equals_bf16_cache_of_the_same_values():
    # every E4M3 value is exact in bf16: the FP8 attention with unit scales is the pinned bf16
    # attention on the decoded values, to the last bit
    d, k8, v8, q2k = _fp8_case()
    a = oracle.attend_decode_fp8(d.q, k8, v8, d.seq_lens, q2k, SCALE, page_table=d.page_table)
    b = oracle.attend_decode(d.q, k8.to(torch.bfloat16), v8.to(torch.bfloat16), d.seq_lens, q2k, SCALE,
                             page_table=d.page_table)
    np.testing.assert_array_equal(a, b)


def test_fp8_scales_are_exact_powers_of_two():
    # scales 2 and 0.25 equal bf16 caches holding 2x and 0.25x the values (exact in bf16)
    d, k8, v8, q2k = _fp8_case(seed=5)
    a = oracle.attend_decode_fp8(d.q, k8, v8, d.seq_lens, q2k, SCALE, k_scale=2.0, v_scale=0.25,
                                 page_table=d.page_table)
    b = oracle.attend_decode(d.q, (k8.float() * 2).to(torch.bfloat16), (v8.float() * 0.25).to(torch.bfloat16),
                             d.seq_lens, q2k, SCALE, page_table=d.page_table)
    np.testing.assert_array_equal(a, b)


def test_fp8_zero_query_gives_the_scaled_mean_of_v():
    # q = 0: equal weights, out = v_scale * the mean of the attended values
    d, k8, v8, q2k = _fp8_case(seed=6, lens=(200,))
    q = torch.zeros_like(d.q)
    out = oracle.attend_decode_fp8(q, k8, v8, d.seq_lens, q2k, SCALE, k_scale=3.0, v_scale=1.5,
                                   page_table=d.page_table)
    v = v8.float().double().numpy()
    pt = d.page_table.numpy()
    L = int(d.seq_lens[0])
    for g in range(4):
        keys = [p for b in q2k[g, 0] if b >= 0 for p in range(128 * b, min(128 * b + 128, L))]
        rows = [pt[0, p // 128] * 128 + p % 128 for p in keys]
        want = 1.5 * v[rows, g, :].mean(axis=0)
        for hh in range(16):
            np.testing.assert_allclose(out[0, 16 * g + hh], want, rtol=1e-12, atol=1e-12)
