"""Pins for the oracle's index producer (no GPU): L2 norm, storage cast and
insertion into the paged index-K cache.

The pins are values worked by hand from the definition (the bit patterns of
0.6 and 0.8 in bf16 and E4M3), closed forms (one non-zero element gives +-1,
four equal ones 0.5, 128 ones 1/sqrt(128)), invariants (power-of-two scaling,
unit norm within the storage rounding, the sign of every element) and slot
geometry worked by hand from page tables.
"""
import numpy as np
import pytest
import torch

import oracle


def _vec(values, n=128):
    x = np.zeros(n, np.float32)
    x[: len(values)] = values
    return torch.from_numpy(x).to(torch.bfloat16)


def test_three_four_five_bf16():
    # s = 25, r = 5, y = (0.6, 0.8): 0.6 = 1.0011001|1001... x 2^-1 rounds up to
    # 1.0011010 x 2^-1 = 0.6015625 (bits 0x3F1A); 0.8 = 1.1001100|1100... x 2^-1
    # rounds up to 1.1001101 x 2^-1 = 0.80078125 (bits 0x3F4D)
    y = oracle.index_normalize(_vec([3.0, 4.0]))
    assert y[0] == 0x3F1A and y[1] == 0x3F4D and not y[2:].any()


def test_three_four_five_e4m3():
    # E4M3 of 0.6: quantum 2^-4 at exponent -1, 0.6 / 2^-4 = 9.6 -> 10 -> 0.625,
    # byte 0 0110 010 = 0x32; 0.8: 12.8 -> 13 -> 0.8125, byte 0 0110 101 = 0x35
    y = oracle.index_normalize(_vec([3.0, 4.0]), "e4m3")
    assert y[0] == 0x32 and y[1] == 0x35 and not y[2:].any()


@pytest.mark.parametrize("v", [1.0, -3.0, 0.0078125, 96.0, -2.0 ** -60])
def test_single_nonzero_element_is_plus_minus_one(v):
    x = np.zeros(128, np.float32)
    x[37] = v
    xb = torch.from_numpy(x).to(torch.bfloat16)
    y = oracle.index_normalize(xb)
    want = 0x3F80 if v > 0 else 0xBF80      # +-1.0 in bf16
    assert y[37] == want and not np.delete(y, 37).any()
    y8 = oracle.index_normalize(xb, "e4m3")
    assert y8[37] == (0x38 if v > 0 else 0xB8) and not np.delete(y8, 37).any()


def test_four_equal_elements_give_one_half():
    y = oracle.index_normalize(_vec([-5.0, -5.0, -5.0, -5.0]))
    assert (y[:4] == 0xBF00).all() and not y[4:].any()       # -0.5
    y8 = oracle.index_normalize(_vec([7.0, 7.0, 7.0, 7.0]), "e4m3")
    assert (y8[:4] == 0x30).all() and not y8[4:].any()       # 0.5: 0 0110 000


def test_all_ones():
    # y = 1 / sqrt(128) = 0.0883883... = 1.0110101|0000 0100... x 2^-4: rounds down to
    # 1.0110101 x 2^-4 (exponent field 123), bits 0 01111011 0110101 = 0x3DB5
    y = oracle.index_normalize(torch.ones(128, dtype=torch.bfloat16))
    assert (y == 0x3DB5).all()


def test_zero_and_underflowing_vectors_are_stored_as_zeros():
    assert not oracle.index_normalize(torch.zeros(128, dtype=torch.bfloat16)).any()
    # every square is below binary32's range (2^-200), so s = 0
    tiny = torch.full((128,), 2.0 ** -100, dtype=torch.bfloat16)
    assert not oracle.index_normalize(tiny).any()
    assert not oracle.index_normalize(tiny, "e4m3").any()


def test_power_of_two_scaling_and_signs():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(64, 128, generator=g).to(torch.bfloat16)
    y = oracle.index_normalize(x)
    for k in (-8, 3, 20):
        np.testing.assert_array_equal(oracle.index_normalize((x.float() * 2.0 ** k).to(torch.bfloat16)), y)
    yf = torch.from_numpy(y.view(np.int16)).view(torch.bfloat16).float().numpy()
    xf = x.float().numpy()
    assert (np.sign(yf) == np.sign(xf)).all()
    # unit norm within the bf16 rounding of each element (relative 2^-9)
    n2 = (yf.astype(np.float64) ** 2).sum(axis=1)
    assert np.abs(n2 - 1).max() < 2 * 2.0 ** -9 + 1e-6


def test_decode_insertion_slots():
    # request 0: length 130, its new key at position 129 -> page_table[0][1] = 1 -> slot 128 + 1;
    # request 1: length 1, position 0 -> page_table[1][0] = 2 -> slot 256
    pt = np.array([[3, 1], [2, 0]], np.int32)
    np.testing.assert_array_equal(oracle.index_slots_decode(np.array([130, 1], np.int32), page_table=pt),
                                  [129, 256])
    # contiguous: cu_seqlens_k = [0, 130, 131] -> rows 129 and 130
    np.testing.assert_array_equal(
        oracle.index_slots_decode(np.array([130, 1], np.int32), cu_seqlens_k=np.array([0, 130, 131], np.int64)),
        [129, 130])


def test_decode_produce_writes_only_the_new_rows():
    g = torch.Generator().manual_seed(1)
    iq = torch.randn(2, 4, 128, generator=g).to(torch.bfloat16)
    ik = torch.randn(2, 1, 128, generator=g).to(torch.bfloat16)
    cache = torch.randn(512, 1, 128, generator=g).to(torch.bfloat16)
    pt = np.array([[3, 1], [2, 0]], np.int32)
    q_out, new = oracle.index_produce_decode(iq, ik, cache, np.array([130, 1], np.int32), page_table=pt)
    before = cache.view(torch.int16).numpy().view(np.uint16)
    changed = np.nonzero((new != before).any(axis=(1, 2)))[0]
    assert set(changed.tolist()) <= {129, 256}
    np.testing.assert_array_equal(new[[129, 256]], oracle.index_normalize(ik))
    np.testing.assert_array_equal(q_out, oracle.index_normalize(iq))


def test_prefill_insertion_slots():
    # documents of 3 and 130 tokens; document 0 on page 2 (slots 256..258), document 1 on
    # pages 0 and 1 (positions 0..127 -> slots 0..127, positions 128, 129 -> slots 128, 129)
    cu = np.array([0, 3, 133], np.int32)
    pt = np.array([[2, -1], [0, 1]], np.int32)
    want = [256, 257, 258] + list(range(130))
    np.testing.assert_array_equal(oracle.index_slots_prefill(cu, pt), want)


def test_negative_zero_elements_keep_their_sign():
    # y = -0.0 / 5 = -0.0: bf16 0x8000, E4M3 0x80 (signed zeros of both formats)
    x = _vec([3.0, 4.0, -0.0])
    assert oracle.index_normalize(x)[2] == 0x8000 and oracle.index_normalize(x)[3] == 0
    assert oracle.index_normalize(x, "e4m3")[2] == 0x80 and oracle.index_normalize(x, "e4m3")[3] == 0
