"""Pins of the oracle's MXFP8 quantizer (the MXFP8 emission of the attention
output): hand-worked blocks from the OCP MX definition, the element encoding
against PyTorch's float8_e4m3fn cast, and the scale rule on random blocks."""
import numpy as np
import torch

import oracle


def _q(vals):
    x = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).reshape(1, -1)
    q, s = oracle.mxfp8_quantize(x)
    return q[0], s[0]


def test_hand_worked_blocks():
    # all ones: amax 1 -> floor(log2) 0 -> scale 2^-8 (byte 119); 1 / 2^-8 = 256 = 1.0 x 2^8 -> 0x78
    q, s = _q([1.0] * 32)
    assert s.tolist() == [119] and q.tolist() == [0x78] * 32
    # amax 448 = 1.75 x 2^8 -> scale 2^0 (byte 127): 448 -> 0x7E, -2 -> 0xC0 (sign, exponent 8), 0 -> 0
    q, s = _q([448.0, -2.0] + [0.0] * 30)
    assert s.tolist() == [127] and q[:3].tolist() == [0x7E, 0xC0, 0x00]
    # amax 500 -> floor(log2) 8 -> scale 1: 500 saturates to 448; 464 (midway 448 / 480) ties to even:
    # 448; 3 = 1.5 x 2^1 -> exponent field 8, mantissa 4 -> 0x44
    q, s = _q([500.0, 464.0, 3.0] + [0.0] * 29)
    assert s.tolist() == [127] and q[:3].tolist() == [0x7E, 0x7E, 0x44]
    # amax 0.75 -> floor(log2) -1 -> scale 2^-9 (byte 118); 0.75 / 2^-9 = 384 = 1.5 x 2^8 -> 0x7C;
    # 2^-18 / 2^-9 = 2^-9: the smallest subnormal 0x01; 3 x 2^-20 / 2^-9 = 1.5 x 2^-10 = 0.75 of the
    # subnormal quantum 2^-9 -> rounds to one quantum -> 0x01
    q, s = _q([0.75, 2.0 ** -18, 3 * 2.0 ** -20] + [0.0] * 29)
    assert s.tolist() == [118] and q[:3].tolist() == [0x7C, 0x01, 0x01]
    # a zero block: byte 0 and zero elements
    q, s = _q([0.0] * 32)
    assert s.tolist() == [0] and q.tolist() == [0] * 32
    # two blocks are scaled independently
    q, s = _q([1.0] * 32 + [4.0] * 32)
    assert s.tolist() == [119, 121] and set(q.tolist()) == {0x78}


def test_element_encoding_matches_torch_e4m3():
    # in-range elements: with amax at 448 the scale is 1, so each byte is the plain E4M3 rounding
    rng = np.random.default_rng(0)
    for _ in range(20):
        v = np.concatenate([[448.0], rng.uniform(-448, 448, 31) * rng.choice([1, 1e-1, 1e-2, 1e-3], 31)])
        x = torch.tensor(v, dtype=torch.float32).to(torch.bfloat16)
        q, s = oracle.mxfp8_quantize(x.reshape(1, 32))
        assert s[0, 0] == 127
        ref = x.float().to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert (q[0] == ref).all()


def test_scale_rule_and_round_trip():
    rng = np.random.default_rng(1)
    e4m3_vals = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for _ in range(50):
        v = rng.standard_normal(32) * 10.0 ** rng.uniform(-6, 6)
        x = torch.tensor(v, dtype=torch.float32).to(torch.bfloat16)
        q, s = oracle.mxfp8_quantize(x.reshape(1, 32))
        b = x.double().numpy()
        X = 2.0 ** (int(s[0, 0]) - 127)
        y = np.abs(b) / X
        assert 256.0 <= y.max() < 512.0          # floor(log2 amax) - 8
        deq = e4m3_vals[q[0]].astype(np.float64) * X
        sat = np.abs(b) / X > 448.0
        assert np.all(np.abs(deq[sat]) == 448.0 * X)
        # otherwise within half an E4M3 quantum (relative 2^-4, or 2^-10 absolute for subnormals)
        ok = ~sat
        tol = np.maximum(np.abs(b[ok]) * 2.0 ** -4, 2.0 ** -10 * X) + 1e-300
        assert np.all(np.abs(deq[ok] - b[ok]) <= tol)


def test_negative_zero_keeps_its_sign():
    # OCP E4M3 has a signed zero: -0.0 encodes as S=1, E=0, M=0 (0x80), as PyTorch's cast does
    q, s = _q([-0.0] * 32)
    assert s.tolist() == [0] and q.tolist() == [0x80] * 32
    assert torch.tensor([-0.0]).to(torch.float8_e4m3fn).view(torch.uint8).item() == 0x80
