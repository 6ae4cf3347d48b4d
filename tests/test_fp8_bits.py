"""The decode attention reads an FP8 (E4M3) K/V cache without a conversion
instruction: it moves each byte's exponent and mantissa bits (eeee mmm) into
bits 14..7 of an fp16 and keeps the sign in bit 15, which gives the E4M3 value
times 2^-8 exactly, and folds 2^8 into its scales.  This checks that claim for
every finite E4M3 byte against PyTorch's own E4M3 decoding (OCP E4M3, "fn")."""
import numpy as np
import torch


def _f16_times_256(byte):
    h = np.uint32(byte) << np.uint32(8)
    bits = ((h >> np.uint32(1)) & np.uint32(0x3F80)) | (h & np.uint32(0x8000))
    return float(np.array([bits], dtype=np.uint16).view(np.float16)[0]) * 256.0


def test_every_finite_e4m3_byte():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    checked = 0
    for b in range(256):
        if np.isnan(ref[b]):  # 0x7f and 0xff: the NaN encodings, never in a cache of finite values
            continue
        got = _f16_times_256(b)
        assert got == ref[b] and np.signbit(got) == np.signbit(ref[b]), (hex(b), got, ref[b])
        checked += 1
    assert checked == 254
