"""Pins for the oracle's storage-format decoders and encoders (CPU only).

Values are fixed by the definitions of BF16 (binary32 truncated to 7 stored
mantissa bits) and of FP8-e4m3 ("FP8 Formats for Deep Learning", reference 6 of
"Kernel Fusion for Large-Scale LLM Inference": bias 7, no infinities, S.1111.111
is NaN, largest finite 448)."""
import numpy as np
import pytest
import torch

from oracle.numerics import E4M3_VALUES, bf16_decode, e4m3_decode, round_bf16, round_e4m3


def test_bf16_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x7F7F, 0x0001, 0x3F81], np.uint16)
    want = [1.0, -2.0, 0.0, -0.0, (2 - 2 ** -7) * 2.0 ** 127, 2.0 ** -133, 1 + 2 ** -7]
    got = bf16_decode(bits)
    assert list(got) == want
    assert np.signbit(got[3])


def test_e4m3_known_codes():
    assert e4m3_decode(np.array([0x38]))[0] == 1.0          # exp field 7 = bias
    assert e4m3_decode(np.array([0x7E]))[0] == 448.0        # 1.75 * 2^8
    assert e4m3_decode(np.array([0x01]))[0] == 2.0 ** -9    # smallest subnormal
    assert e4m3_decode(np.array([0x07]))[0] == 7 * 2.0 ** -9
    assert e4m3_decode(np.array([0x08]))[0] == 2.0 ** -6    # smallest normal
    assert e4m3_decode(np.array([0xC0]))[0] == -2.0
    assert np.isnan(e4m3_decode(np.array([0x7F, 0xFF]))).all()
    assert np.isfinite(E4M3_VALUES[[c for c in range(256) if c & 0x7F != 0x7F]]).all()
    # 126 distinct positive finite values plus zero, strictly increasing in the code
    pos = E4M3_VALUES[:0x7F]
    assert np.all(np.diff(pos) > 0)


def test_roundtrip_every_code():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    assert np.array_equal(round_e4m3(e4m3_decode(codes)), codes)
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = np.isfinite(bf16_decode(b))
    assert np.array_equal(round_bf16(bf16_decode(b[finite])), b[finite])


def test_ties_to_even_and_saturation():
    pos = E4M3_VALUES[:0x7F]
    mids = (pos[:-1] + pos[1:]) / 2
    lo = np.arange(0x7E)
    got = round_e4m3(mids)
    want = np.where(lo % 2 == 0, lo, lo + 1)            # even code = even mantissa
    assert np.array_equal(got, want)
    above = np.nextafter(mids, np.inf)
    assert np.array_equal(round_e4m3(above), lo + 1)
    assert list(round_e4m3(np.array([448.0, 464.0, 1e6, -1e6]))) == [0x7E, 0x7E, 0x7E, 0xFE]
    # bf16: 1 + 2^-8 is the midpoint of 1 and 1 + 2^-7 -> even (1.0); 1 + 3*2^-8 -> 1 + 2^-6
    assert list(round_bf16(np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -30]))) == \
        [0x3F80, 0x3F82, 0x3F81]


def test_matches_library_conversions_on_float32_inputs():
    """Where the input is already float32 the single rounding from float64 and
    torch's float32 -> bf16 / e4m3 casts are the same operation."""
    g = torch.Generator().manual_seed(5)
    x = torch.randn(200000, generator=g) * torch.exp(torch.randn(200000, generator=g) * 3)
    b = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(round_bf16(x.double().numpy()), b)
    y = x.clamp(-448, 448)
    e = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(round_e4m3(y.double().numpy()), e)


def test_nonfinite_rejected():
    with pytest.raises(ValueError):
        round_bf16(np.array([np.nan]))
    with pytest.raises(ValueError):
        round_e4m3(np.array([np.inf]))
