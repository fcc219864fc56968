"""The four-term e4m3 split of activation rows that the e4m3 tensor-core path
multiplies (x = s (c0 + c1/16 + c2/256 + c3/4096), s a power of two with
max|x| / s < 448, each code the round-to-nearest-even e4m3 of the scaled
residual), restated step by step in float32 with the oracle's e4m3 codec, and
held to the bound the design relies on: every residual is exact in fp32, and
|x - rebuilt| <= 2^-16 |x| + 2^-29 max|x| over rows with a wide dynamic range.
The GPU side of the same split is pinned through the C ABI by
test_gpu_tc.test_tc8_term_split_identity."""
import numpy as np
import pytest

from oracle.numerics import e4m3_decode, round_e4m3


def _split(x: np.ndarray):
    m = float(np.max(np.abs(x)))
    if m == 0.0:
        return 1.0, np.zeros((4,) + x.shape, np.uint8), []
    _, e = np.frexp(np.float32(m) * np.float32(1.0 / 448.0))
    s = np.ldexp(1.0, int(e))
    r = (x.astype(np.float32) * np.float32(1.0 / s)).astype(np.float32)      # exact: power of two
    codes, exact = [], []
    for _ in range(4):
        c = round_e4m3(r.astype(np.float64))
        d = e4m3_decode(c)
        nxt = (r - d.astype(np.float32)).astype(np.float32)                  # fp32, as on the GPU
        exact.append(np.array_equal(nxt.astype(np.float64), r.astype(np.float64) - d))
        codes.append(c)
        r = (nxt * np.float32(16.0)).astype(np.float32)
    return s, np.stack(codes), exact


def _rebuild(s, codes):
    return s * sum(e4m3_decode(codes[j]) * 16.0 ** -j for j in range(4))


@pytest.mark.parametrize("seed", range(6))
def test_term_split_error_bound(seed):
    rng = np.random.default_rng(seed)
    mag = 10.0 ** rng.uniform(-10, 3, size=4096)
    x = np.where(rng.random(4096) < 0.5, -mag, mag).astype(np.float32)
    x[rng.random(4096) < 0.02] = 0.0
    s, codes, exact = _split(x)
    assert all(exact)                                       # every residual is exact in fp32
    assert np.max(np.abs(x)) / s < 448.0 and np.max(np.abs(x)) / s >= 224.0
    xd = x.astype(np.float64)
    err = np.abs(_rebuild(s, codes) - xd)
    assert np.all(err <= 2.0 ** -16 * np.abs(xd) + 2.0 ** -29 * np.max(np.abs(xd)))
    # the bound is about tight for values near the row's largest: an FP16 rounding
    # (2^-12) is far coarser, all of fp32 (2^-24) finer
    big = np.abs(xd) > 1e-3 * np.max(np.abs(xd))
    rel = err[big] / np.abs(xd[big])
    assert 2.0 ** -24 < rel.max() <= 2.0 ** -16


def test_term_split_gaussian_rows_and_zero_row():
    rng = np.random.default_rng(11)
    x = rng.normal(size=8192).astype(np.float32) * np.float32(3.7)
    s, codes, exact = _split(x)
    assert all(exact)
    err = np.abs(_rebuild(s, codes) - x.astype(np.float64))
    assert np.all(err <= 2.0 ** -16 * np.abs(x) + 2.0 ** -29 * np.max(np.abs(x)))
    s0, c0, _ = _split(np.zeros(64, np.float32))
    assert s0 == 1.0 and not c0.any()
