"""Pins for the oracle's sampler (CPU only).

* Philox4x32-10 reproduces its published known-answer vectors
  (tests/golden/philox4x32_10_kat.json).
* The uniforms lie strictly inside (0, 1) on the 2^-23 grid (exact in
  float32) and look uniform
  (mean, variance and a 16-bin chi-square over 2^16 draws, fixed seeds).
* Gumbel-max draws follow softmax(z / T): empirical frequencies over many
  steps against the closed-form probabilities (chi-square, fixed seeds).
* Special cases: top_k = 1, or a vanishing temperature, gives the arg-max;
  a tiny top_p keeps only the most probable token; draws never leave the
  top-k set; the top-p set is minimal (its sum reaches p, dropping its least
  probable member does not).
"""
import json
import os

import numpy as np
import pytest

from oracle.sampling import gumbel, keep_set, philox4x32_10, sample, uniforms

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.json")


def test_philox_known_answers():
    for v in json.load(open(GOLDEN))["vectors"]:
        ctr = [np.uint64(int(x, 16)) for x in v["counter"]]
        key = [np.uint64(int(x, 16)) for x in v["key"]]
        got = [int(x) for x in philox4x32_10(ctr, key)]
        assert got == [int(x, 16) for x in v["output"]]


def test_uniforms_grid_and_moments():
    u = uniforms(12345, 3, 7, np.arange(1 << 16))
    assert np.all(u > 0) and np.all(u < 1)
    assert np.all((u * 2 ** 23 - 0.5) == np.round(u * 2 ** 23 - 0.5))
    assert np.array_equal(u.astype(np.float32).astype(np.float64), u)      # exact in float32
    assert abs(u.mean() - 0.5) < 0.005 and abs(u.var() - 1 / 12) < 0.002
    counts = np.bincount((u * 16).astype(int), minlength=16)
    exp = len(u) / 16
    chi2 = ((counts - exp) ** 2 / exp).sum()
    assert chi2 < 37.7                      # 99.9 % point of chi-square with 15 dof
    # different rows / steps / seeds give different streams
    assert not np.array_equal(u, uniforms(12345, 4, 7, np.arange(1 << 16)))
    assert not np.array_equal(u, uniforms(12346, 3, 7, np.arange(1 << 16)))


@pytest.mark.parametrize("T", [1.0, 0.5])
def test_gumbel_max_follows_softmax(T):
    logits = np.array([1.0, 0.2, -0.5, 2.0, 0.0, -1.5, 0.7, 1.1])
    n = 20000
    counts = np.bincount([sample(logits, T, 0, 1.0, 99, 0, s) for s in range(n)], minlength=8)
    p = np.exp(logits / T - (logits / T).max())
    p /= p.sum()
    exp = n * p
    chi2 = ((counts - exp) ** 2 / exp).sum()
    assert chi2 < 24.3                      # 99.9 % point with 7 dof


def test_gumbel_of_uniform():
    u = np.array([np.exp(-1.0), 0.5, np.exp(-np.exp(-2.0))])
    np.testing.assert_allclose(gumbel(u), [0.0, -np.log(np.log(2.0)), 2.0], rtol=1e-12)


def test_special_cases():
    rng = np.random.default_rng(0)
    logits = rng.normal(size=500) * 2
    top = int(np.argmax(logits))
    for s in range(50):
        assert sample(logits, 1.0, 1, 1.0, 7, 2, s) == top
        assert sample(logits, 1e-6, 0, 1.0, 7, 2, s) == top
        assert sample(logits, 1.0, 0, 1e-9, 7, 2, s) == top
        k = 20
        allowed = set(np.argsort(-logits)[:k].tolist())
        assert sample(logits, 0.8, k, 1.0, 7, 2, s) in allowed


@pytest.mark.parametrize("p", [0.1, 0.5, 0.9, 0.99])
def test_top_p_set_is_minimal(p):
    rng = np.random.default_rng(1)
    logits = rng.normal(size=300)
    for T, k in ((1.0, 0), (0.7, 64)):
        kept = keep_set(logits, T, k, p)
        z = logits / T
        cand = np.argsort(-z, kind="stable")[: k] if k else np.argsort(-z, kind="stable")
        pr = np.exp(z[cand] - z[cand].max())
        pr /= pr.sum()
        probs = dict(zip(cand.tolist(), pr.tolist()))
        total = sum(probs[i] for i in kept)
        assert total >= p - 1e-12
        assert total - min(probs[i] for i in kept) < p
        # the kept tokens are the most probable ones
        rest = set(cand.tolist()) - set(kept.tolist())
        if rest:
            assert min(probs[i] for i in kept) >= max(probs[i] for i in rest)
