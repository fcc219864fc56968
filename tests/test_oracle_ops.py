"""Pins for the oracle's elementwise definitions and paged attention (CPU only).

RMSNorm: unit RMS at gamma = 1 and scale invariance ("Root Mean Square Layer
Normalization"). RoPE: rotation of each pair, per-pair angle, norm preservation,
relative-position invariance ("RoFormer"). SiLU closed forms ("GLU Variants
Improve Transformer"). Paged attention against brute-force softmax over a
contiguous cache ("GPU Inference Internals", "Kernels: FlashAttention and the
Memory Hierarchy": the tiled/paged form must equal the naive N x N form)."""
import math

import numpy as np
import pytest

from oracle.decode import OracleKV, paged_attention, rmsnorm, rope, silu, swiglu
from tests import bruteforce as bf


def test_rmsnorm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(0)
    x = rng.normal(size=(7, 333)) * 5
    y = rmsnorm(x, np.ones(333), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(rmsnorm(3.7 * x, np.ones(333), 0.0), y, rtol=0, atol=1e-12)
    g = rng.normal(size=333)
    np.testing.assert_allclose(rmsnorm(x, g, 0.0), y * g, rtol=0, atol=1e-12)
    # eps sits inside the root: RMS of the output is sqrt(ms / (ms + eps))
    ms = np.mean(x * x, axis=1)
    y2 = rmsnorm(x, np.ones(333), 0.5)
    np.testing.assert_allclose(np.sqrt(np.mean(y2 * y2, axis=1)), np.sqrt(ms / (ms + 0.5)), atol=1e-12)


def test_rope_pairs_and_angles():
    # d = 2: one pair rotated by p * theta^0 = p radians, counter-clockwise
    for p in (0, 1, 5, 77):
        np.testing.assert_allclose(rope(np.array([1.0, 0.0]), p, 1e4), [math.cos(p), math.sin(p)], atol=1e-12)
        np.testing.assert_allclose(rope(np.array([0.0, 1.0]), p, 1e4), [-math.sin(p), math.cos(p)], atol=1e-12)
    # pair i is (i, i + d/2) and turns by p * theta^(-2i/d)
    d, theta, p = 16, 10000.0, 3
    for i in range(d // 2):
        e = np.zeros(d)
        e[i] = 1.0
        out = rope(e, p, theta)
        assert np.count_nonzero(np.abs(out) > 1e-15) <= 2
        ang = math.atan2(out[i + d // 2], out[i])
        want = math.remainder(p * theta ** (-2 * i / d), 2 * math.pi)
        assert abs(ang - want) < 1e-12


def test_rope_norm_identity_relative():
    rng = np.random.default_rng(1)
    d = 128
    q, k = rng.normal(size=d), rng.normal(size=d)
    assert np.array_equal(rope(q, 0, 1e4), q)
    for p in (1, 17, 4095):
        assert abs(np.linalg.norm(rope(q, p, 1e4)) - np.linalg.norm(q)) < 1e-12
    for m, n, t in ((5, 3, 100), (0, 9, 1), (2047, 12, 33)):
        a = rope(q, m, 1e4) @ rope(k, n, 1e4)
        b = rope(q, m + t, 1e4) @ rope(k, n + t, 1e4)
        assert abs(a - b) < 1e-9


def test_silu_closed_forms():
    assert silu(np.array(0.0)) == 0.0
    assert abs(silu(np.array(1.0)) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    assert abs(silu(np.array(40.0)) - 40.0) < 1e-12
    assert abs(silu(np.array(-40.0))) < 1e-15
    assert abs(swiglu(np.array(2.0), np.array(-3.0)) - (-3.0 * 2.0 / (1 + math.exp(-2.0)))) < 1e-14


def _attn_case(nq, nkv, S, bs=16, d=8, fp8=False, seed=0, scale=1.0):
    rng = np.random.default_rng(seed)
    nblk = -(-S // bs)
    num_blocks = nblk + 4
    if fp8:
        vals = rng.normal(size=(1, 2, num_blocks + 1, nkv, bs, d))
        raw = np.array([[bf.to_e4m3_code(v) for v in row] for row in vals.reshape(-1, d)],
                       np.uint8).reshape(vals.shape)
    else:
        raw = rng.integers(0x3C00, 0x4000, size=(1, 2, num_blocks + 1, nkv, bs, d)).astype(np.uint16)
        raw |= (rng.integers(0, 2, size=raw.shape).astype(np.uint16) << 15)
    kv = OracleKV(raw, np.array([scale]), np.array([scale * 0.5]))
    table = rng.permutation(num_blocks)[:nblk]
    q = rng.normal(size=(nq, d))
    return kv, table, q


def _brute(kv, table, q, S, nkv):
    nq, d = q.shape
    bs = kv.block_size
    dec = bf.e4m3 if kv.fp8 else bf.bf16
    out = []
    for h in range(nq):
        g = h // (nq // nkv)
        K, V = [], []
        for t in range(S):
            blk, slot = int(table[t // bs]), t % bs
            K.append([dec(kv.raw[0, 0, blk, g, slot, i]) * kv.k_scale[0] for i in range(d)])
            V.append([dec(kv.raw[0, 1, blk, g, slot, i]) * kv.v_scale[0] for i in range(d)])
        s = [sum(q[h][i] * K[t][i] for i in range(d)) / math.sqrt(d) for t in range(S)]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        z = sum(e)
        out.append([sum(e[t] / z * V[t][i] for t in range(S)) for i in range(d)])
    return np.array(out)


@pytest.mark.parametrize("S", [1, 15, 16, 17, 33])
@pytest.mark.parametrize("nq,nkv", [(2, 2), (4, 2), (10, 2), (8, 1)])
def test_paged_attention_matches_bruteforce(S, nq, nkv):
    kv, table, q = _attn_case(nq, nkv, S, seed=S * 31 + nq)
    got = paged_attention(q, kv, 0, table, S)
    np.testing.assert_allclose(got, _brute(kv, table, q, S, nkv), rtol=0, atol=1e-12)


def test_paged_attention_fp8_scaled():
    kv, table, q = _attn_case(4, 2, 21, fp8=True, seed=3, scale=0.75)
    np.testing.assert_allclose(paged_attention(q, kv, 0, table, 21), _brute(kv, table, q, 21, 2),
                               rtol=0, atol=1e-12)


def test_paged_attention_special_cases():
    kv, table, q = _attn_case(4, 2, 40, seed=9)
    # S = 1: the only token gets all the weight, o = V_0
    o = paged_attention(q, kv, 0, table, 1)
    v0 = kv.decode(0, 1, np.array([table[0]]))[0, :, 0, :]
    np.testing.assert_allclose(o, np.repeat(v0, 2, axis=0), atol=1e-15)
    # q = 0: uniform weights, o = mean of V over the context
    o = paged_attention(np.zeros_like(q), kv, 0, table, 40)
    vd = kv.decode(0, 1, table[:3])                          # 3 blocks cover 40 tokens
    V = vd.transpose(1, 0, 2, 3).reshape(2, 48, -1)[:, :40]
    np.testing.assert_allclose(o, np.repeat(V.mean(axis=1), 2, axis=0), atol=1e-14)
