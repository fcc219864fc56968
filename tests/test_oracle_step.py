"""Pins for the oracle's whole decode step (CPU only).

* A scalar pure-Python step on tiny models (tests/bruteforce.py) must agree
  with the vectorised step to 1e-12 and write the same cache bytes.
* Closed form: with the O and down projections zeroed every layer is the
  identity on the residual stream, so logits = W_lm . RMSNorm(E[tok]) * g_final.
* Relative position: keys stored at positions j + t and a query at m + t give
  the same attention output as j and m ("RoFormer"), up to the cache rounding.
* Prefill: ingesting a prompt at once gives the logits and cache of feeding
  it one token at a time.
* FLOPs: "A transformer forward pass performs roughly 2 x P FLOPs per token"
  ("GPU Inference Internals", "Roofline: Why Decode Is Memory-Bound").
"""
import numpy as np
import pytest

from oracle.decode import OracleKV, decode_step, paged_attention, prefill, rmsnorm, rope
from oracle.numerics import bf16_decode, round_bf16
from synth import ONE_B, tensor_shape, SynthModel
from tests import bruteforce as bf
from tests.helpers import MICRO, MICRO_FP8, kv_numpy, make_case, oracle_weights


@pytest.mark.parametrize("cfg", [MICRO, MICRO_FP8], ids=lambda c: c.name)
def test_step_matches_scalar_bruteforce(cfg):
    model = SynthModel(cfg, seed=11)
    W = oracle_weights(model)
    case = make_case(cfg, 3, 4, 40, seed=21)
    raw = kv_numpy(case["pool"])
    ks = np.array([0.875, 1.25]) if cfg.kv_dtype == "fp8" else np.ones(2)
    vs = np.array([1.5, 0.625]) if cfg.kv_dtype == "fp8" else np.ones(2)
    toks = np.array([5, 127, 64], np.int32)
    pos = case["ctx"]
    sl = pos + 1
    kv = OracleKV(raw.copy(), ks, vs)
    res = decode_step(W, cfg, kv, toks, pos, case["tables"], sl)
    logits_bf, kvl = bf.step(W, cfg, raw.copy(), ks, vs, toks, pos, case["tables"], sl)
    np.testing.assert_allclose(res.logits, np.array(logits_bf), rtol=1e-12, atol=1e-14)
    assert np.array_equal(kv.raw, np.array(kvl, dtype=raw.dtype))
    assert np.array_equal(res.next_ids, np.argmax(np.array(logits_bf), axis=1))


def test_zeroed_projections_closed_form():
    cfg = MICRO
    base = oracle_weights(SynthModel(cfg, seed=12))

    def W(name, layer):
        t = base(name, layer)
        if name in ("w_o", "w_down"):
            return {"w": np.zeros_like(t["w"])}
        return t
    case = make_case(cfg, 2, 3, 20, seed=5)
    kv = OracleKV(kv_numpy(case["pool"]), np.ones(2), np.ones(2))
    toks = np.array([3, 99], np.int32)
    res = decode_step(W, cfg, kv, toks, case["ctx"], case["tables"], case["ctx"] + 1)
    e = bf16_decode(base("embed", -1)["w"][toks])
    y = rmsnorm(e, bf16_decode(base("g_final", -1)["w"]), cfg.eps)
    want = y @ bf16_decode(base("lm_head", -1)["w"]).T
    np.testing.assert_allclose(res.logits, want, rtol=1e-12, atol=1e-15)


def test_relative_position_through_the_cache():
    rng = np.random.default_rng(3)
    nq, nkv, d, S, bs = 4, 2, 64, 37, 16
    q = rng.normal(size=(nq, d))
    keys = rng.normal(size=(S, nkv, d))
    vals = rng.normal(size=(S, nkv, d))
    nblk = -(-S // bs)

    def attend(t):
        raw = np.zeros((1, 2, nblk + 1, nkv, bs, d), np.uint16)
        kv = OracleKV(raw, np.ones(1), np.ones(1))
        table = np.arange(nblk)
        for j in range(S):
            kv.store(0, 0, j // bs, j % bs, rope(keys[j], j + t, 1e4))
            kv.store(0, 1, j // bs, j % bs, vals[j])
        return paged_attention(rope(q, S - 1 + t, 1e4), kv, 0, table, S)
    a = attend(0)
    for t in (1, 250, 3000):
        # the only difference is how the rotated keys round to BF16 (2^-9 relative)
        np.testing.assert_allclose(attend(t), a, atol=2e-2)
    # a wrong relative convention (query rotated the other way) is far outside that
    raw = np.zeros((1, 2, nblk + 1, nkv, bs, d), np.uint16)
    kv = OracleKV(raw, np.ones(1), np.ones(1))
    for j in range(S):
        kv.store(0, 0, j // bs, j % bs, rope(keys[j], j, 1e4))
        kv.store(0, 1, j // bs, j % bs, vals[j])
    bad = paged_attention(rope(q, -(S - 1), 1e4), kv, 0, np.arange(nblk), S)
    assert np.max(np.abs(bad - a)) > 0.1


def test_flops_about_twice_params():
    """Run the oracle on the 1B-class shape (zero weights: the count depends on
    shapes only) and compare its multiply-add count with the parameter count."""
    cfg = ONE_B

    def W(name, layer):
        shape = tensor_shape(cfg, name)
        return {"w": np.zeros(shape, np.uint16)}
    S = 16
    raw = np.zeros((cfg.n_layers, 2, 2, cfg.n_kv_heads, cfg.block_size, cfg.head_dim), np.uint16)
    kv = OracleKV(raw, np.ones(cfg.n_layers), np.ones(cfg.n_layers))
    res = decode_step(W, cfg, kv, [1], [S - 1], np.array([[0]], np.int32), [S])
    mats = ("w_qkv", "w_o", "w_gu", "w_down")
    p_matmul = cfg.n_layers * sum(np.prod(tensor_shape(cfg, m)) for m in mats) + \
        np.prod(tensor_shape(cfg, "lm_head"))
    p_total = p_matmul + np.prod(tensor_shape(cfg, "embed")) + (2 * cfg.n_layers + 1) * cfg.hidden
    attn = 4 * cfg.n_q_heads * cfg.head_dim * S * cfg.n_layers
    assert abs(res.flops - (2 * p_matmul + attn)) <= 0.01 * res.flops
    assert abs(res.flops / (2 * p_total) - 1) <= 0.10
    assert res.attn_flops == attn


@pytest.mark.parametrize("cfg", [MICRO, MICRO_FP8], ids=lambda c: c.name)
@pytest.mark.parametrize("start,n", [(0, 1), (0, 19), (23, 9)])
def test_prefill_equals_token_by_token(cfg, start, n):
    """Prefill of n tokens from `start` = n decode steps of one token each
    (positions start, start + 1, ...): same last-token logits, same cache."""
    model = SynthModel(cfg, seed=31)
    W = oracle_weights(model)
    nblk = -(-(start + n) // 16) + 1
    table = np.random.default_rng(4).permutation(nblk + 2)[:nblk].astype(np.int32)
    from synth import random_kv_pool
    raw = kv_numpy(random_kv_pool(cfg, nblk + 2, seed=8))
    ks = np.array([0.75, 1.5]) if cfg.kv_dtype == "fp8" else np.ones(2)
    toks = np.random.default_rng(5).integers(0, cfg.vocab, size=n).astype(np.int32)
    a = OracleKV(raw.copy(), ks, ks[::-1].copy())
    res = prefill(W, cfg, a, toks, start, table)
    b = OracleKV(raw.copy(), ks, ks[::-1].copy())
    for i in range(n):
        r1 = decode_step(W, cfg, b, toks[i:i + 1], [start + i], table[None, :], [start + i + 1])
    np.testing.assert_allclose(res.logits[-1], r1.logits[0], rtol=1e-9, atol=1e-12)
    # the two runs round the same values to the cache format; their fp64
    # inputs differ only in summation order, so codes agree except (rarely)
    # at a rounding boundary, where they are neighbours
    dec = (lambda r: bf16_decode(r)) if cfg.kv_dtype == "bf16" else None
    if dec is None:
        from oracle.numerics import e4m3_decode as dec
    diff = a.raw != b.raw
    assert diff.sum() <= 2
    if diff.any():
        ga, gb = dec(a.raw[diff]), dec(b.raw[diff])
        assert np.all(np.abs(ga - gb) <= 0.13 * np.maximum(np.abs(ga), np.abs(gb)))
    # slots outside the prompt's positions are untouched
    untouched = np.ones(raw.shape[2:5], bool)
    for p in range(start, start + n):
        untouched[table[p // 16], :, p % 16] = False
    assert np.array_equal(a.raw[:, :, untouched], raw[:, :, untouched])
