"""Per-kernel parity through the C ABI (include/mbt_ops.h) against the oracle.

Activations are fp32 on both sides of every kernel (only weights and the KV
cache have narrow formats), so the oracle receives exactly the GPU's inputs.
Tolerances (derived from the arithmetic, written per test):
* fp32 dot products of length K: |gpu - exact| <= 2e-5 * sum_k |w_k x_k| + 1e-7
  (K <= 28672 products accumulated in fp32 by 256 threads and a tree, each
  partial sum with relative error ~K_partial * 2^-24; 2e-5 is ~3x that bound).
* RMSNorm in fp32: relative 1e-5 (sum of squares over <= 42 rounding steps,
  then three multiplications).
* bit-exact where both sides round the same exact value once (V writes,
  K writes at position 0, arg-max decided on the GPU's own logits)."""
import numpy as np
import pytest
import torch

from memory_bound_transformer_gb300 import capi
from oracle.decode import OracleKV, decode_weight, paged_attention, rmsnorm, rope, silu
from oracle.numerics import bf16_decode, e4m3_decode, round_bf16, round_e4m3
from synth import ModelConfig, gen_tensor, random_kv_pool, seeded_block_tables
from tests.helpers import kv_numpy

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_REL, TOL_ABS = 2e-5, 1e-7


def _bf16_rand(shape, seed, scale=1.0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def _f32_rand(shape, seed, scale=1.0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randn(shape, generator=g) * scale


def _np_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _weights(wt, rows, K, seed):
    cfg = ModelConfig("op", 1, K, 1, 1, 64, 16, rows, weight_dtype=wt)
    t = gen_tensor(cfg, seed, "lm_head", -1, device=DEV)      # [rows][K], N(0, 0.02)
    raw = {"w": (t["w"].view(torch.int16).cpu().numpy().view(np.uint16) if wt == "bf16"
                 else t["w"].cpu().numpy())}
    if "s" in t:
        raw["s"] = t["s"].cpu().numpy()
    return t, raw


def _ulp(x, sig, min_e):
    """Spacing of the format's grid at magnitude x (sig significant bits)."""
    e = np.maximum(np.floor(np.log2(np.maximum(x, 2.0 ** min_e))), min_e)
    return 2.0 ** (e - (sig - 1))


def _dtype(wt):
    return capi.DTYPE_E4M3 if wt == "fp8" else capi.DTYPE_BF16


@pytest.mark.parametrize("wt", ["bf16", "fp8"])
@pytest.mark.parametrize("B", [1, 2, 3, 8, 13])
@pytest.mark.parametrize("N,K", [(1000, 1040), (64, 16), (4099, 2048)])
def test_gemv_partial(cuda_lib, wt, B, N, K):
    t, raw = _weights(wt, N, K, seed=N + K + B)
    x = _f32_rand((B, K), seed=B).to(DEV)
    ns = capi.op_gemv_nsplit(capi.EPI_PARTIAL, _dtype(wt), B, N, K)
    for force in (0, 3):
        out = torch.full((max(force, ns), B, N), float("nan"), device=DEV)
        used = capi.op_gemv(capi.EPI_PARTIAL, _dtype(wt), t["w"], t.get("s"), N, K, x, B,
                            force_nsplit=force, out=out)
        # a forced split count is clamped to the number of 16-byte vectors per row
        assert used == (min(force, K // (8 if wt == "bf16" else 16)) if force else ns)
        got = out[:used].sum(0).double().cpu().numpy()
        W = decode_weight(raw)
        xv = x.double().cpu().numpy()
        ref = xv @ W.T
        bound = TOL_REL * (np.abs(xv) @ np.abs(W).T) + TOL_ABS
        assert np.all(np.abs(got - ref) <= bound)


@pytest.mark.parametrize("wt", ["bf16", "fp8"])
@pytest.mark.parametrize("B", [1, 4, 8, 11])
def test_gemv_swiglu(cuda_lib, wt, B):
    F, K = 688, 256
    t, raw = _weights(wt, 2 * F, K, seed=7 + B)
    x = _f32_rand((B, K), seed=3 + B, scale=3.0).to(DEV)
    act = torch.zeros((B, F), device=DEV)
    capi.op_gemv(capi.EPI_SWIGLU, _dtype(wt), t["w"], t.get("s"), F, K, x, B, act=act)
    W = decode_weight(raw)
    xv = x.double().cpu().numpy()
    gu = xv @ W.T
    bound_gu = TOL_REL * (np.abs(xv) @ np.abs(W).T) + TOL_ABS
    g, u = gu[:, :F], gu[:, F:]
    ref = silu(g) * u
    got = act.double().cpu().numpy()
    # fp32 error of g and u propagated (|silu'| <= 1.1), plus fp32 evaluation of silu(g) * u
    bound = 1e-6 * np.abs(ref) + 1.1 * np.abs(u) * bound_gu[:, :F] + np.abs(silu(g)) * bound_gu[:, F:] + 1e-30
    assert np.all(np.abs(got - ref) <= bound)


@pytest.mark.parametrize("wt", ["bf16", "fp8"])
@pytest.mark.parametrize("B", [1, 3, 4, 9])
@pytest.mark.parametrize("epi", ["partial", "swiglu"])
def test_gemv_norm_prologue(cuda_lib, wt, B, epi):
    """The projection with the step's residual add + RMSNorm prologue: x =
    rmsnorm(r + d0 + d1) * gamma formed per CTA, the new residual stored."""
    K = 1040
    N = 1000 if epi == "partial" else 344
    rows = N if epi == "partial" else 2 * N
    t, raw = _weights(wt, rows, K, seed=5 + B)
    r = _f32_rand((B, K), seed=40 + B, scale=2.0).to(DEV)
    delta = _f32_rand((2, B, K), seed=50 + B, scale=0.5).to(DEV)
    gamma = (1.0 + 0.1 * _f32_rand((K,), seed=60)).to(torch.bfloat16).to(DEV)
    r_out = torch.full((B, K), float("nan"), device=DEV)
    out = torch.full((1, B, N), float("nan"), device=DEV)
    act = torch.full((B, N), float("nan"), device=DEV)
    e = capi.EPI_PARTIAL if epi == "partial" else capi.EPI_SWIGLU
    capi.op_gemv_norm(e, _dtype(wt), t["w"], t.get("s"), N, K, r, delta, gamma, 1e-6, r_out,
                      out=out if epi == "partial" else None, act=act if epi == "swiglu" else None)
    torch.cuda.synchronize()
    rsum = r.double() + delta.double()[0] + delta.double()[1]
    # the residual: fp32 sums in the fixed order (r + d0) + d1, bit for bit
    r32, d32 = r.cpu().numpy(), delta.cpu().numpy()
    assert np.array_equal(r_out.cpu().numpy(), (r32 + d32[0]) + d32[1])
    xv = rmsnorm(rsum.cpu().numpy(), bf16_decode(_np_bits(gamma)), 1e-6)
    W = decode_weight(raw)
    ref = xv @ W.T
    # norm in fp32 (relative 1e-5 of each x element) then the fp32 dot product
    bound = (TOL_REL + 1e-5) * (np.abs(xv) @ np.abs(W).T) + TOL_ABS
    if epi == "partial":
        got = out[0].double().cpu().numpy()
        assert np.all(np.abs(got - ref) <= bound)
    else:
        g, u = ref[:, :N], ref[:, N:]
        want = silu(g) * u
        got = act.double().cpu().numpy()
        tol = 1e-6 * np.abs(want) + 1.1 * np.abs(u) * bound[:, :N] + np.abs(silu(g)) * bound[:, N:] + 1e-30
        assert np.all(np.abs(got - want) <= tol)


@pytest.mark.parametrize("wt", ["bf16", "fp8"])
@pytest.mark.parametrize("B", [1, 5, 8, 9])
def test_gemv_argmax(cuda_lib, wt, B):
    V, K = 3001, 512
    t, raw = _weights(wt, V, K, seed=11 + B)
    x = _f32_rand((B, K), seed=21 + B, scale=2.0).to(DEV)
    logits = torch.zeros((B, V), device=DEV)
    ids = torch.full((B,), -1, dtype=torch.int32, device=DEV)
    capi.op_gemv(capi.EPI_ARGMAX, _dtype(wt), t["w"], t.get("s"), V, K, x, B, logits=logits, next_ids=ids)
    lg = logits.cpu().numpy().astype(np.float64)
    got_ids = ids.cpu().numpy()
    # the decision is taken on the GPU's own fp32 logits: first maximum
    assert np.array_equal(got_ids, np.argmax(lg, axis=1))
    W = decode_weight(raw)
    xv = x.double().cpu().numpy()
    ref = xv @ W.T
    bound = TOL_REL * (np.abs(xv) @ np.abs(W).T) + TOL_ABS
    assert np.all(np.abs(lg - ref) <= bound)
    srt = np.sort(ref, axis=1)
    margin = srt[:, -1] - srt[:, -2]
    clear = margin > 2 * bound.max()
    assert np.array_equal(got_ids[clear], np.argmax(ref, axis=1)[clear])
    # without logits the ids are the same
    ids2 = torch.full((B,), -1, dtype=torch.int32, device=DEV)
    capi.op_gemv(capi.EPI_ARGMAX, _dtype(wt), t["w"], t.get("s"), V, K, x, B, next_ids=ids2)
    assert torch.equal(ids, ids2)


@pytest.mark.parametrize("wt", ["bf16", "fp8"])
@pytest.mark.parametrize("B", [1, 3])
def test_gemv_work_queue_every_row(cuda_lib, wt, B):
    """Projections tall enough for the work-queue tail (every CTA owns several
    8-row groups, half of them claimed at run time): every output row of the
    three epilogues against the oracle, and the same ids with and without
    logits (rows reach a CTA out of order across CTAs)."""
    K = 256
    N = 16384
    t, raw = _weights(wt, N, K, seed=101 + B)
    x = _f32_rand((B, K), seed=31 + B, scale=2.0).to(DEV)
    W = decode_weight(raw)
    xv = x.double().cpu().numpy()
    ref = xv @ W.T
    bound = TOL_REL * (np.abs(xv) @ np.abs(W).T) + TOL_ABS
    ns = capi.op_gemv_nsplit(capi.EPI_PARTIAL, _dtype(wt), B, N, K)
    out = torch.full((ns, B, N), float("nan"), device=DEV)
    capi.op_gemv(capi.EPI_PARTIAL, _dtype(wt), t["w"], t.get("s"), N, K, x, B, out=out)
    assert np.all(np.abs(out.sum(0).double().cpu().numpy() - ref) <= bound)
    # SwiGLU over the same rows read as [gate; up]
    F = N // 2
    act = torch.full((B, F), float("nan"), device=DEV)
    capi.op_gemv(capi.EPI_SWIGLU, _dtype(wt), t["w"], t.get("s"), F, K, x, B, act=act)
    g, u = ref[:, :F], ref[:, F:]
    want = silu(g) * u
    b_act = 1e-6 * np.abs(want) + 1.1 * np.abs(u) * bound[:, :F] + np.abs(silu(g)) * bound[:, F:] + 1e-30
    assert np.all(np.abs(act.double().cpu().numpy() - want) <= b_act)
    # arg-max over all rows
    logits = torch.zeros((B, N), device=DEV)
    ids = torch.full((B,), -1, dtype=torch.int32, device=DEV)
    capi.op_gemv(capi.EPI_ARGMAX, _dtype(wt), t["w"], t.get("s"), N, K, x, B, logits=logits, next_ids=ids)
    lg = logits.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(lg - ref) <= bound)
    assert np.array_equal(ids.cpu().numpy(), np.argmax(lg, axis=1))
    ids2 = torch.full((B,), -1, dtype=torch.int32, device=DEV)
    capi.op_gemv(capi.EPI_ARGMAX, _dtype(wt), t["w"], t.get("s"), N, K, x, B, next_ids=ids2)
    assert torch.equal(ids, ids2)
    # caller-owned counters: three launches in a row on one zeroed array give
    # the same bits as op_gemv, and the array is zero again afterwards
    n_int = capi.op_gemv_sched_ints(capi.EPI_PARTIAL, _dtype(wt), B, N, K)
    assert n_int >= 1
    sched = torch.zeros(n_int, dtype=torch.int32, device=DEV)
    for _ in range(3):
        out2 = torch.full_like(out, float("nan"))
        capi.op_gemv_ex(capi.EPI_PARTIAL, _dtype(wt), t["w"], t.get("s"), N, K, x, B, sched, out=out2)
        torch.cuda.synchronize()
        assert torch.equal(out2, out)
        assert int(sched.abs().sum().item()) == 0


@pytest.mark.parametrize("wt,N,K,B", [("bf16", 28672, 4096, 1), ("bf16", 4096, 14336, 8),
                                      ("fp8", 8192, 28672, 8), ("fp8", 57344, 8192, 1),
                                      ("bf16", 128256, 4096, 1)])
def test_gemv_full_size_sampled(cuda_lib, wt, N, K, B):
    """Full model-size projections (8B gate/up, down, LM head; 70B down,
    gate/up): 64 sampled output rows checked one by one by the oracle."""
    t, _ = _weights(wt, N, K, seed=N ^ K)
    x = _f32_rand((B, K), seed=5).to(DEV)
    ns = capi.op_gemv_nsplit(capi.EPI_PARTIAL, _dtype(wt), B, N, K)
    out = torch.zeros((ns, B, N), device=DEV)
    capi.op_gemv(capi.EPI_PARTIAL, _dtype(wt), t["w"], t.get("s"), N, K, x, B, out=out)
    got = out.sum(0).double().cpu().numpy()
    rows = np.sort(np.random.default_rng(N).choice(N, 64, replace=False))
    rows[-1] = N - 1
    sub = {"w": (t["w"][rows].view(torch.int16).cpu().numpy().view(np.uint16) if wt == "bf16"
                 else t["w"][rows].cpu().numpy())}
    if "s" in t:
        sub["s"] = t["s"][rows].cpu().numpy()
    W = decode_weight(sub)
    xv = x.double().cpu().numpy()
    ref = xv @ W.T
    bound = TOL_REL * (np.abs(xv) @ np.abs(W).T) + TOL_ABS
    assert np.all(np.abs(got[:, rows] - ref) <= bound)


@pytest.mark.parametrize("H", [256, 4096, 8192, 336, 5120, 1480])
def test_norms(cuda_lib, H):
    B, V = 5, 777
    emb = _bf16_rand((V, H), 1, 0.02).to(DEV)
    gamma = (1 + 0.1 * torch.randn(H)).to(torch.bfloat16).to(DEV)
    tok = torch.tensor([0, 5, 776, 123, 5], dtype=torch.int32, device=DEV)
    r = torch.zeros((B, H), device=DEV)
    y = torch.zeros((B, H), device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    capi.op_embed_rmsnorm(tok, emb, gamma, 1e-6, r, y, err)
    e = bf16_decode(_np_bits(emb.cpu()))[tok.cpu().numpy()]
    g = bf16_decode(_np_bits(gamma.cpu()))
    assert np.array_equal(r.cpu().numpy().astype(np.float64), e)
    ref = rmsnorm(e, g, 1e-6)
    got = y.double().cpu().numpy()
    assert np.all(np.abs(got - ref) <= 1e-5 * np.abs(ref) + 1e-30)
    assert err.item() == 0
    # residual add of 3 split partials, then the norm
    delta = torch.randn((3, B, H), device=DEV)
    r0 = r.double().cpu().numpy()
    capi.op_add_rmsnorm(r, delta, gamma, 1e-6, y)
    rr = r0 + delta.double().cpu().numpy().sum(0)
    np.testing.assert_allclose(r.double().cpu().numpy(), rr, rtol=1e-6, atol=1e-6)
    ref = rmsnorm(rr, g, 1e-6)
    got = y.double().cpu().numpy()
    assert np.all(np.abs(got - ref) <= 1e-5 * np.abs(ref) + 1e-6)
    # out-of-range token: error bit, token 0 used
    bad = torch.tensor([-1, V], dtype=torch.int32, device=DEV)
    capi.op_embed_rmsnorm(bad, emb, gamma, 1e-6, r[:2], y[:2], err)
    torch.cuda.synchronize()
    assert err.item() & capi.DEV_TOKEN_RANGE


def _rope_case(nq, nkv, d, kv, B, seed):
    rng = np.random.default_rng(seed)
    qkv = torch.tensor(rng.normal(size=(B, (nq + 2 * nkv) * d)) * 1.5, dtype=torch.float32, device=DEV)
    pos = np.array(rng.integers(0, 200, size=B), np.int32)
    pos[0] = 0
    nb = int(sum(p // 16 + 1 for p in pos)) + 2
    tables = seeded_block_tables(pos + 1, 16, nb, seed)
    return qkv, pos, tables, nb


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("nq,nkv,d", [(4, 2, 64), (32, 8, 128), (10, 2, 64), (64, 8, 128)])
def test_rope_kv_write(cuda_lib, kv, nq, nkv, d):
    B = 6
    qkv, pos, tables, nb = _rope_case(nq, nkv, d, kv, B, seed=nq + d)
    esz = 1 if kv == "fp8" else 2
    half = (nb + 1) * nkv * 16 * d * esz
    sentinel = 0x5A
    pool = torch.full((2 * half,), sentinel, dtype=torch.uint8, device=DEV)
    q_out = torch.zeros((B, nq, d), device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    posd = torch.tensor(pos, device=DEV)
    btd = torch.tensor(tables, device=DEV)
    capi.op_rope_kv_write(qkv, nq, nkv, d, posd, btd, 512, 10000.0, pool[:half], pool[half:], nb,
                          _dtype(kv), 1.0, 1.0, q_out, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    x = qkv.double().cpu().numpy()
    shape = (nb + 1, nkv, 16, d)
    dt = np.uint8 if kv == "fp8" else np.uint16
    P = pool.cpu().numpy()
    Kp, Vp = P[:half].view(dt).reshape(shape), P[half:].view(dt).reshape(shape)
    dec = e4m3_decode if kv == "fp8" else bf16_decode
    written = np.zeros(shape[:3], bool)
    for b in range(B):
        p = int(pos[b])
        blk, slot = int(tables[b][p // 16]), p % 16
        written[blk, :, slot] = True
        q = rope(x[b, :nq * d].reshape(nq, d), p, 1e4)
        np.testing.assert_allclose(q_out[b].double().cpu().numpy(), q, rtol=0, atol=1e-5 * (1 + np.abs(q).max()))
        k = rope(x[b, nq * d:(nq + nkv) * d].reshape(nkv, d), p, 1e4)
        v = x[b, (nq + nkv) * d:].reshape(nkv, d)
        # V: the same fp32 value rounded once on both sides -> bit-exact
        rnd = round_e4m3 if kv == "fp8" else round_bf16
        assert np.array_equal(Vp[blk, :, slot], rnd(v))
        if p == 0:
            assert np.array_equal(Kp[blk, :, slot], rnd(k))          # cos 1, sin 0: exact
        else:
            # fp32 rotation vs fp64: at most one step of the cache grid apart
            got, want = dec(Kp[blk, :, slot]), dec(rnd(k))
            sig, min_e = (4, -6) if kv == "fp8" else (8, -126)
            assert np.all(np.abs(got - want) <= _ulp(np.maximum(np.abs(got), np.abs(want)), sig, min_e))
    # nothing else was touched
    untouched = ~written
    kb = P[:half].reshape(nb + 1, nkv, 16, d * esz)
    vb = P[half:].reshape(nb + 1, nkv, 16, d * esz)
    assert np.all(kb[untouched] == sentinel) and np.all(vb[untouched] == sentinel)


def test_rope_kv_write_range_errors(cuda_lib):
    nq, nkv, d, B = 4, 2, 64, 2
    qkv, pos, tables, nb = _rope_case(nq, nkv, d, "bf16", B, seed=1)
    half = (nb + 1) * nkv * 16 * d * 2
    pool = torch.full((2 * half,), 0x33, dtype=torch.uint8, device=DEV)
    q_out = torch.zeros((B, nq, d), device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    bad_tab = torch.tensor(tables, device=DEV)
    bad_tab[:, :] = nb + 5                                   # beyond the null block
    capi.op_rope_kv_write(qkv, nq, nkv, d, torch.tensor(pos, device=DEV), bad_tab, 512, 1e4,
                          pool[:half], pool[half:], nb, capi.DTYPE_BF16, 1.0, 1.0, q_out, err)
    torch.cuda.synchronize()
    assert err.item() & capi.DEV_BLOCK_RANGE
    assert torch.all(pool == 0x33)
    err.zero_()
    capi.op_rope_kv_write(qkv, nq, nkv, d, torch.tensor([600, -1], dtype=torch.int32, device=DEV),
                          torch.tensor(tables, device=DEV), 512, 1e4, pool[:half], pool[half:], nb,
                          capi.DTYPE_BF16, 1.0, 1.0, q_out, err)
    torch.cuda.synchronize()
    assert err.item() & capi.DEV_POS_RANGE
    assert torch.all(pool == 0x33)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("nq,nkv,d", [(4, 4, 64), (4, 2, 64), (32, 8, 128), (10, 2, 64), (64, 8, 128),
                                      (16, 1, 128), (40, 8, 128)])
@pytest.mark.parametrize("lens", [[1], [15, 16, 17], [128, 1, 33, 64, 65], [1000], [2049, 7]])
def test_paged_attention(cuda_lib, kv, nq, nkv, d, lens):
    B = len(lens)
    lens_a = np.array(lens, np.int32)
    nb = int(sum(-(-l // 16) for l in lens)) + 3
    stride = max(-(-l // 16) for l in lens) + 2                 # wider than needed
    tables = seeded_block_tables(lens_a, 16, nb, seed=sum(lens), stride=stride)
    tables[tables < 0] = nb                                     # unused entries: null block
    cfg = ModelConfig("a", 1, 64, nq, nkv, d, 16, 16, kv_dtype=kv)
    pool = random_kv_pool(cfg, nb, seed=nq + d + B, device=DEV)    # [1][2][nb+1][nkv][16][d]
    raw = kv_numpy(pool)
    ks, vs = (0.75, 1.25) if kv == "fp8" else (1.0, 1.0)
    okv = OracleKV(raw, np.array([ks]), np.array([vs]))
    rng = np.random.default_rng(B + nq)
    q = rng.normal(size=(B, nq, d)) * 0.6
    qd = torch.tensor(q, dtype=torch.float32, device=DEV)
    out = torch.zeros((B, nq * d), device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    flat = pool.view(torch.uint8).reshape(2, -1)
    capi.op_paged_attention(qd, nkv, flat[0], flat[1], _dtype(kv), ks, vs, torch.tensor(tables, device=DEV),
                            torch.tensor(lens_a, device=DEV), nb, out, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    got = out.double().cpu().numpy().reshape(B, nq, d)
    for b in range(B):
        ref = paged_attention(qd[b].double().cpu().numpy(), okv, 0, tables[b], int(lens_a[b]))
        # fp32 scores, exp2 and accumulation over <= 2049 tokens: ~1e-5 of max|V|
        vmax = np.abs(okv.decode(0, 1, tables[b][: -(-int(lens_a[b]) // 16)])).max()
        assert np.all(np.abs(got[b] - ref) <= 2e-5 * vmax)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_paged_attention_one_wave_batch(cuda_lib, kv):
    """48 rows x 8 KV heads with ~1000-token contexts: the e4m3 kernel plans one
    wave of single-split CTAs (the output written without a merge), the BF16 one
    two splits per (row, KV head); sampled rows against the oracle."""
    nq, nkv, d, B = 64, 8, 128, 48
    rng = np.random.default_rng(48)
    lens_a = rng.integers(900, 1100, size=B).astype(np.int32)
    nb = int(sum(-(-int(l) // 16) for l in lens_a)) + 2
    tables = seeded_block_tables(lens_a, 16, nb, seed=5)
    tables[tables < 0] = nb
    cfg = ModelConfig("a", 1, 64, nq, nkv, d, 16, 16, kv_dtype=kv)
    pool = random_kv_pool(cfg, nb, seed=9, device=DEV)
    okv = OracleKV(kv_numpy(pool), np.array([1.0]), np.array([1.0]))
    qd = torch.tensor(rng.normal(size=(B, nq, d)) * 0.6, dtype=torch.float32, device=DEV)
    out = torch.zeros((B, nq * d), device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    flat = pool.view(torch.uint8).reshape(2, -1)
    capi.op_paged_attention(qd, nkv, flat[0], flat[1], _dtype(kv), 1.0, 1.0, torch.tensor(tables, device=DEV),
                            torch.tensor(lens_a, device=DEV), nb, out, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    got = out.double().cpu().numpy().reshape(B, nq, d)
    for b in (0, 17, 47):
        ref = paged_attention(qd[b].double().cpu().numpy(), okv, 0, tables[b], int(lens_a[b]))
        vmax = np.abs(okv.decode(0, 1, tables[b][: -(-int(lens_a[b]) // 16)])).max()
        assert np.all(np.abs(got[b] - ref) <= 2e-5 * vmax)


def test_paged_attention_bad_seq_len(cuda_lib):
    nq, nkv, d, nb = 4, 2, 64, 4
    cfg = ModelConfig("a", 1, 64, nq, nkv, d, 16, 16)
    pool = random_kv_pool(cfg, nb, seed=1, device=DEV)
    flat = pool.view(torch.uint8).reshape(2, -1)
    q = torch.randn((2, nq, d), device=DEV)
    tables = torch.tensor([[0, 1], [2, 3]], dtype=torch.int32, device=DEV)
    out = torch.full((2, nq * d), 7.0, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    capi.op_paged_attention(q, nkv, flat[0], flat[1], capi.DTYPE_BF16, 1.0, 1.0, tables,
                            torch.tensor([0, 33], dtype=torch.int32, device=DEV), nb, out, err)
    torch.cuda.synchronize()
    assert err.item() & capi.DEV_SEQLEN_RANGE
    assert torch.all(out == 0)
