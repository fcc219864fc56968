"""Sampling beyond greedy (decode_step_sample) through the C ABI against the
oracle's sampler.

The draw is a decision taken in floating point (the top-k boundary, the
top-p cut, the arg-max of z + Gumbel), so both sides decide from the same
numbers: the GPU returns its fp32 logits with the draw and the oracle samples
from those logits (as float64) with the same seed, row and step. The ids must
be equal unless the decision sits within rounding of a boundary: the GPU's
token is then still in the oracle's kept set for top_p moved by 1e-5, and its
z + g is within 1e-4 of the oracle's best. The logits themselves are the
decode step's (bit-identical to a greedy step of a twin engine)."""
import numpy as np
import pytest
import torch

from memory_bound_transformer_gb300 import capi
from oracle.sampling import gumbel, keep_set, sample, uniforms
from synth import EIGHT_B, random_tokens
from tests.helpers import SMALL, SMALL_FP8
from tests.test_gpu_step import Case

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _eff_k(k, p):
    return k if k > 0 else (capi.TOPK_MAX if p < 1.0 else 0)


def _check_draw(logits, got, T, k, p, seed, row, step):
    k = _eff_k(k, p)
    want = sample(logits, T, k, p, seed, row, step)
    if got == want:
        return True
    z = logits / T
    kept = set()
    for pp in (max(p - 1e-5, 1e-9), p, min(p + 1e-5, 1.0)):
        kept |= set(keep_set(logits, T, k, pp).tolist())
    assert got in kept, f"draw {got} outside the kept set (oracle {want})"
    score = lambda i: z[i] + gumbel(uniforms(seed, row, step, [i]))[0]
    assert score(got) >= score(want) - 1e-4, f"draw {got} not a near-tie of {want}"
    return False


PARAMS = [(1.0, 0, 1.0), (0.7, 0, 1.0), (1.3, 50, 1.0), (0.8, 5, 0.9), (1.0, 0, 0.5), (1.0, 1024, 0.95),
          (0.5, 1, 1.0)]


@pytest.mark.parametrize("cfg", [SMALL, SMALL_FP8], ids=lambda c: c.name)
@pytest.mark.parametrize("B", [1, 5, 17])
def test_sampling_matches_oracle_draw(cuda_lib, cfg, B):
    rng = np.random.default_rng(B)
    case = Case(cfg, 60 + B, B, rng.integers(1, 200, size=B), len(PARAMS))
    twin = Case(cfg, 60 + B, B, case.ctx, len(PARAMS))
    exact = 0
    for t, (T, k, p) in enumerate(PARAMS):
        pos = case.ctx + t
        tok = torch.tensor(case.toks[t], device=DEV)
        posd = torch.tensor(pos, device=DEV)
        ids = torch.full((B,), -1, dtype=torch.int32, device=DEV)
        lg = torch.zeros((B, cfg.vocab), device=DEV)
        seed, step = 1000 + t, 7 * t
        case.eng.step_sample(tok, posd, case.bt_dev, posd + 1, ids, T, k, p, seed, step, lg)
        gid = torch.full((B,), -1, dtype=torch.int32, device=DEV)
        glg = torch.zeros((B, cfg.vocab), device=DEV)
        twin.eng.step(tok, posd, twin.bt_dev, posd + 1, gid, glg)
        torch.cuda.synchronize()
        assert torch.equal(lg, glg), "sampling changed the logits of the step"
        L = lg.double().cpu().numpy()
        got = ids.cpu().numpy()
        for b in range(B):
            exact += _check_draw(L[b], int(got[b]), T, k, p, seed, b, step)
        if (T, k, p) == (0.5, 1, 1.0):
            assert np.array_equal(got, gid.cpu().numpy())          # top-1: the greedy id
    assert case.eng.errors() == 0 and twin.eng.errors() == 0
    assert exact >= 0.9 * B * len(PARAMS)


def test_sampling_draws_vary_with_step_and_seed(cuda_lib):
    """Fresh draws per step, the same draw for the same (seed, step), and
    temperature sampling spreads over tokens the greedy step never picks."""
    cfg = SMALL
    case = Case(cfg, 5, 1, [40], 1)
    tok = torch.tensor(case.toks[0], device=DEV)
    pos = torch.tensor(case.ctx, device=DEV)
    seen, first = set(), None
    for s in range(64):
        ids = torch.zeros(1, dtype=torch.int32, device=DEV)
        case.eng.step_sample(tok, pos, case.bt_dev, pos + 1, ids, 3.0, 0, 1.0, 11, s)
        seen.add(int(ids.item()))
        if s == 0:
            first = int(ids.item())
    again = torch.zeros(1, dtype=torch.int32, device=DEV)
    case.eng.step_sample(tok, pos, case.bt_dev, pos + 1, again, 3.0, 0, 1.0, 11, 0)
    torch.cuda.synchronize()
    assert int(again.item()) == first
    assert len(seen) > 8


def test_sampling_keeps_graphs_and_rejects_bad_params(cuda_lib):
    cfg = SMALL
    case = Case(cfg, 6, 2, [30, 50], 1, ladder=[1, 2], graph=True)
    m, kv = case.eng.model, case.eng.kv
    d = torch.zeros(2, dtype=torch.int32, device=DEV)
    bt = case.bt_dev
    for T, k, p in ((0.0, 0, 1.0), (1.0, -1, 1.0), (1.0, 1025, 1.0), (1.0, 0, 0.0), (1.0, 0, 1.5),
                    (float("nan"), 0, 1.0)):
        sp = capi.Sampling(T, k, p, 0, 1, 1)
        assert capi.decode_step_sample_raw(m, kv, 2, d, d, bt, bt.shape[1], d + 1, sp, d) == -1
    assert capi.decode_step_sample_raw(m, kv, 2, d, d, bt, bt.shape[1], d + 1, None, d) == -1
    ids = torch.zeros(2, dtype=torch.int32, device=DEV)
    pos = torch.tensor(case.ctx, device=DEV)
    case.eng.step_sample(torch.tensor(case.toks[0], device=DEV), pos, bt, pos + 1, ids, 1.0, 10, 0.9, 3, 4)
    assert case.eng.stats(2)[1]
    assert case.eng.errors() == 0


@pytest.mark.parametrize("B", [1, 16])
def test_sampling_8b_full_size(cuda_lib, B):
    """8B-class BF16 vocabulary (128256 logits per row): the fused draw at
    batch 1 (CUDA-core LM head) and 16 (tensor-core LM head), and top-k /
    top-p draws, against the oracle's sampler on the GPU's logits."""
    from memory_bound_transformer_gb300 import blob as mblob
    from memory_bound_transformer_gb300.engine import Engine
    from synth import SynthModel, random_kv_pool, seeded_block_tables
    cfg = EIGHT_B
    model = SynthModel(cfg, 1237, device=DEV, cache=False)
    blob = mblob.pack(cfg, model.tensors(), device=DEV)
    ctx = np.random.default_rng(3).integers(256, 2048, size=B).astype(np.int32)
    nb = int(sum(-(-int(c + 1) // 16) for c in ctx)) + 2
    tables = seeded_block_tables(ctx + 1, 16, nb, 4)
    tables[tables < 0] = nb
    eng = Engine(blob, nb)
    del blob
    try:
        eng.pool().copy_(random_kv_pool(cfg, nb, 5, device=DEV).view(torch.uint8).reshape(-1))
        tok = torch.tensor(random_tokens(B, cfg.vocab, 9), device=DEV)
        pos = torch.tensor(ctx, device=DEV)
        bt = torch.tensor(tables, device=DEV)
        for i, (T, k, p) in enumerate([(1.0, 0, 1.0), (0.8, 40, 0.9), (1.2, 0, 0.7)]):
            ids = torch.full((B,), -1, dtype=torch.int32, device=DEV)
            lg = torch.zeros((B, cfg.vocab), device=DEV)
            eng.step_sample(tok, pos, bt, pos + 1, ids, T, k, p, 77, i, lg)
            torch.cuda.synchronize()
            L = lg.double().cpu().numpy()
            for b in range(B):
                _check_draw(L[b], int(ids[b].item()), T, k, p, 77, b, i)
        assert eng.errors() == 0
    finally:
        eng.close()
