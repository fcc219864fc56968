"""Whole decode-step parity through the C ABI (include/mbt.h) against the oracle.

Acceptance: max |logit - oracle| <= 3e-2 for BF16 models and 1.5e-1 for FP8
models over every checked row and step; greedy ids equal wherever the oracle's
top-2 margin exceeds 1e-2; the set of cache bytes a step writes is exactly the
slots of the rows' positions (sentinel bytes elsewhere unchanged, padding rows
only in the null block), and the written values agree with the oracle's to the
tolerance of the values that produce them.

Both sides start from the same random cache and each keeps its own cache across
steps (the oracle never reads GPU results); tokens are random at every step, so
a disagreement in one step's id cannot cascade."""
import json
import os

import numpy as np
import pytest
import torch

from memory_bound_transformer_gb300 import blob as mblob
from memory_bound_transformer_gb300 import capi
from memory_bound_transformer_gb300.engine import Engine
from oracle.decode import OracleKV, decode_step
from oracle.numerics import bf16_decode, e4m3_decode
from synth import (ONE_B, TINY, WORKLOADS, SynthModel, random_contexts, raw_numpy, random_kv_pool,
                   random_tokens, seeded_block_tables)
from tests.helpers import SMALL, SMALL_D128, SMALL_FP8, SMALL_G5, kv_numpy, oracle_weights

pytestmark = pytest.mark.gpu
DEV = "cuda"


def tol_logits(cfg):
    return 1.5e-1 if cfg.weight_dtype == "fp8" or cfg.kv_dtype == "fp8" else 3e-2


class Case:
    """Model + cache + block tables shared by the GPU engine and the oracle."""

    def __init__(self, cfg, seed, B, ctx, steps, cache_weights=True, ladder=None, graph=False):
        self.cfg, self.B, self.steps = cfg, B, steps
        self.model = SynthModel(cfg, seed, device=DEV, cache=cache_weights)
        self.blob = mblob.pack(cfg, self.model.tensors(), device=DEV)
        self.ctx = np.asarray(ctx, np.int32)
        cap = self.ctx + steps
        self.nb = int(sum(-(-int(c) // 16) for c in cap)) + 2
        self.tables = seeded_block_tables(cap, 16, self.nb, seed + 1)
        self.tables[self.tables < 0] = self.nb
        self.eng = Engine(self.blob, self.nb)
        del self.blob
        pool0 = random_kv_pool(cfg, self.nb, seed + 2, device=DEV)
        self.eng.pool().copy_(pool0.view(torch.uint8).reshape(-1))
        self.pool0 = kv_numpy(pool0)
        self.toks = random_tokens(B * steps, cfg.vocab, seed + 3).reshape(steps, B)
        if graph:
            self.eng.capture(ladder, max_blocks_per_seq=self.tables.shape[1])
        self.bt_dev = torch.tensor(self.tables, device=DEV)

    def gpu_step(self, t, logits=True):
        B = self.B
        pos = self.ctx + t
        tok = torch.tensor(self.toks[t], device=DEV)
        posd = torch.tensor(pos, device=DEV)
        sl = torch.tensor(pos + 1, device=DEV)
        ids = torch.full((B,), -1, dtype=torch.int32, device=DEV)
        lg = torch.zeros((B, self.cfg.vocab), device=DEV) if logits else None
        self.eng.step(tok, posd, self.bt_dev, sl, ids, lg)
        torch.cuda.synchronize()
        return ids.cpu().numpy(), (lg.double().cpu().numpy() if logits else None)

    def gpu_pool(self):
        raw = self.eng.pool().cpu().numpy()
        dt = np.uint8 if self.cfg.kv_dtype == "fp8" else np.uint16
        return raw.view(dt).reshape(self.pool0.shape)


def parity_log(what, value):
    """Append a measured error to the file MBT_PARITY_LOG names (if set), one
    JSON line per check, tagged with the running test."""
    path = os.environ.get("MBT_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"test": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0],
                                what: value}) + "\n")


def _check_step(cfg, ids, lg, res):
    tol = tol_logits(cfg)
    err = np.abs(lg - res.logits).max()
    parity_log("max_logit_err", float(err))
    assert err <= tol, f"max logit error {err}"
    srt = np.sort(res.logits, axis=1)
    clear = (srt[:, -1] - srt[:, -2]) > 1e-2
    assert np.array_equal(ids[clear], res.next_ids[clear])
    assert np.array_equal(ids, np.argmax(lg, axis=1))
    return err


def grid_step(x, fmt):
    """Spacing of the cache format's value grid at |x| (one unit in the last
    place): BF16 keeps 8 significant bits, e4m3 4 with subnormals below 2^-6."""
    a = np.abs(np.asarray(x, np.float64))
    _, e = np.frexp(np.where(a > 0, a, 1.0))
    if fmt == "fp8":
        return np.ldexp(1.0, np.maximum(e - 1, -6) - 3)
    return np.ldexp(1.0, np.maximum(e - 1, -126) - 7)


def check_cache(gp, pool0, oraw, mask, fmt, skip_null_block=None):
    """gp, pool0, oraw: [L][2][blocks][nkv][16][d] raw storage (GPU after the
    steps, initial, oracle after the steps); mask [blocks][nkv][16] marks the
    written (block, head, slot). Bytes elsewhere equal the initial pool on both
    sides. Every written element is within one step of the cache grid of the
    oracle's value plus a third of the logit tolerance relative to the row's
    largest magnitude: the GPU's K and V are projections of its fp32 residual
    stream, which after many layers deviates from the fp64 one by the same
    relative amount the logit tolerance bounds (a value from a wrong head or
    slot differs by about the row's magnitude and fails)."""
    for arr, skip in ((gp, skip_null_block), (oraw, None)):
        same = np.all(arr == pool0, axis=-1)             # [L][2][blocks][nkv][16]
        keep = ~mask
        if skip is not None:                             # graph padding rows write the null block
            keep[skip] = False
        assert np.all(same[:, :, keep]), "a byte outside the written slots changed"
    dec = e4m3_decode if fmt == "fp8" else bf16_decode
    g = dec(gp[:, :, mask])
    o = dec(oraw[:, :, mask])
    assert np.all(np.isfinite(g))
    row = np.abs(o).max(axis=-1, keepdims=True)
    rel = (1.5e-1 if fmt == "fp8" else 3e-2) / 3
    bound = grid_step(np.maximum(np.abs(g), np.abs(o)), fmt) + rel * row
    worst = np.max(np.abs(g - o) - bound)
    parity_log("kv_excess_over_bound", float(worst))
    assert worst <= 0, f"written K/V beyond the bound by {worst}"


def _check_pool(case, okv, written):
    """written: set of (block, slot) of the whole batch."""
    mask = np.zeros(case.pool0.shape[2:5], bool)         # [nb+1][nkv][16]
    for blk, slot in written:
        mask[blk, :, slot] = True
    check_cache(case.gpu_pool(), case.pool0, okv.raw, mask, case.cfg.kv_dtype, skip_null_block=case.nb)


def _run(case, W, okv, steps):
    cfg = case.cfg
    written = set()
    worst = 0.0
    for t in range(steps):
        pos = case.ctx + t
        ids, lg = case.gpu_step(t)
        res = decode_step(W, cfg, okv, case.toks[t], pos, case.tables, pos + 1)
        worst = max(worst, _check_step(cfg, ids, lg, res))
        for b in range(case.B):
            written.add((int(case.tables[b][pos[b] // 16]), int(pos[b] % 16)))
    assert case.eng.errors() == 0
    _check_pool(case, okv, written)
    return worst


def test_tiny_layer_workload(cuda_lib):
    """Single decoder layer + LM head, batch 1, 128 tokens of random KV, 8 decode
    steps from random token ids, replayed from a captured graph."""
    cfg = TINY
    case = Case(cfg, 1235, 1, [128], 8, ladder=[1], graph=True)
    okv = OracleKV(case.pool0.copy(), np.ones(cfg.n_layers), np.ones(cfg.n_layers))
    assert case.eng.stats(1)[1]
    _run(case, oracle_weights(case.model), okv, 8)


@pytest.mark.parametrize("cfg", [SMALL, SMALL_FP8, SMALL_D128, SMALL_G5], ids=lambda c: c.name)
@pytest.mark.parametrize("B", [1, 3, 13])
def test_small_models_eager(cuda_lib, cfg, B):
    rng = np.random.default_rng(B)
    ctx = rng.integers(0, 300, size=B)
    ctx[0] = 0
    if B > 2:
        ctx[1], ctx[2] = 15, 16
    case = Case(cfg, 77 + B, B, ctx, 3)
    okv = OracleKV(case.pool0.copy(), np.ones(cfg.n_layers), np.ones(cfg.n_layers))
    _run(case, oracle_weights(case.model), okv, 3)


def test_fp8_cache_scales(cuda_lib):
    cfg = SMALL_FP8
    case = Case(cfg, 5, 3, [40, 1, 70], 2)
    ks, vs = [0.5, 1.5], [2.0, 0.75]
    case.eng.set_kv_scales(ks, vs)
    okv = OracleKV(case.pool0.copy(), np.array(ks), np.array(vs))
    _run(case, oracle_weights(case.model), okv, 2)


def test_graph_replay_bit_identical_to_eager(cuda_lib):
    """Graphs change how the step is launched, not what it computes: replaying
    the rung-4 graph for 4 rows gives the eager run's bits exactly."""
    cfg = SMALL
    B = 4
    ctx = [20, 47, 5, 160]
    a = Case(cfg, 9, B, ctx, 3)
    b = Case(cfg, 9, B, ctx, 3, ladder=[1, 2, 4, 8], graph=True)
    assert b.eng.stats(B)[1] and not a.eng.stats(B)[1]
    for t in range(3):
        ia, la = a.gpu_step(t)
        ib, lb = b.gpu_step(t)
        assert np.array_equal(ia, ib)
        assert np.array_equal(la, lb)
    # the capture's warm-up ran padding rows, which write the null block only
    pa, pb = a.gpu_pool(), b.gpu_pool()
    assert np.array_equal(pa[:, :, :a.nb], pb[:, :, :b.nb])
    assert a.eng.errors() == 0 and b.eng.errors() == 0


def test_graph_ladder_padding_and_fallback(cuda_lib):
    """13 live rows replay the graph captured for 16; 70 rows exceed the top
    rung and run eagerly; both match the oracle. The eager step needs more
    workspace than the graphs were captured with, and must leave them in
    place: 13 rows replay the graph again afterwards."""
    cfg = SMALL
    B = 70
    rng = np.random.default_rng(B)
    case = Case(cfg, 31, B, rng.integers(1, 100, size=B), 3, ladder=[1, 2, 4, 8, 16], graph=True)
    okv = OracleKV(case.pool0.copy(), np.ones(cfg.n_layers), np.ones(cfg.n_layers))
    W = oracle_weights(case.model)
    assert case.eng.stats(13)[1] and not case.eng.stats(70)[1]
    written = set()
    for t, rows in ((0, np.arange(13)), (1, np.arange(70)), (2, np.arange(13))):
        _step_rows(case, W, okv, t, rows, written)
        assert case.eng.stats(13)[1], "an eager step dropped the captured graphs"
    assert case.eng.errors() == 0
    _check_pool(case, okv, written)


def _step_rows(case, W, okv, t, rows, written, bt=None, sl=None, check=True):
    """Step t for a subset of the case's rows (their own tables unless `bt`),
    on the GPU and, when `check`, on the oracle; returns (ids, logits)."""
    cfg = case.cfg
    pos = case.ctx[rows] + t
    tables = case.tables[rows] if bt is None else bt
    seq = pos + 1 if sl is None else sl
    lg = torch.zeros((len(rows), cfg.vocab), device=DEV)
    ids = torch.full((len(rows),), -1, dtype=torch.int32, device=DEV)
    case.eng.step(torch.tensor(case.toks[t][rows], device=DEV), torch.tensor(pos, device=DEV),
                  torch.tensor(np.ascontiguousarray(tables), device=DEV), torch.tensor(seq, device=DEV), ids, lg)
    torch.cuda.synchronize()
    ids, lg = ids.cpu().numpy(), lg.double().cpu().numpy()
    if check:
        res = decode_step(W, cfg, okv, case.toks[t][rows], pos, tables, seq)
        _check_step(cfg, ids, lg, res)
        for b, p in zip(rows, pos):
            written.add((int(case.tables[b][p // 16]), int(p % 16)))
    return ids, lg


def test_graph_table_width(cuda_lib):
    """Graphs captured for tables of 10 entries. A caller table of 7 entries
    replays the graph and matches the oracle. A row whose seq_len needs more
    blocks than the caller's 7 is flagged MBT_DEV_SEQLEN_RANGE and attends over
    nothing, on the graph and on the eager path alike (same logits). A table of
    12 entries with a 180-token context runs eagerly, matches the oracle, and
    leaves the graphs in place."""
    cfg = SMALL
    B = 4
    ctx = np.array([20, 47, 5, 100])
    g = Case(cfg, 12, B, ctx, 2)
    e = Case(cfg, 12, B, ctx, 2)
    assert g.tables.shape[1] == 7
    g.eng.capture([1, 2, 4, 8], max_blocks_per_seq=10)
    e.eng.set_eager(True)
    okv = OracleKV(g.pool0.copy(), np.ones(cfg.n_layers), np.ones(cfg.n_layers))
    W = oracle_weights(g.model)
    rows = np.arange(B)
    written = set()
    # narrower caller table: the graph serves it
    assert g.eng.stats(B)[1]
    _step_rows(g, W, okv, 0, rows, written)
    _step_rows(e, W, OracleKV(e.pool0.copy(), np.ones(2), np.ones(2)), 0, rows, set())
    assert g.eng.errors() == 0 and e.eng.errors() == 0
    # row 3's seq_len needs 8 blocks, one more than its table holds
    sl = ctx + 2
    sl[3] = 7 * 16 + 5
    ig, lgg = _step_rows(g, W, okv, 1, rows, written, sl=sl, check=False)
    ie, lge = _step_rows(e, W, okv, 1, rows, set(), sl=sl, check=False)
    assert g.eng.errors() & capi.DEV_SEQLEN_RANGE
    assert e.eng.errors() & capi.DEV_SEQLEN_RANGE
    assert np.abs(lgg[3] - lge[3]).max() <= 1e-3
    # wider table with a longer context: eager, correct, graphs kept
    wide = Case(cfg, 13, 1, [180], 1)
    wide.eng.capture([1, 2, 4], max_blocks_per_seq=10)
    assert wide.tables.shape[1] == 12
    wokv = OracleKV(wide.pool0.copy(), np.ones(cfg.n_layers), np.ones(cfg.n_layers))
    ww = set()
    _step_rows(wide, oracle_weights(wide.model), wokv, 0, np.arange(1), ww)
    assert wide.eng.errors() == 0
    assert wide.eng.stats(1)[1]
    _check_pool(wide, wokv, ww)


@pytest.mark.parametrize("B", [1, 8])
def test_1b_workload(cuda_lib, B):
    """1B-class decoder at batch 1 and 8 with the graph ladder 1, 2, 4, 8:
    all 64 decode steps after a 512-token (random) context, every row."""
    cfg = ONE_B
    case = Case(cfg, 1236, B, [512] * B, 64, ladder=[1, 2, 4, 8], graph=True)
    okv = OracleKV(case.pool0.copy(), np.ones(cfg.n_layers), np.ones(cfg.n_layers))
    _run(case, oracle_weights(case.model), okv, 64)


class SampledCase:
    """A full-size workload: the GPU steps every row of the batch (graph
    replay), the oracle only the sampled rows. Sequences are independent
    within a step, so the oracle needs only those rows' tokens, positions,
    tables and cache blocks: its cache is the sampled rows' blocks (and the
    null block) cut out of the initial pool, their tables renumbered."""

    def __init__(self, cfg, seed, ctx, span, sample, ladder):
        self.cfg = cfg
        self.ctx = np.asarray(ctx, np.int32)
        self.B = len(self.ctx)
        self.sample = np.asarray(sample)
        self.model = SynthModel(cfg, seed, device=DEV, cache=False)
        blob = mblob.pack(cfg, self.model.tensors(), device=DEV)
        cap = self.ctx + span
        self.nb = int(sum(-(-int(c) // 16) for c in cap)) + 2
        self.tables = seeded_block_tables(cap, 16, self.nb, seed + 1)
        self.tables[self.tables < 0] = self.nb
        self.eng = Engine(blob, self.nb)
        del blob
        torch.cuda.empty_cache()
        pool0 = random_kv_pool(cfg, self.nb, seed + 2, device=DEV)
        self.eng.pool().copy_(pool0.view(torch.uint8).reshape(-1))
        used = sorted({int(x) for x in self.tables[self.sample].ravel()} - {self.nb})
        self.blocks = np.array(used + [self.nb])         # oracle block i = pool block blocks[i]
        remap = {b: i for i, b in enumerate(self.blocks.tolist())}
        self.otables = np.vectorize(remap.get)(self.tables[self.sample]).astype(np.int32)
        self.idx = torch.tensor(self.blocks, device=DEV)
        self.pool0 = kv_numpy(pool0.index_select(2, self.idx))
        del pool0
        torch.cuda.empty_cache()
        L = cfg.n_layers
        self.okv = OracleKV(self.pool0.copy(), np.ones(L), np.ones(L))
        self.eng.capture(ladder, max_blocks_per_seq=self.tables.shape[1])
        assert self.eng.stats(self.B)[1]
        self.bt_dev = torch.tensor(self.tables, device=DEV)
        self.W = lambda n, l: {k: raw_numpy(v) for k, v in self.model.get(n, l).items()}
        self.mask = np.zeros(self.pool0.shape[2:5], bool)
        self.worst = 0.0

    def step(self, pos, tok):
        cfg, B = self.cfg, self.B
        lg = torch.zeros((B, cfg.vocab), device=DEV)
        ids = torch.full((B,), -1, dtype=torch.int32, device=DEV)
        self.eng.step(torch.tensor(tok, device=DEV), torch.tensor(pos, device=DEV), self.bt_dev,
                      torch.tensor(pos + 1, device=DEV), ids, lg)
        torch.cuda.synchronize()
        sm = self.sample
        ids = ids.cpu().numpy()[sm]
        lg = lg[torch.tensor(sm, device=DEV)].double().cpu().numpy()
        res = decode_step(self.W, cfg, self.okv, tok[sm], pos[sm], self.otables, pos[sm] + 1)
        self.worst = max(self.worst, _check_step(cfg, ids, lg, res))
        for i, p in enumerate(pos[sm]):
            self.mask[self.otables[i][p // 16], :, p % 16] = True

    def finish(self):
        assert self.eng.errors() == 0
        cfg = self.cfg
        dt = torch.uint8 if cfg.kv_dtype == "fp8" else torch.int16
        shape = (cfg.n_layers, 2, self.nb + 1, cfg.n_kv_heads, 16, cfg.head_dim)
        gp = kv_numpy(self.eng.pool(dt).view(shape).index_select(2, self.idx))
        check_cache(gp, self.pool0, self.okv.raw, self.mask, cfg.kv_dtype, skip_null_block=len(self.blocks) - 1)
        return self.worst


def _sampled(wl_key, B, steps, n_sample, gap=1, seed_off=0):
    """Workload `wl_key` at batch B: contexts drawn from its range, `steps`
    decode steps `gap` positions apart (random tokens each step), the oracle
    on n_sample seeded rows (first and last included)."""
    wl = WORKLOADS[wl_key]
    seed = wl.seed + seed_off
    ctx = random_contexts(B, wl.context[0], wl.context[1], seed + 2000)
    if n_sample >= B:
        sample = list(range(B))
    else:
        mid = np.random.default_rng(seed).choice(np.arange(1, B - 1), size=n_sample - 2, replace=False)
        sample = sorted([0, B - 1] + mid.tolist())
    span = (steps - 1) * gap + 1
    case = SampledCase(wl.model, seed, ctx, span, sample, [B])
    try:
        toks = random_tokens(B * steps, wl.model.vocab, seed + 1000).reshape(steps, B)
        for t in range(steps):
            case.step(ctx + t * gap, toks[t])
        return case.finish()
    finally:
        case.eng.close()                  # a failed check must not leave ~100 GB on the device
        torch.cuda.empty_cache()


def test_8b_full_size_batch1(cuda_lib):
    """8B-class BF16, batch 1, context from [256, 2048], eight steps spread
    over 128 positions (18 apart: the slots between keep their cache values
    on both sides)."""
    _sampled("8b", 1, 8, 1, gap=18)


@pytest.mark.parametrize("B", [16, 64])
def test_8b_full_size_batched(cuda_lib, B):
    """8B-class BF16 at batch 16 and 64 (the tensor-core path), contexts from
    [256, 2048], four steps, eight sampled rows."""
    _sampled("8b", B, 4, 8)


def test_32b_fp8_full_size_batch32(cuda_lib):
    """32B-class FP8 (e4m3 weights with per-channel scales, FP8 cache, 40 q /
    8 kv heads of 128), batch 32, 64-256 token contexts, four steps, four
    sampled rows."""
    _sampled("32b_fp8", 32, 4, 4)


@pytest.mark.slow
def test_70b_fp8_full_size_batch1(cuda_lib):
    """70B-class FP8, batch 1, context 2048, two steps (the oracle streams the
    ~70 GB of e4m3 weights through float64 once per step)."""
    _sampled("70b_fp8", 1, 2, 1)


@pytest.mark.slow
def test_70b_fp8_full_size_batch64(cuda_lib):
    """70B-class FP8, batch 64 (the e4m3 tensor-core path), context 2048, four
    steps, four sampled rows."""
    _sampled("70b_fp8", 64, 4, 4)


def test_host_detected_errors(cuda_lib):
    cfg = SMALL
    case = Case(cfg, 3, 2, [5, 9], 1)
    m, kv = case.eng.model, case.eng.kv
    d = torch.zeros(4, dtype=torch.int32, device=DEV)
    bt = case.bt_dev
    assert capi.decode_step_raw(m, kv, 0, d, d, bt, bt.shape[1], d, d) == -2        # MBT_ERR_BATCH
    assert capi.decode_step_raw(m, kv, 2, None, d, bt, bt.shape[1], d, d) == -1     # MBT_ERR_BAD_ARG
    assert capi.decode_step_raw(m, kv, 2, d, d, bt, 0, d, d) == -1
    assert capi.decode_step_raw(m, None, 2, d, d, bt, bt.shape[1], d, d) == -1
    assert capi.status_string(-2) == "batch size must be >= 1"


def test_device_detected_errors(cuda_lib):
    cfg = SMALL
    case = Case(cfg, 4, 2, [5, 9], 1)
    bt = case.bt_dev
    ids = torch.zeros(2, dtype=torch.int32, device=DEV)
    ok_pos = torch.tensor([5, 9], dtype=torch.int32, device=DEV)
    # token out of range
    case.eng.step(torch.tensor([cfg.vocab, 1], dtype=torch.int32, device=DEV), ok_pos, bt,
                  ok_pos + 1, ids)
    assert case.eng.errors() & capi.DEV_TOKEN_RANGE
    # seq_len beyond the block table
    case.eng.step(torch.tensor([1, 1], dtype=torch.int32, device=DEV), ok_pos, bt,
                  torch.tensor([6, 10 ** 6], dtype=torch.int32, device=DEV), ids)
    assert case.eng.errors() & capi.DEV_SEQLEN_RANGE
    # block id out of range: nothing written
    before = case.gpu_pool().copy()
    bad = bt.clone()
    bad[:, :] = case.nb + 7
    case.eng.step(torch.tensor([1, 1], dtype=torch.int32, device=DEV), ok_pos, bad, ok_pos + 1, ids)
    assert case.eng.errors() & capi.DEV_BLOCK_RANGE
    assert np.array_equal(before, case.gpu_pool())
    assert case.eng.errors() == 0
