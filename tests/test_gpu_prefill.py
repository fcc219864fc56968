"""Prefill (prompt ingestion) through the C ABI against the oracle.

The oracle's prefill is the prompt fed as rows of one decode step, each row
writing its K and V before it attends (pinned on the CPU against feeding the
prompt one token at a time). Acceptance is the decode step's: the last token's
logits within 3e-2 (BF16) / 1.5e-1 (FP8) of the oracle's, its arg-max equal
where the oracle's top-2 margin exceeds 1e-2, every prompt position's K and V
within the decode tests' bound of the oracle's (one step of the cache grid plus
a third of the logit tolerance relative to the row's magnitude), and every
other cache byte unchanged. Prompt lengths cover one pass (1, 15, 16, 17 tokens), several
128-token passes with a ragged tail on the CUDA cores (130) or on the tensor
cores (300), and a prompt continued from a later start position."""
import numpy as np
import pytest
import torch

from memory_bound_transformer_gb300 import blob as mblob
from memory_bound_transformer_gb300 import capi
from memory_bound_transformer_gb300.engine import Engine
from oracle.decode import OracleKV, prefill
from synth import ONE_B, SynthModel, random_kv_pool, random_tokens, raw_numpy
from tests.helpers import SMALL, SMALL_D128, SMALL_FP8, SMALL_G5, kv_numpy, oracle_weights
from tests.test_gpu_step import check_cache, parity_log, tol_logits

pytestmark = pytest.mark.gpu
DEV = "cuda"


class PrefillCase:
    def __init__(self, cfg, seed, span, cache_weights=True):
        self.cfg = cfg
        self.model = SynthModel(cfg, seed, device=DEV, cache=cache_weights)
        blob = mblob.pack(cfg, self.model.tensors(), device=DEV)
        self.nblk = -(-span // 16)
        self.nb = self.nblk + 5
        self.table = np.random.default_rng(seed).permutation(self.nb)[:self.nblk].astype(np.int32)
        self.eng = Engine(blob, self.nb)
        del blob
        pool0 = random_kv_pool(cfg, self.nb, seed + 2, device=DEV)
        self.eng.pool().copy_(pool0.view(torch.uint8).reshape(-1))
        self.pool0 = kv_numpy(pool0)
        del pool0
        torch.cuda.empty_cache()
        L = cfg.n_layers
        self.okv = OracleKV(self.pool0.copy(), np.ones(L), np.ones(L))
        self.written = np.zeros(self.pool0.shape[2:5], bool)

    def gpu_pool(self):
        raw = self.eng.pool().cpu().numpy()
        dt = np.uint8 if self.cfg.kv_dtype == "fp8" else np.uint16
        return raw.view(dt).reshape(self.pool0.shape)

    def run(self, toks, start, W):
        cfg = self.cfg
        nid = torch.full((1,), -1, dtype=torch.int32, device=DEV)
        lg = torch.zeros(cfg.vocab, device=DEV)
        self.eng.prefill(torch.tensor(toks, device=DEV), start, torch.tensor(self.table, device=DEV), nid, lg)
        torch.cuda.synchronize()
        res = prefill(W, cfg, self.okv, toks, start, self.table)
        got = lg.double().cpu().numpy()
        err = np.abs(got - res.logits[-1]).max()
        parity_log("max_logit_err", float(err))
        assert err <= tol_logits(cfg), f"max logit error {err}"
        srt = np.sort(res.logits[-1])
        if srt[-1] - srt[-2] > 1e-2:
            assert int(nid.item()) == int(res.next_ids[-1])
        assert int(nid.item()) == int(np.argmax(got))
        for p in range(start, start + len(toks)):
            self.written[self.table[p // 16], :, p % 16] = True
        return err

    def check(self, graphs=False):
        assert self.eng.errors() == 0
        # a graph capture's warm-up runs padding rows, which write the null block
        check_cache(self.gpu_pool(), self.pool0, self.okv.raw, self.written, self.cfg.kv_dtype,
                    skip_null_block=self.nb if graphs else None)


@pytest.mark.parametrize("cfg", [SMALL, SMALL_FP8, SMALL_D128, SMALL_G5], ids=lambda c: c.name)
@pytest.mark.parametrize("n", [1, 15, 16, 17, 130, 300])
def test_prefill_small(cuda_lib, cfg, n):
    case = PrefillCase(cfg, 40 + n, n + 1)
    toks = random_tokens(n, cfg.vocab, n)
    case.run(toks, 0, oracle_weights(case.model))
    case.check()


@pytest.mark.parametrize("cfg", [SMALL, SMALL_FP8], ids=lambda c: c.name)
def test_prefill_continues_and_decode_follows(cuda_lib, cfg):
    """A prompt in two calls (positions 0..69, then 70..219): the second
    attends over the first's cache; then decode steps at 220, 221 read it."""
    case = PrefillCase(cfg, 7, 240)
    W = oracle_weights(case.model)
    toks = random_tokens(222, cfg.vocab, 3)
    case.run(toks[:70], 0, W)
    case.run(toks[70:220], 70, W)
    from oracle.decode import decode_step
    from tests.test_gpu_step import _check_step
    bt = torch.tensor(case.table[None, :], device=DEV)
    for p in (220, 221):
        ids = torch.full((1,), -1, dtype=torch.int32, device=DEV)
        lg = torch.zeros((1, cfg.vocab), device=DEV)
        pos = torch.tensor([p], dtype=torch.int32, device=DEV)
        case.eng.step(torch.tensor(toks[p:p + 1], device=DEV), pos, bt, pos + 1, ids, lg)
        torch.cuda.synchronize()
        res = decode_step(W, cfg, case.okv, toks[p:p + 1], [p], case.table[None, :], [p + 1])
        _check_step(cfg, ids.cpu().numpy(), lg.double().cpu().numpy(), res)
        case.written[case.table[p // 16], :, p % 16] = True
    case.check()


def test_prefill_keeps_graphs(cuda_lib):
    """Prefill runs eagerly beside captured graphs without invalidating them."""
    cfg = SMALL
    case = PrefillCase(cfg, 9, 200)
    case.eng.capture([1, 2, 4], max_blocks_per_seq=4)
    case.run(random_tokens(150, cfg.vocab, 1), 0, oracle_weights(case.model))
    assert case.eng.stats(1)[1] and case.eng.stats(4)[1]
    case.check(graphs=True)


def test_prefill_1b_prompt512(cuda_lib):
    """The 1B-class workload's prompt: 512 random tokens (four tensor-core passes)."""
    cfg = ONE_B
    case = PrefillCase(cfg, 1236, 513)
    case.run(random_tokens(512, cfg.vocab, 1236 + 1000), 0, oracle_weights(case.model))
    case.check()


@pytest.mark.slow
def test_prefill_8b_prompt300(cuda_lib):
    """8B-class BF16, a 300-token prompt (two full passes and a ragged one)."""
    from synth import EIGHT_B
    cfg = EIGHT_B
    case = PrefillCase(cfg, 1237, 301, cache_weights=False)
    W = lambda n, l: {k: raw_numpy(v) for k, v in case.model.get(n, l).items()}
    try:
        case.run(random_tokens(300, cfg.vocab, 77), 0, W)
        case.check()
    finally:
        case.eng.close()


def test_prefill_host_detected_errors(cuda_lib):
    cfg = SMALL
    case = PrefillCase(cfg, 3, 40)
    m, kv = case.eng.model, case.eng.kv
    t = torch.zeros(64, dtype=torch.int32, device=DEV)
    bt = torch.tensor(case.table, device=DEV)
    nid = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert capi.prefill_raw(m, kv, 0, t, 0, bt, bt.numel(), nid) == -2            # MBT_ERR_BATCH
    assert capi.prefill_raw(m, kv, 8, None, 0, bt, bt.numel(), nid) == -1          # MBT_ERR_BAD_ARG
    assert capi.prefill_raw(m, kv, 8, t, -1, bt, bt.numel(), nid) == -1
    assert capi.prefill_raw(m, kv, 8, t, cfg.max_pos - 4, bt, bt.numel(), nid) == -1   # beyond max_pos
    assert capi.prefill_raw(m, kv, 60, t, 0, bt, 3, nid) == -1                     # beyond the table
    assert case.eng.errors() == 0
