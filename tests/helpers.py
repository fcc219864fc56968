"""Shared test plumbing: weight-source adapters and small model shapes."""
import numpy as np
import torch

from synth import ModelConfig, SynthModel, raw_numpy, random_kv_pool, seeded_block_tables

# Small shapes that still span several kernel tiles and leave ragged tails.
MICRO = ModelConfig("micro", 2, 64, 4, 2, 16, 96, 128, max_pos=64)
MICRO_FP8 = MICRO.replace(name="micro-fp8", weight_dtype="fp8", kv_dtype="fp8")
SMALL = ModelConfig("small", 2, 384, 6, 2, 64, 1040, 2000, max_pos=512)
SMALL_FP8 = SMALL.replace(name="small-fp8", weight_dtype="fp8", kv_dtype="fp8")
SMALL_D128 = ModelConfig("small-d128", 2, 512, 8, 2, 128, 1376, 3001, max_pos=1024)
SMALL_G5 = ModelConfig("small-g5", 1, 640, 10, 2, 64, 704, 1500, max_pos=512,
                       weight_dtype="fp8", kv_dtype="fp8")


def oracle_weights(model: SynthModel):
    """Adapter: synthetic model -> the oracle's weight source (raw numpy arrays)."""
    cache = {}

    def get(name, layer):
        key = (name, layer)
        if key not in cache:
            t = model.get(name, layer)
            cache[key] = {k: raw_numpy(v) for k, v in t.items()}
        return cache[key]
    return get


def kv_numpy(pool: torch.Tensor) -> np.ndarray:
    a = pool.cpu().numpy()
    return a.view(np.uint16) if a.dtype == np.int16 else a


def make_case(cfg, batch, ctx_lo, ctx_hi, seed, slack_blocks=3, device="cpu"):
    """Random context lengths, non-contiguous block tables and a random pool.
    Returns dict with contexts (tokens already cached), tables, pool, num_blocks."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(ctx_lo, ctx_hi + 1, size=batch).astype(np.int32)
    cap = ctx + 1
    nblk = int(sum(-(-int(c) // cfg.block_size) for c in cap)) + slack_blocks
    tables = seeded_block_tables(cap, cfg.block_size, nblk, seed + 1)
    pool = random_kv_pool(cfg, nblk, seed + 2, device=device)
    return dict(ctx=ctx, tables=tables, pool=pool, num_blocks=nblk)
