"""Seeded synthetic inputs shared by the oracle and the CUDA path.

This module holds no arithmetic of the decode step. It only draws random
numbers and lays them out:

* model shapes for the five workloads (tiny layer, 1B, 8B, 32B FP8, 70B FP8),
* random-init weights, N(0, 0.02) as the workloads state, rounded to BF16 or
  quantised to FP8-e4m3 with one fp32 scale per output channel (the weight
  artifact the decode step reads; FP8 weights with per-channel scales follow
  "Kernel Fusion for Large-Scale LLM Inference", section 11, "Epilogue and
  dequant fusion" and "FP8 weights and KV cache"),
* random KV-cache contents, token ids, positions, block tables, seq lens.

Everything is produced with torch generators so that large models can be
generated directly on a GPU. Each tensor has its own generator seed, so any
single tensor can be regenerated on demand and yields the same bytes on the
same device.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

__all__ = [
    "ModelConfig", "Workload", "WORKLOADS", "TINY", "ONE_B", "EIGHT_B",
    "THIRTYTWO_B_FP8", "SEVENTY_B_FP8", "matmul_names", "tensor_shape",
    "gen_tensor", "SynthModel", "random_kv_pool", "seeded_block_tables",
    "raw_numpy",
]


@dataclasses.dataclass(frozen=True)
class ModelConfig:
    """Shape of a dense Llama-style decoder."""
    name: str
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    weight_dtype: str = "bf16"   # "bf16" or "fp8" (e4m3 + fp32 per-row scale)
    kv_dtype: str = "bf16"       # "bf16" or "fp8" (e4m3, per-layer fp32 scale)
    eps: float = 1e-6
    rope_theta: float = 10000.0
    block_size: int = 16
    max_pos: int = 4096

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    def replace(self, **kw) -> "ModelConfig":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One benchmarked configuration: a model plus its batch/context recipe."""
    key: str
    model: ModelConfig
    batches: Tuple[int, ...]
    context: Tuple[int, int]       # initial context length range [lo, hi]
    steps: int                     # decode steps
    ladder: Tuple[int, ...]        # CUDA-graph batch ladder to capture
    seed: int                      # weights seed; tokens use seed+1000, contexts seed+2000
    description: str


TINY = ModelConfig("tiny-layer", 1, 256, 4, 2, 64, 688, 1024, max_pos=512)
ONE_B = ModelConfig("1B-class", 16, 2048, 32, 8, 64, 8192, 32000, max_pos=1024)
EIGHT_B = ModelConfig("8B-class", 32, 4096, 32, 8, 128, 14336, 128256, max_pos=4096)
THIRTYTWO_B_FP8 = ModelConfig("32B-class-fp8", 64, 5120, 40, 8, 128, 27648, 152064,
                              weight_dtype="fp8", kv_dtype="fp8", max_pos=512)
SEVENTY_B_FP8 = ModelConfig("70B-class-fp8", 80, 8192, 64, 8, 128, 28672, 128256,
                            weight_dtype="fp8", kv_dtype="fp8", max_pos=4096)

WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", TINY, (1,), (128, 128), 8, (1,), 1235,
                     "single decoder layer + LM head, batch 1, 128 tokens of random KV, "
                     "8 decode steps from random token ids"),
    "1b": Workload("1b", ONE_B, (1, 8), (512, 512), 64, (1, 2, 4, 8), 1236,
                   "1B-class dense decoder, batch 1 and 8, 512-token context, 64 decode steps"),
    "8b": Workload("8b", EIGHT_B, (1, 16, 64), (256, 2048), 128, (1, 2, 4, 8, 16, 24, 32, 40, 48, 56, 64), 1237,
                   "8B-class dense decoder, batch 1/16/64, per-sequence context uniform in "
                   "[256, 2048], 128 decode steps"),
    "32b_fp8": Workload("32b_fp8", THIRTYTWO_B_FP8, (32,), (64, 256), 40, (32,), 1238,
                        "32B-class FP8 decoder, batch 32, 64-256 token prompts, 40 decode steps"),
    "70b_fp8": Workload("70b_fp8", SEVENTY_B_FP8, (1, 64), (2048, 2048), 64, (1, 2, 4, 8, 16, 24, 32, 40, 48, 56, 64), 1239,
                        "70B-class FP8 decoder, batch 1 and 64, context 2048, 64 decode steps"),
}

# ---------------------------------------------------------------------------
# weight tensors

_MATMULS = ("w_qkv", "w_o", "w_gu", "w_down")
_NORMS = ("g_attn", "g_ffn")


def matmul_names() -> Tuple[str, ...]:
    return _MATMULS


def tensor_shape(cfg: ModelConfig, name: str) -> Tuple[int, ...]:
    """[rows, cols] (row-major, one output channel per row) or [n] for gains."""
    h = cfg.hidden
    return {
        "embed": (cfg.vocab, h),
        "w_qkv": (cfg.qkv_rows, h),            # rows: q heads, then k heads, then v heads
        "w_o": (h, cfg.q_dim),
        "w_gu": (2 * cfg.ffn, h),              # rows: gate (ffn rows), then up (ffn rows)
        "w_down": (h, cfg.ffn),
        "lm_head": (cfg.vocab, h),
        "g_attn": (h,), "g_ffn": (h,), "g_final": (h,),
    }[name]


def _tensor_seed(seed: int, name: str, layer: int) -> int:
    digest = hashlib.sha256(f"{seed}/{name}/{layer}".encode()).digest()
    return int.from_bytes(digest[:8], "little") & ((1 << 62) - 1)


def _randn(shape, seed: int, device) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def gen_tensor(cfg: ModelConfig, seed: int, name: str, layer: int = -1,
               device="cpu") -> Dict[str, torch.Tensor]:
    """Generate one tensor of a random-init model.

    Returns {"w": tensor} where w is bfloat16 for BF16 weights, gains and the
    embedding, or uint8 e4m3 codes for FP8 weights, in which case "s" holds
    the fp32 per-row scale (row amax / 448, so each row uses the full e4m3
    range). Gains are 1 + N(0, 0.1) so that a wrong gain index is visible.
    """
    shape = tensor_shape(cfg, name)
    ts = _tensor_seed(seed, name, layer)
    if name.startswith("g_"):
        w = 1.0 + 0.1 * _randn(shape, ts, device)
        return {"w": w.to(torch.bfloat16)}
    w = 0.02 * _randn(shape, ts, device)
    fp8 = cfg.weight_dtype == "fp8" and name != "embed"
    if not fp8:
        return {"w": w.to(torch.bfloat16)}
    amax = w.abs().amax(dim=1).clamp_min(1e-30)
    s = (amax / 448.0).to(torch.float32)
    q = (w / s[:, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return {"w": q.view(torch.uint8), "s": s}


class SynthModel:
    """Lazy, cached access to the random-init tensors of one model."""

    def __init__(self, cfg: ModelConfig, seed: int, device="cpu", cache: bool = True):
        self.cfg, self.seed, self.device, self.cache = cfg, seed, device, cache
        self._cache: Dict[Tuple[str, int], Dict[str, torch.Tensor]] = {}

    def get(self, name: str, layer: int = -1) -> Dict[str, torch.Tensor]:
        key = (name, layer)
        if key in self._cache:
            return self._cache[key]
        t = gen_tensor(self.cfg, self.seed, name, layer, self.device)
        if self.cache:
            self._cache[key] = t
        return t

    def tensors(self):
        """Yield (name, layer, dict) in blob order."""
        yield "embed", -1, self.get("embed")
        for l in range(self.cfg.n_layers):
            for n in ("g_attn", "w_qkv", "w_o", "g_ffn", "w_gu", "w_down"):
                yield n, l, self.get(n, l)
        yield "g_final", -1, self.get("g_final")
        yield "lm_head", -1, self.get("lm_head")


def raw_numpy(t: torch.Tensor) -> np.ndarray:
    """Raw storage of a tensor as numpy: bf16 -> uint16 bits, uint8 stays, fp32 stays."""
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


# ---------------------------------------------------------------------------
# KV cache, tokens, tables

def random_kv_pool(cfg: ModelConfig, num_blocks: int, seed: int, device="cpu",
                   std: float = 1.0) -> torch.Tensor:
    """Random cache contents: [L][2][num_blocks + 1][nkv][block][d] raw storage.

    The last block is the reserved null block. BF16 caches hold bf16(N(0, std²));
    FP8 caches hold e4m3 codes of N(0, std²) (per-layer scale 1.0). Returned as
    int16 (bf16 bits) or uint8 (e4m3 codes).
    """
    shape = (2, num_blocks + 1, cfg.n_kv_heads, cfg.block_size, cfg.head_dim)
    fp8 = cfg.kv_dtype == "fp8"
    out = torch.empty((cfg.n_layers,) + shape, dtype=torch.uint8 if fp8 else torch.int16, device=device)
    for layer in range(cfg.n_layers):          # one layer at a time: no full-size fp32 temporary
        x = std * _randn(shape, _tensor_seed(seed, "kv", layer), device)
        if fp8:
            out[layer] = x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
        else:
            out[layer] = x.to(torch.bfloat16).view(torch.int16)
        del x
    return out


def seeded_block_tables(seq_capacity: Sequence[int], block_size: int, num_blocks: int,
                        seed: int, stride: Optional[int] = None) -> np.ndarray:
    """Non-contiguous block tables: row b gets ceil(cap_b / block) distinct ids
    drawn from a seeded permutation of [0, num_blocks). Unused entries are -1."""
    need = [-(-c // block_size) for c in seq_capacity]
    if sum(need) > num_blocks:
        raise ValueError("not enough blocks")
    stride = stride or max(need)
    perm = np.random.default_rng(seed).permutation(num_blocks)
    bt = np.full((len(need), stride), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[off:off + n]
        off += n
    return bt


def random_tokens(n: int, vocab: int, seed: int) -> np.ndarray:
    return np.random.default_rng(seed).integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)


def random_contexts(batch: int, lo: int, hi: int, seed: int) -> np.ndarray:
    return np.random.default_rng(seed).integers(lo, hi + 1, size=batch).astype(np.int32)
