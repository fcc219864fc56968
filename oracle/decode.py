"""One decode step of a dense Llama-style decoder with a paged KV cache, written
as its plain definition in float64.

Test infrastructure only (see the package docstring).

What the step computes is fixed by the pages as follows; kernel fusion and CUDA
graphs "change how the math executes, not what it computes" ("Kernel Fusion for
Large-Scale LLM Inference", section 11, closing remark), so the oracle runs the
unfused sequence one operation at a time:

* per layer: norm, QKV projection, rotary embedding, paged attention, O
  projection, norm, gate/up projection, activation, down projection, with
  residual adds ("CUDA graphs & kernel fusion", "Direct answer": the per-layer
  list of norms, QKV/O projections, attention, gate/up/down, activations and
  residual adds; "Kernels, Fusion & CUDA Graphs", "Fix 1: kernel fusion" table);
* RMSNorm, RoPE and SwiGLU by the definitions of the works that "Kernel Fusion
  for Large-Scale LLM Inference" lists as references 9, 8 and 7;
* grouped-query attention over a paged cache of fixed-size blocks ("GPU
  Inference Internals", "The KV-Cache Ledger"; "Kernel Fusion for Large-Scale
  LLM Inference", section 11, "Continuous batching + PagedAttention");
* FP8 weights are e4m3 codes times one scale per output channel, dequantised
  before the multiply ("Kernel Fusion for Large-Scale LLM Inference",
  section 11, "Epilogue and dequant fusion");
* greedy sampling: the next token is the arg-max of the logits ("Kernels,
  Fusion & CUDA Graphs", "The serving engine's kernel stack" and the
  "Sampling" row of the fusion table).

Readings where the pages are silent (each is listed with its reason in the
design notes): rotate-half RoPE pairing (i, i + d/2) with angle
p * theta^(-2i/d); RMSNorm x / sqrt(mean(x^2) + eps) * gamma; SiLU(x) = x *
sigmoid(x) with the gate rows first in the fused gate/up matrix; attention
scale 1/sqrt(d) with no mask beyond seq_len; new K/V are written to the cache
(rounded to the cache format) before the step attends over seq_len tokens;
lowest index wins an exact arg-max tie.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Callable, Dict, Optional

import numpy as np

from .numerics import bf16_decode, e4m3_decode, round_bf16, round_e4m3

__all__ = ["rmsnorm", "rope", "silu", "swiglu", "decode_weight", "matmul",
           "OracleKV", "paged_attention", "decode_step", "StepResult", "prefill"]


# ---------------------------------------------------------------------------
# elementwise definitions

def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm ("Root Mean Square Layer Normalization", reference 9 of "Kernel
    Fusion for Large-Scale LLM Inference"): x / sqrt(mean(x^2) + eps) * gamma,
    over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * gamma


def rope(x: np.ndarray, pos: int, theta: float) -> np.ndarray:
    """Rotary position embedding ("RoFormer", reference 8 of "Kernel Fusion for
    Large-Scale LLM Inference") of the last axis (length d) at position `pos`.

    Pair i (i < d/2) is (x[i], x[i + d/2]) and is rotated by the angle
    pos * theta^(-2i/d)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    i = np.arange(half, dtype=np.float64)
    ang = float(pos) * theta ** (-2.0 * i / d)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    """SiLU(x) = x * sigmoid(x) = x / (1 + e^-x)."""
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def swiglu(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """SwiGLU activation ("GLU Variants Improve Transformer", reference 7 of
    "Kernel Fusion for Large-Scale LLM Inference"): SiLU(gate) * up."""
    return silu(gate) * np.asarray(up, dtype=np.float64)


# ---------------------------------------------------------------------------
# weights

WeightSource = Callable[[str, int], Dict[str, np.ndarray]]


def decode_weight(t: Dict[str, np.ndarray], rows: Optional[slice] = None) -> np.ndarray:
    """Raw stored weight -> float64 matrix. BF16 (uint16 bits) decodes exactly;
    FP8 is e4m3(code) * scale[row]."""
    w = t["w"] if rows is None else t["w"][rows]
    if w.dtype == np.uint16:
        return bf16_decode(w)
    if w.dtype == np.uint8:
        s = t["s"] if rows is None else t["s"][rows]
        return e4m3_decode(w) * np.asarray(s, dtype=np.float64)[:, None]
    raise TypeError(f"unsupported weight storage {w.dtype}")


_THREADS = max(1, os.cpu_count() or 1)


def matmul(t: Dict[str, np.ndarray], x: np.ndarray, chunk_bytes: int = 1 << 24) -> np.ndarray:
    """y[b, n] = sum_k W[n, k] x[b, k] in float64 (W decoded row chunk by row chunk
    so that large matrices never exist whole in float64).

    Each output element is one float64 dot product over k; the pages fix no
    summation order. For a few input rows (decode batches) the row chunks are
    independent and run on a thread pool, each decoded and multiplied with
    NumPy's own loops (einsum, no BLAS, so the threads do not oversubscribe the
    cores); larger inputs use one BLAS product per chunk."""
    n, k = t["w"].shape
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    out = np.empty((x.shape[0], n), dtype=np.float64)
    step = max(1, chunk_bytes // (8 * k))
    starts = range(0, n, step)
    if x.shape[0] > 16 or _THREADS == 1 or len(starts) == 1:
        for r0 in starts:
            r1 = min(n, r0 + step)
            out[:, r0:r1] = x @ decode_weight(t, slice(r0, r1)).T
        return out

    def chunk(r0):
        r1 = min(n, r0 + step)
        out[:, r0:r1] = np.einsum("bk,nk->bn", x, decode_weight(t, slice(r0, r1)))

    with ThreadPoolExecutor(min(_THREADS, len(starts))) as ex:
        list(ex.map(chunk, starts))
    return out


# ---------------------------------------------------------------------------
# paged KV cache

@dataclasses.dataclass
class OracleKV:
    """The oracle's own copy of the paged cache.

    raw: [layers][2 (K, V)][num_blocks + 1][kv_heads][block][head_dim] storage,
    uint16 BF16 bits or uint8 e4m3 codes; block `num_blocks` is the reserved
    null block. Stored value = format(x / scale) with one fp32 scale per layer
    for K and for V (1.0 for BF16 caches)."""
    raw: np.ndarray
    k_scale: np.ndarray
    v_scale: np.ndarray

    @property
    def fp8(self) -> bool:
        return self.raw.dtype == np.uint8

    @property
    def num_blocks(self) -> int:
        return self.raw.shape[2] - 1

    @property
    def block_size(self) -> int:
        return self.raw.shape[4]

    def decode(self, layer: int, which: int, blocks: np.ndarray) -> np.ndarray:
        """Decoded values of whole blocks: [len(blocks)][kv_heads][block][d]."""
        r = self.raw[layer, which, blocks]
        v = e4m3_decode(r) if self.fp8 else bf16_decode(r)
        scale = (self.k_scale if which == 0 else self.v_scale)[layer]
        return v * np.float64(scale)

    def store(self, layer: int, which: int, block: int, slot: int, x: np.ndarray) -> None:
        """Round x[kv_heads][d] / scale to the cache format and store it."""
        scale = np.float64((self.k_scale if which == 0 else self.v_scale)[layer])
        y = np.asarray(x, dtype=np.float64) / scale
        self.raw[layer, which, block, :, slot, :] = round_e4m3(y) if self.fp8 else round_bf16(y)


def slot_of(block_table: np.ndarray, pos: int, block_size: int):
    """Physical (block id, slot) of logical token `pos` of a sequence."""
    return int(block_table[pos // block_size]), pos % block_size


def paged_attention(q: np.ndarray, kv: OracleKV, layer: int, block_table: np.ndarray,
                    seq_len: int) -> np.ndarray:
    """softmax(q_h . K_t / sqrt(d)) . V over tokens t < seq_len of one sequence.

    q: [nq][d]. Query head h reads KV head h // (nq / nkv) (grouped-query
    attention). K_t, V_t are gathered through the block table: token t lives in
    block block_table[t // block] at slot t % block."""
    nq, d = q.shape
    bs = kv.block_size
    nblk = -(-seq_len // bs)
    blocks = np.asarray(block_table[:nblk], dtype=np.int64)
    kd = kv.decode(layer, 0, blocks)                       # [nblk][nkv][bs][d]
    vd = kv.decode(layer, 1, blocks)
    nkv = kd.shape[1]
    K = kd.transpose(1, 0, 2, 3).reshape(nkv, nblk * bs, d)[:, :seq_len]
    V = vd.transpose(1, 0, 2, 3).reshape(nkv, nblk * bs, d)[:, :seq_len]
    group = nq // nkv
    out = np.empty((nq, d), dtype=np.float64)
    for h in range(nq):
        g = h // group
        s = K[g] @ q[h] / np.sqrt(d)
        p = np.exp(s - s.max())
        p /= p.sum()
        out[h] = p @ V[g]
    return out


# ---------------------------------------------------------------------------
# the step

@dataclasses.dataclass
class StepResult:
    logits: np.ndarray          # [B][V] float64
    next_ids: np.ndarray        # [B] int64
    flops: int                  # multiply-adds x 2 actually performed
    matmul_flops: int
    attn_flops: int


def _check_inputs(cfg, kv: OracleKV, tokens, positions, block_tables, seq_lens):
    bs = cfg.block_size
    for b in range(len(tokens)):
        if not (0 <= tokens[b] < cfg.vocab):
            raise ValueError("token id out of range")
        p, s = int(positions[b]), int(seq_lens[b])
        if not (0 <= p < cfg.max_pos) or not (1 <= s <= cfg.max_pos) or p >= s:
            raise ValueError("position / seq_len out of range")
        nblk = -(-s // bs)
        if nblk > block_tables.shape[1]:
            raise ValueError("seq_len beyond the block table")
        blk = block_tables[b, :nblk]
        if np.any(blk < 0) or np.any(blk > kv.num_blocks):
            raise ValueError("block id out of range")


def decode_step(weights: WeightSource, cfg, kv: OracleKV, tokens, positions, block_tables,
                seq_lens, layers: Optional[range] = None) -> StepResult:
    """One decode step for B sequences.

    Row b embeds token tokens[b] at position positions[b], writes its K and V
    into the slot of that position, attends over its first seq_lens[b] tokens
    (the written one included) and returns its next-token logits and arg-max.
    `kv` is updated in place. `layers` restricts the layers run (used only to
    time a bounded sample of a large model).
    """
    tokens = np.asarray(tokens, dtype=np.int64)
    positions = np.asarray(positions, dtype=np.int64)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    block_tables = np.asarray(block_tables, dtype=np.int64)
    _check_inputs(cfg, kv, tokens, positions, block_tables, seq_lens)
    B = len(tokens)
    H, d, nq, nkv = cfg.hidden, cfg.head_dim, cfg.n_q_heads, cfg.n_kv_heads
    F = cfg.ffn
    mm = 0
    at = 0

    emb = weights("embed", -1)
    r = bf16_decode(emb["w"][tokens])                        # [B][H]

    for l in (layers if layers is not None else range(cfg.n_layers)):
        g_attn = bf16_decode(weights("g_attn", l)["w"])
        g_ffn = bf16_decode(weights("g_ffn", l)["w"])

        y = rmsnorm(r, g_attn, cfg.eps)
        qkv = matmul(weights("w_qkv", l), y)
        mm += 2 * B * cfg.qkv_rows * H
        q = qkv[:, : nq * d].reshape(B, nq, d)
        k = qkv[:, nq * d: (nq + nkv) * d].reshape(B, nkv, d)
        v = qkv[:, (nq + nkv) * d:].reshape(B, nkv, d)

        o = np.empty((B, nq, d), dtype=np.float64)
        for b in range(B):
            p = int(positions[b])
            qb = rope(q[b], p, cfg.rope_theta)
            kb = rope(k[b], p, cfg.rope_theta)
            blk, slot = slot_of(block_tables[b], p, cfg.block_size)
            kv.store(l, 0, blk, slot, kb)
            kv.store(l, 1, blk, slot, v[b])
            o[b] = paged_attention(qb, kv, l, block_tables[b], int(seq_lens[b]))
            at += 2 * 2 * nq * int(seq_lens[b]) * d

        r = r + matmul(weights("w_o", l), o.reshape(B, nq * d))
        mm += 2 * B * H * nq * d

        y = rmsnorm(r, g_ffn, cfg.eps)
        gu = matmul(weights("w_gu", l), y)
        mm += 2 * B * 2 * F * H
        a = swiglu(gu[:, :F], gu[:, F:])
        r = r + matmul(weights("w_down", l), a)
        mm += 2 * B * H * F

    y = rmsnorm(r, bf16_decode(weights("g_final", -1)["w"]), cfg.eps)
    logits = matmul(weights("lm_head", -1), y)
    mm += 2 * B * cfg.vocab * H
    ids = np.argmax(logits, axis=1)                           # first maximum on ties
    return StepResult(logits, ids, mm + at, mm, at)


def prefill(weights: WeightSource, cfg, kv: OracleKV, tokens, start_pos: int, block_table) -> StepResult:
    """Ingest the prompt tokens of one sequence at positions start_pos,
    start_pos + 1, ... ("GPU Inference Internals", "Roofline: Why Decode Is
    Memory-Bound": prefill runs the whole prompt through the model at once;
    what it computes is the same as feeding the prompt one token at a time).

    Every prompt token is one row of a decode step over the sequence's block
    table, at its own position and attending over position + 1 tokens. Within
    each layer decode_step takes the rows in order and writes a row's K and V
    before that row attends, so row i sees exactly the prompt positions up to
    its own: causal attention. The last row's logits and arg-max are the
    prompt's next token; `kv` holds every prompt token's K and V."""
    tokens = np.asarray(tokens, dtype=np.int64)
    n = len(tokens)
    pos = int(start_pos) + np.arange(n, dtype=np.int64)
    tables = np.repeat(np.asarray(block_table, dtype=np.int64)[None, :], n, axis=0)
    return decode_step(weights, cfg, kv, tokens, pos, tables, pos + 1)
