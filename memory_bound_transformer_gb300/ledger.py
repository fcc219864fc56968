"""Byte and FLOP ledger of a decode step, the roofline terms the benchmark
reports against.

* Machine balance = peak compute / memory bandwidth ("GPU Inference
  Internals", "The Hardware Ledger").
* A forward pass is about 2 x P FLOPs per token; batch-1 decode reads every
  weight once, so the single-stream ceiling is bandwidth / weight bytes
  ("GPU Inference Internals", "Roofline: Why Decode Is Memory-Bound").
* KV bytes per token = 2 (K and V) x layers x kv_heads x head_dim x bytes
  ("GPU Inference Internals", "The KV-Cache Ledger").
* Step bytes D = W + B S K (+ activations), step FLOPs F = 2 P B ("GPU Inference
  Internals", "Batching Economics").
* Launch tax: T_eager = T_compute + N tau, T_graph = T_compute + tau ("CUDA
  graphs & kernel fusion", "Direct answer").
"""
from __future__ import annotations

from typing import Sequence, Tuple


def machine_balance(peak_flops: float, bandwidth: float) -> float:
    return peak_flops / bandwidth


def single_stream_ceiling(bandwidth: float, bytes_per_token: float) -> float:
    """Upper bound on tokens/s for one sequence: every weight byte read once per token."""
    return bandwidth / bytes_per_token


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, bytes_per_elem: int) -> int:
    return 2 * layers * kv_heads * head_dim * bytes_per_elem


def weight_intensity(batch: int, bytes_per_weight: float) -> float:
    """Weight-only arithmetic intensity of decode at batch B: 2B / b_w FLOP per byte."""
    return 2.0 * batch / bytes_per_weight


def launch_tax(weight_gib: float, n_kernels: int = 430, tau_us: float = 5.0,
               bandwidth: float = 1e12) -> Tuple[float, float, float, float]:
    """(compute, eager, graph) milliseconds and eager/graph for a step that
    streams `weight_gib` GiB at `bandwidth` bytes/s and launches n_kernels."""
    compute = weight_gib * (1 << 30) / bandwidth * 1e3
    eager = compute + n_kernels * tau_us * 1e-3
    graph = compute + tau_us * 1e-3
    return compute, eager, graph, eager / graph


def weight_bytes(cfg) -> int:
    """Bytes of every tensor one decode step reads in full: all projection
    matrices (with FP8 scales), the LM head and the norm gains. The embedding
    table is excluded (a step reads only B of its rows)."""
    w = 1 if cfg.weight_dtype == "fp8" else 2
    H, F, V = cfg.hidden, cfg.ffn, cfg.vocab
    per_layer_rows = cfg.qkv_rows + H + 2 * F + H                    # qkv, o, gate+up, down
    per_layer = (cfg.qkv_rows * H + H * cfg.q_dim + 2 * F * H + H * F) * w + 2 * H * 2
    scales = (cfg.n_layers * per_layer_rows + V) * 4 if cfg.weight_dtype == "fp8" else 0
    return cfg.n_layers * per_layer + V * H * w + H * 2 + scales


def matmul_params(cfg) -> int:
    H, F, V = cfg.hidden, cfg.ffn, cfg.vocab
    return cfg.n_layers * (cfg.qkv_rows * H + H * cfg.q_dim + 3 * F * H) + V * H


def kv_read_bytes(cfg, seq_lens: Sequence[int]) -> int:
    """KV bytes one step reads: every row reads K and V of its seq_len tokens in every layer."""
    k = 1 if cfg.kv_dtype == "fp8" else 2
    return sum(int(s) for s in seq_lens) * kv_bytes_per_token(cfg.n_layers, cfg.n_kv_heads, cfg.head_dim, k)


def step_bytes(cfg, seq_lens: Sequence[int]) -> int:
    """Algorithmic bytes of one decode step: weights once + the KV read term
    (activations and the new K/V writes are below 0.1 % and left out)."""
    return weight_bytes(cfg) + kv_read_bytes(cfg, seq_lens)


def step_flops(cfg, seq_lens: Sequence[int]) -> int:
    attn = sum(4 * cfg.n_q_heads * cfg.head_dim * int(s) for s in seq_lens) * cfg.n_layers
    return 2 * matmul_params(cfg) * len(seq_lens) + attn
