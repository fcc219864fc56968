"""Weight/config blob writer for model_create (format: include/mbt.h).

A blob is a header, a tensor table and 256-byte aligned tensor data in one byte
buffer, built here as a torch uint8 tensor on the host or directly on the GPU
(so a 70 GB FP8 model never passes through host memory)."""
from __future__ import annotations

import struct
from typing import Iterable, List, Tuple

import torch

MAGIC = b"MBTBLOB1"
VERSION = 1
HEADER = struct.Struct("<8sI7I4I2f2IQ")      # 80 bytes
ENTRY = struct.Struct("<IiII4Q")             # 48 bytes
assert HEADER.size == 80 and ENTRY.size == 48

DTYPE_BF16, DTYPE_E4M3, DTYPE_F32 = 0, 1, 2
KINDS = {"embed": 0, "g_attn": 1, "w_qkv": 2, "s_qkv": 3, "w_o": 4, "s_o": 5, "g_ffn": 6,
         "w_gu": 7, "s_gu": 8, "w_down": 9, "s_down": 10, "g_final": 11, "lm_head": 12, "s_lm": 13}
_SCALE_OF = {"w_qkv": "s_qkv", "w_o": "s_o", "w_gu": "s_gu", "w_down": "s_down", "lm_head": "s_lm"}


def _align(x: int, a: int = 256) -> int:
    return (x + a - 1) // a * a


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype in (torch.bfloat16, torch.int16):
        return DTYPE_BF16
    if t.dtype == torch.uint8:
        return DTYPE_E4M3
    if t.dtype == torch.float32:
        return DTYPE_F32
    raise TypeError(t.dtype)


def pack(cfg, tensors: Iterable[Tuple[str, int, dict]], device="cpu") -> torch.Tensor:
    """cfg: a model config (n_layers, hidden, ... fields); tensors yields
    (name, layer, {"w": tensor, "s": scales?}) as synth.SynthModel.tensors() does."""
    items: List[Tuple[int, int, torch.Tensor]] = []
    for name, layer, d in tensors:
        items.append((KINDS[name], layer, d["w"]))
        if "s" in d:
            items.append((KINDS[_SCALE_OF[name]], layer, d["s"]))
    table_off = HEADER.size
    off = _align(table_off + ENTRY.size * len(items))
    entries = []
    for kind, layer, t in items:
        rows = t.shape[0]
        cols = t.shape[1] if t.dim() == 2 else 1
        nbytes = t.numel() * t.element_size()
        entries.append((kind, layer, _dtype_code(t), rows, cols, off, nbytes))
        off = _align(off + nbytes)
    total = off
    head = HEADER.pack(MAGIC, VERSION, cfg.n_layers, cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads,
                       cfg.head_dim, cfg.ffn, cfg.vocab,
                       DTYPE_E4M3 if cfg.weight_dtype == "fp8" else DTYPE_BF16,
                       DTYPE_E4M3 if cfg.kv_dtype == "fp8" else DTYPE_BF16,
                       cfg.block_size, cfg.max_pos, cfg.eps, cfg.rope_theta, len(items), 0, table_off)
    meta = bytearray(head)
    for kind, layer, dt, rows, cols, o, n in entries:
        meta += ENTRY.pack(kind, layer, dt, 0, rows, cols, o, n)
    blob = torch.zeros(total, dtype=torch.uint8, device=device)
    blob[: len(meta)] = torch.frombuffer(bytearray(meta), dtype=torch.uint8).to(device)
    for (kind, layer, t), (_, _, _, _, _, o, n) in zip(items, entries):
        blob[o:o + n] = t.detach().contiguous().view(-1).view(torch.uint8).to(device)
    return blob
