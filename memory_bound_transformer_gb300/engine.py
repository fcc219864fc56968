"""Session wrapper over the C ABI: one model, one paged KV cache, optional
graph ladder. Marshals torch device tensors to the library; computes nothing."""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from . import capi

DEFAULT_LADDER = (1, 2, 4, 8, 16, 24, 32, 40, 48, 56, 64)


class Engine:
    def __init__(self, blob: torch.Tensor, num_blocks: int, kv_mem: Optional[torch.Tensor] = None,
                 stream=None):
        self.stream = stream
        self.model = capi.model_create(blob, stream)
        self.kv = None
        try:
            self.kv = capi.kv_alloc(self.model, num_blocks, kv_mem)
        except Exception:
            capi.model_destroy(self.model)
            raise
        self.num_blocks = num_blocks
        self._kv_mem = kv_mem

    # -- cache -------------------------------------------------------------
    def pool(self, dtype=torch.uint8) -> torch.Tensor:
        """The KV pool as a flat device tensor view (no copy)."""
        ptr, nbytes = capi.kv_pool(self.kv)
        return _wrap_device(ptr, nbytes).view(dtype)

    def set_kv_scales(self, k: Sequence[float], v: Sequence[float]) -> None:
        capi.kv_set_scales(self.kv, k, v)

    # -- graphs ------------------------------------------------------------
    def capture(self, ladder: Optional[Sequence[int]] = DEFAULT_LADDER, max_blocks_per_seq: int = 1):
        capi.model_capture(self.model, self.kv, ladder, max_blocks_per_seq, self.stream)

    def set_eager(self, eager: bool) -> None:
        capi.model_set_eager(self.model, eager)

    # -- step --------------------------------------------------------------
    def step(self, tokens, positions, block_tables, seq_lens, next_ids, logits=None):
        capi.decode_step(self.model, self.kv, tokens, positions, block_tables, seq_lens, next_ids,
                         logits, self.stream)

    def step_sample(self, tokens, positions, block_tables, seq_lens, next_ids, temperature, top_k, top_p, seed,
                    step, logits=None):
        capi.decode_step_sample(self.model, self.kv, tokens, positions, block_tables, seq_lens, next_ids,
                                temperature, top_k, top_p, seed, step, logits, self.stream)

    def prefill(self, tokens, start_pos, block_table, next_id, logits=None):
        capi.prefill(self.model, self.kv, tokens, start_pos, block_table, next_id, logits, self.stream)

    def errors(self) -> int:
        return capi.model_poll_errors(self.model, self.stream)

    def stats(self, B: int):
        return capi.model_stats(self.model, B)

    def close(self) -> None:
        if self.kv is not None:
            capi.kv_free(self.kv)
            self.kv = None
        if self.model is not None:
            capi.model_destroy(self.model)
            self.model = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _wrap_device(ptr: int, nbytes: int) -> torch.Tensor:
    """A uint8 torch view of library-owned device memory (valid while the
    handle lives)."""
    class _Holder:
        def __init__(self, p, n):
            self.__cuda_array_interface__ = {"shape": (n,), "typestr": "|u1", "data": (p, False),
                                             "version": 3}
    return torch.as_tensor(_Holder(ptr, nbytes), device="cuda")
