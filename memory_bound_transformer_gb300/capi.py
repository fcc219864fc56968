"""ctypes binding of libmbt.so (include/mbt.h, include/mbt_ops.h).

Argument marshalling only: tensors are passed as raw device (or host) pointers
and every step of the decode path runs in the library's CUDA kernels. There is
no fallback: if the library is missing or no sm_103 GPU is present the calls
raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmbt.so")

MBT_OK = 0
STATUS = {0: "MBT_OK", -1: "MBT_ERR_BAD_ARG", -2: "MBT_ERR_BATCH", -3: "MBT_ERR_CUDA",
          -4: "MBT_ERR_OOM", -5: "MBT_ERR_BLOB", -6: "MBT_ERR_UNSUPPORTED", -7: "MBT_ERR_NO_DEVICE",
          -8: "MBT_ERR_SCRATCH"}
DEV_TOKEN_RANGE, DEV_BLOCK_RANGE, DEV_POS_RANGE, DEV_SEQLEN_RANGE, DEV_NONFINITE = 1, 2, 4, 8, 16
EPI_PARTIAL, EPI_SWIGLU, EPI_ARGMAX = 0, 1, 2
DTYPE_BF16, DTYPE_E4M3, DTYPE_F32 = 0, 1, 2

# every symbol the headers declare, with (restype, argtypes)
_P, _I, _Z, _F, _U = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float, ctypes.c_uint32
SIGNATURES = {
    # mbt.h
    "model_create": (_I, [_P, _Z, _I, _P, ctypes.POINTER(_P)]),
    "model_destroy": (_I, [_P]),
    "model_info": (_I, [_P, _P]),
    "kv_bytes": (_Z, [_P, _I]),
    "kv_alloc": (_I, [_P, _I, _P, ctypes.POINTER(_P)]),
    "kv_free": (_I, [_P]),
    "kv_pool": (_I, [_P, ctypes.POINTER(_P), ctypes.POINTER(_Z)]),
    "kv_set_scales": (_I, [_P, _P, _P]),
    "model_capture": (_I, [_P, _P, _P, _I, _I, _P]),
    "model_set_eager": (_I, [_P, _I]),
    "decode_step": (_I, [_P, _P, _I, _P, _P, _P, _I, _P, _P, _P, _P]),
    "prefill": (_I, [_P, _P, _I, _P, _I, _P, _I, _P, _P, _P]),
    "decode_step_sample": (_I, [_P, _P, _I, _P, _P, _P, _I, _P, _P, _P, _P, _P]),
    "model_poll_errors": (_I, [_P, _P, ctypes.POINTER(_U)]),
    "model_stats": (_I, [_P, _I, ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "status_string": (ctypes.c_char_p, [_I]),
    # mbt_ops.h
    "op_embed_rmsnorm": (_I, [_I, _I, _I, _P, _P, _P, _F, _P, _P, _P, _P]),
    "op_add_rmsnorm": (_I, [_I, _I, _P, _P, _I, _P, _F, _P, _P]),
    "op_gemv_nsplit": (_I, [_I, _I, _I, _I, _I]),
    "op_gemv": (_I, [_I, _I, _P, _P, _I, _I, _P, _I, _I, _P, _P, _P, _P, ctypes.POINTER(_I), _P, _P]),
    "op_gemv_sched_ints": (_I, [_I, _I, _I, _I, _I]),
    "op_gemv_ex": (_I, [_I, _I, _P, _P, _I, _I, _P, _I, _I, _P, _P, _P, _P, ctypes.POINTER(_I), _P, _P, _P]),
    "op_gemv_norm_sched_ints": (_I, [_I, _I, _I, _I, _I]),
    "op_gemv_norm": (_I, [_I, _I, _P, _P, _I, _I, _P, _P, _I, _P, _F, _P, _I, _P, _P, _P, _P, _P, _P, _P]),
    "op_gemm_tc": (_I, [_I, _P, _P, _I, _I, _P, _I, _I, _P, _P, _P, _P, _P, _P]),
    "op_gemm_tc_e4m3": (_I, [_I, _P, _P, _I, _I, _P, _I, _I, _P, _P, _P, _P, _P, _P]),
    "op_rope_kv_write": (_I, [_I, _P, _I, _I, _I, _P, _P, _I, _I, _F, _P, _P, _I, _I, _F, _F, _P, _P, _P]),
    "op_paged_attention": (_I, [_I, _P, _I, _I, _I, _P, _P, _I, _F, _F, _P, _I, _P, _I, _P, _P, _P]),
    "op_paged_attention_noalloc": (_I, [_I, _P, _I, _I, _I, _P, _P, _I, _F, _F, _P, _I, _P, _I, _P, _P, _P]),
    "op_paged_attention_noalloc_limit": (_Z, []),
}

_lib: Optional[ctypes.CDLL] = None


class MbtError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)}")
        self.code = code


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (built by memory_bound_transformer_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -m memory_bound_transformer_gb300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    _lib = lib
    return lib


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return t.data_ptr()
    return int(t)


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(fn: str, rc: int) -> None:
    if rc != MBT_OK:
        raise MbtError(fn, rc)


def _require_cuda(*ts):
    for t in ts:
        if t is not None and isinstance(t, torch.Tensor) and not t.is_cuda:
            raise ValueError("device tensor expected")


# ---------------------------------------------------------------------------
# mbt.h

def model_create(blob: torch.Tensor, stream=None) -> int:
    lib = load()
    h = ctypes.c_void_p()
    on_dev = 1 if blob.is_cuda else 0
    _check("model_create", lib.model_create(_ptr(blob), blob.numel() * blob.element_size(), on_dev,
                                            _stream(stream), ctypes.byref(h)))
    return h.value


def model_destroy(model: int) -> None:
    _check("model_destroy", load().model_destroy(model))


def kv_bytes(model: int, num_blocks: int) -> int:
    return load().kv_bytes(model, num_blocks)


def kv_alloc(model: int, num_blocks: int, mem: Optional[torch.Tensor] = None) -> int:
    lib = load()
    h = ctypes.c_void_p()
    _require_cuda(mem)
    if mem is not None and mem.numel() * mem.element_size() < kv_bytes(model, num_blocks):
        raise ValueError("kv_alloc: the caller's memory is smaller than kv_bytes(model, num_blocks)")
    _check("kv_alloc", lib.kv_alloc(model, num_blocks, _ptr(mem), ctypes.byref(h)))
    return h.value


def kv_free(kv: int) -> None:
    _check("kv_free", load().kv_free(kv))


def kv_pool(kv: int):
    p, n = ctypes.c_void_p(), ctypes.c_size_t()
    _check("kv_pool", load().kv_pool(kv, ctypes.byref(p), ctypes.byref(n)))
    return p.value, n.value


def kv_set_scales(kv: int, k_scales: Sequence[float], v_scales: Sequence[float]) -> None:
    ks = (ctypes.c_float * len(k_scales))(*k_scales)
    vs = (ctypes.c_float * len(v_scales))(*v_scales)
    _check("kv_set_scales", load().kv_set_scales(kv, ks, vs))


def model_capture(model: int, kv: int, ladder: Optional[Sequence[int]], max_blocks_per_seq: int,
                  stream=None) -> None:
    lib = load()
    if ladder is None:
        arr, n = None, 0
    else:
        arr, n = (ctypes.c_int * len(ladder))(*ladder), len(ladder)
    _check("model_capture", lib.model_capture(model, kv, arr, n, max_blocks_per_seq, _stream(stream)))


def model_set_eager(model: int, eager: bool) -> None:
    _check("model_set_eager", load().model_set_eager(model, 1 if eager else 0))


def decode_step(model: int, kv: int, token_ids: torch.Tensor, positions: torch.Tensor,
                block_tables: torch.Tensor, seq_lens: torch.Tensor, next_ids: torch.Tensor,
                logits: Optional[torch.Tensor] = None, stream=None) -> None:
    """All tensors int32 on the device (logits fp32 [B][vocab] or None)."""
    _require_cuda(token_ids, positions, block_tables, seq_lens, next_ids, logits)
    B = token_ids.shape[0]
    bt_stride = block_tables.shape[1] if block_tables.dim() == 2 else block_tables.numel() // max(B, 1)
    _check("decode_step", load().decode_step(model, kv, B, _ptr(token_ids), _ptr(positions),
                                             _ptr(block_tables), bt_stride, _ptr(seq_lens),
                                             _ptr(next_ids), _ptr(logits), _stream(stream)))


def decode_step_raw(model: int, kv: int, B: int, tok, pos, bt, bt_stride: int, sl, next_ids,
                    logits=None, stream=None) -> int:
    """Pointer-level call; returns the status code instead of raising."""
    return load().decode_step(model, kv, B, _ptr(tok), _ptr(pos), _ptr(bt), bt_stride, _ptr(sl),
                              _ptr(next_ids), _ptr(logits), _stream(stream))


class Sampling(ctypes.Structure):
    """mbt_sampling (include/mbt.h)."""
    _fields_ = [("temperature", ctypes.c_float), ("top_k", ctypes.c_int32), ("top_p", ctypes.c_float),
                ("reserved", ctypes.c_uint32), ("seed", ctypes.c_uint64), ("step", ctypes.c_uint64)]


TOPK_MAX = 1024


def decode_step_sample(model: int, kv: int, token_ids, positions, block_tables, seq_lens, next_ids,
                       temperature: float, top_k: int, top_p: float, seed: int, step: int,
                       logits=None, stream=None) -> None:
    """decode_step with the next token drawn (temperature, top-k, top-p, seeded)."""
    _require_cuda(token_ids, positions, block_tables, seq_lens, next_ids, logits)
    B = token_ids.shape[0]
    sp = Sampling(float(temperature), int(top_k), float(top_p), 0, int(seed), int(step))
    _check("decode_step_sample", load().decode_step_sample(
        model, kv, B, _ptr(token_ids), _ptr(positions), _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
        ctypes.byref(sp), _ptr(next_ids), _ptr(logits), _stream(stream)))


def decode_step_sample_raw(model: int, kv: int, B: int, tok, pos, bt, bt_stride: int, sl, params, next_ids,
                           logits=None, stream=None) -> int:
    """Pointer-level call; returns the status code instead of raising."""
    return load().decode_step_sample(model, kv, B, _ptr(tok), _ptr(pos), _ptr(bt), bt_stride, _ptr(sl),
                                     ctypes.byref(params) if params is not None else None, _ptr(next_ids),
                                     _ptr(logits), _stream(stream))


def prefill(model: int, kv: int, tokens: torch.Tensor, start_pos: int, block_table: torch.Tensor,
            next_id: torch.Tensor, logits: Optional[torch.Tensor] = None, stream=None) -> None:
    """tokens [n] int32, block_table [bt_len] int32, next_id [1] int32 (device);
    logits [vocab] fp32 or None."""
    _require_cuda(tokens, block_table, next_id, logits)
    _check("prefill", load().prefill(model, kv, tokens.numel(), _ptr(tokens), int(start_pos), _ptr(block_table),
                                     block_table.numel(), _ptr(next_id), _ptr(logits), _stream(stream)))


def prefill_raw(model: int, kv: int, n: int, tokens, start_pos: int, block_table, bt_len: int, next_id,
                logits=None, stream=None) -> int:
    """Pointer-level call; returns the status code instead of raising."""
    return load().prefill(model, kv, n, _ptr(tokens), start_pos, _ptr(block_table), bt_len, _ptr(next_id),
                          _ptr(logits), _stream(stream))


def model_poll_errors(model: int, stream=None) -> int:
    bits = ctypes.c_uint32()
    _check("model_poll_errors", load().model_poll_errors(model, _stream(stream), ctypes.byref(bits)))
    return bits.value


def model_stats(model: int, B: int):
    k, g = ctypes.c_int(), ctypes.c_int()
    _check("model_stats", load().model_stats(model, B, ctypes.byref(k), ctypes.byref(g)))
    return k.value, bool(g.value)


def status_string(code: int) -> str:
    return load().status_string(code).decode()


# ---------------------------------------------------------------------------
# mbt_ops.h

def op_embed_rmsnorm(tokens, embed, gamma, eps, r, y, err=None, stream=None):
    B, H = r.shape
    _check("op_embed_rmsnorm", load().op_embed_rmsnorm(B, H, embed.shape[0], _ptr(tokens), _ptr(embed),
                                                       _ptr(gamma), eps, _ptr(r), _ptr(y), _ptr(err),
                                                       _stream(stream)))


def op_add_rmsnorm(r, delta, gamma, eps, y, stream=None):
    B, H = r.shape
    n = 0 if delta is None else delta.shape[0]
    _check("op_add_rmsnorm", load().op_add_rmsnorm(B, H, _ptr(r), _ptr(delta), n, _ptr(gamma), eps,
                                                   _ptr(y), _stream(stream)))


def op_gemv_nsplit(epi: int, w_dtype: int, B: int, N: int, K: int) -> int:
    return load().op_gemv_nsplit(epi, w_dtype, B, N, K)


def op_gemv(epi, w_dtype, W, scales, N, K, x, B, force_nsplit=0, out=None, act=None, logits=None,
            next_ids=None, err=None, stream=None) -> int:
    used = ctypes.c_int()
    _check("op_gemv", load().op_gemv(epi, w_dtype, _ptr(W), _ptr(scales), N, K, _ptr(x), B, force_nsplit,
                                     _ptr(out), _ptr(act), _ptr(logits), _ptr(next_ids),
                                     ctypes.byref(used), _ptr(err), _stream(stream)))
    return used.value


def op_gemv_sched_ints(epi: int, w_dtype: int, B: int, N: int, K: int) -> int:
    return load().op_gemv_sched_ints(epi, w_dtype, B, N, K)


def op_gemv_ex(epi, w_dtype, W, scales, N, K, x, B, sched, force_nsplit=0, out=None, act=None, logits=None,
               next_ids=None, err=None, stream=None) -> int:
    """op_gemv with caller-owned work-queue counters (zeroed int32 device
    tensor of op_gemv_sched_ints(...) elements; left zeroed)."""
    used = ctypes.c_int()
    _check("op_gemv_ex", load().op_gemv_ex(epi, w_dtype, _ptr(W), _ptr(scales), N, K, _ptr(x), B, force_nsplit,
                                           _ptr(out), _ptr(act), _ptr(logits), _ptr(next_ids),
                                           ctypes.byref(used), _ptr(sched), _ptr(err), _stream(stream)))
    return used.value


def op_gemv_norm_sched_ints(epi: int, w_dtype: int, B: int, N: int, K: int) -> int:
    return load().op_gemv_norm_sched_ints(epi, w_dtype, B, N, K)


def op_gemv_norm(epi, w_dtype, W, scales, N, K, r_in, delta, gamma, eps, r_out, sched=None, out=None, act=None,
                 logits=None, next_ids=None, err=None, stream=None) -> None:
    """The norm-prologue projection: r_in, r_out [B][K] fp32, delta [n][B][K]
    fp32 or None, gamma [K] BF16 (int16 bits or bfloat16)."""
    B = r_in.shape[0]
    n = 0 if delta is None else delta.shape[0]
    _check("op_gemv_norm", load().op_gemv_norm(epi, w_dtype, _ptr(W), _ptr(scales), N, K, _ptr(r_in), _ptr(delta),
                                               n, _ptr(gamma), eps, _ptr(r_out), B, _ptr(out), _ptr(act),
                                               _ptr(logits), _ptr(next_ids), _ptr(sched), _ptr(err),
                                               _stream(stream)))


def op_gemm_tc_e4m3(epi, W, scales, N, K, x, B, ksplit=1, out=None, act=None, logits=None, next_ids=None,
                    err=None, stream=None) -> None:
    _check("op_gemm_tc_e4m3", load().op_gemm_tc_e4m3(epi, _ptr(W), _ptr(scales), N, K, _ptr(x), B, ksplit,
                                                     _ptr(out), _ptr(act), _ptr(logits), _ptr(next_ids),
                                                     _ptr(err), _stream(stream)))


def op_gemm_tc(epi, W, scales, N, K, x, B, ksplit=1, out=None, act=None, logits=None, next_ids=None,
               err=None, stream=None) -> None:
    _check("op_gemm_tc", load().op_gemm_tc(epi, _ptr(W), _ptr(scales), N, K, _ptr(x), B, ksplit, _ptr(out),
                                           _ptr(act), _ptr(logits), _ptr(next_ids), _ptr(err), _stream(stream)))


def op_rope_kv_write(qkv, nq, nkv, d, positions, bt, max_pos, theta, kpool, vpool, num_blocks,
                     kv_dtype, k_scale, v_scale, q_out, err=None, stream=None):
    B = qkv.shape[0]
    _check("op_rope_kv_write", load().op_rope_kv_write(
        B, _ptr(qkv), nq, nkv, d, _ptr(positions), _ptr(bt), bt.shape[1], max_pos, theta, _ptr(kpool),
        _ptr(vpool), num_blocks, kv_dtype, k_scale, v_scale, _ptr(q_out), _ptr(err), _stream(stream)))


def op_paged_attention(q, nkv, kpool, vpool, kv_dtype, k_scale, v_scale, bt, seq_lens, num_blocks,
                       out, err=None, stream=None):
    B, nq, d = q.shape
    _check("op_paged_attention", load().op_paged_attention(
        B, _ptr(q), nq, nkv, d, _ptr(kpool), _ptr(vpool), kv_dtype, k_scale, v_scale, _ptr(bt),
        bt.shape[1], _ptr(seq_lens), num_blocks, _ptr(out), _ptr(err), _stream(stream)))


def op_paged_attention_noalloc(q, nkv, kpool, vpool, kv_dtype, k_scale, v_scale, bt, seq_lens,
                               num_blocks, out, err=None, stream=None) -> int:
    """Allocation-free variant; returns the status code (MBT_ERR_SCRATCH when the
    request exceeds the fixed scratch array) instead of raising."""
    B, nq, d = q.shape
    return load().op_paged_attention_noalloc(
        B, _ptr(q), nq, nkv, d, _ptr(kpool), _ptr(vpool), kv_dtype, k_scale, v_scale, _ptr(bt),
        bt.shape[1], _ptr(seq_lens), num_blocks, _ptr(out), _ptr(err), _stream(stream))


def op_paged_attention_noalloc_limit() -> int:
    return load().op_paged_attention_noalloc_limit()
