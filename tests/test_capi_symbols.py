"""Host checks of the boundary: the library builds for sm_103a, loads without a
GPU, and exports every function include/*.h declares with the binding's
signature table covering exactly those names; the blob header layout matches
the C structs."""
import ctypes
import os
import re

import pytest

from memory_bound_transformer_gb300 import blob as mblob
from memory_bound_transformer_gb300 import build, capi

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


def declared_functions():
    names = set()
    for f in os.listdir(INCLUDE):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(INCLUDE, f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s+([a-z_0-9]+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    path = build.build()
    return ctypes.CDLL(path)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "decode_step" in names and "op_gemv" in names and len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert names == set(capi.SIGNATURES), names ^ set(capi.SIGNATURES)


def test_status_strings_without_gpu(lib):
    capi._lib = None
    l = capi.load()
    assert capi.status_string(0) == "ok"
    assert capi.status_string(-4) == "out of device memory"
    assert l.kv_bytes(None, 5) == 0
    assert l.model_destroy(None) == 0
    assert l.decode_step(None, None, 1, None, None, None, 1, None, None, None, None) == -1


def test_blob_layout_matches_header():
    text = open(os.path.join(INCLUDE, "mbt.h")).read()
    assert "} mbt_blob_header;          /* 80 bytes */" in text
    assert "} mbt_blob_tensor;          /* 48 bytes */" in text
    assert mblob.HEADER.size == 80 and mblob.ENTRY.size == 48
    from synth import TINY, SynthModel
    b = mblob.pack(TINY, SynthModel(TINY, 1).tensors())
    raw = bytes(b[:80].numpy())
    f = mblob.HEADER.unpack(raw)
    assert f[0] == b"MBTBLOB1" and f[1] == 1 and f[2:9] == (1, 256, 4, 2, 64, 688, 1024)
    n, off = f[15], f[17]
    ents = [mblob.ENTRY.unpack(bytes(b[off + 48 * i: off + 48 * (i + 1)].numpy())) for i in range(n)]
    assert all(e[6] % 256 == 0 and e[6] + e[7] <= b.numel() for e in ents)
    assert {(e[0], e[1]) for e in ents} >= {(0, -1), (12, -1), (2, 0), (7, 0)}


def test_sampling_struct_matches_header():
    text = open(os.path.join(INCLUDE, "mbt.h")).read()
    assert "} mbt_sampling;             /* 32 bytes */" in text
    assert ctypes.sizeof(capi.Sampling) == 32
    assert "#define MBT_TOPK_MAX 1024" in text and capi.TOPK_MAX == 1024


def test_argument_checks_before_any_device_call(lib):
    """Entry points reject malformed arguments with a status code before they
    touch the device (these run on a machine without a GPU)."""
    capi._lib = None
    l = capi.load()
    BAD = -1
    # op_gemv: unknown epilogue, unknown weight type, K not a multiple of 16
    assert l.op_gemv(7, 0, None, None, 8, 16, None, 1, 0, None, None, None, None, None, None, None) == BAD
    assert l.op_gemv(0, 9, None, None, 8, 16, None, 1, 0, None, None, None, None, None, None, None) == BAD
    assert l.op_gemv(0, 0, 1, None, 8, 17, 1, 1, 0, 1, None, None, None, None, None, None) == BAD
    # e4m3 weights need their per-row scales
    assert l.op_gemv(0, 1, 1, None, 8, 16, 1, 1, 0, 1, None, None, None, None, None, None) == BAD
    assert l.op_gemm_tc_e4m3(0, 1, None, 8, 64, 1, 16, 1, 1, None, None, None, None, None) == BAD
    # tensor-core entry points: batch above 128, K below 64
    assert l.op_gemm_tc(0, 1, None, 8, 64, 1, 129, 1, 1, None, None, None, None, None) == BAD
    assert l.op_gemm_tc(0, 1, None, 8, 32, 1, 16, 1, 1, None, None, None, None, None) == BAD
    # the step: a missing model or kv handle, and B <= 0
    assert l.model_create(None, 0, 0, None, None) == BAD
    assert l.kv_alloc(None, 4, None, None) == BAD
    assert l.model_capture(None, None, None, 0, 0, None) == BAD
    # sampling and prefill without handles or parameters
    assert l.decode_step_sample(None, None, 1, None, None, None, 1, None, None, None, None, None) == BAD
    assert l.prefill(None, None, 4, None, 0, None, 1, None, None, None) == BAD
