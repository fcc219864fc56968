"""Host logic: the byte/FLOP ledger against the numbers the pages print.

The printed values live in tests/golden/ledger_printed.json, each with the page
title and section it comes from: machine balance ("GPU Inference Internals",
"The Hardware Ledger"), the 70B FP8 roofline example ("Roofline: Why Decode Is
Memory-Bound"), KV bytes per token ("The KV-Cache Ledger"), the naive score
matrix ("Kernels: FlashAttention and the Memory Hierarchy") and the launch-tax
step model's printed output ("CUDA graphs & kernel fusion", "Code")."""
import json
import os

import pytest

from memory_bound_transformer_gb300 import ledger
from synth import EIGHT_B, SEVENTY_B_FP8, ONE_B

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "ledger_printed.json")))


@pytest.mark.parametrize("case", GOLD["machine_balance"], ids=lambda c: str(c["printed"]))
def test_machine_balance(case):
    got = ledger.machine_balance(case["peak_flops"], case["hbm_bytes_per_s"])
    assert abs(got - case["printed"]) <= case["tol"]


def test_roofline_70b_example():
    c = GOLD["roofline_70b_fp8"]
    assert 2 * c["params"] == c["flops"]
    assert c["flops"] / c["weight_bytes"] == c["intensity"]
    assert round(ledger.single_stream_ceiling(c["hbm_bytes_per_s"], c["weight_bytes"])) == c["tokens_per_s"]
    # 2B / b_w reaches the BF16 balance (295) near B = 295 with b_w = 2 ...
    assert abs(ledger.weight_intensity(295, 2) - 295) < 1e-9
    # ... and twice that for FP8 (b_w = 1) at the same B
    assert abs(ledger.weight_intensity(295, 1) - 590) < 1e-9


def test_kv_ledger():
    c = GOLD["kv_per_token"]
    per_tok = ledger.kv_bytes_per_token(c["layers"], c["kv_heads"], c["head_dim"], c["bytes_per_elem"])
    assert per_tok == 2 * 80 * 8 * 128 * 2
    assert round(per_tok / 1024) == c["printed_kb"]
    assert abs(per_tok * 128 * 1024 / 2 ** 30 - c["gib_at_128k"]) < 1e-9
    n = GOLD["naive_score_matrix"]
    assert abs(n["tokens"] ** 2 * n["bytes_per_elem"] / 1e6 - n["printed_mb"]) < 0.3


@pytest.mark.parametrize("case", GOLD["launch_tax"], ids=lambda c: str(c["gib"]))
def test_launch_tax_printed_outputs(case):
    c, e, g, s = ledger.launch_tax(case["gib"])
    assert (round(c, 1), round(e, 1), round(g, 1), round(s, 2)) == \
        (case["compute_ms"], case["eager_ms"], case["graph_ms"], case["speedup"])
    # the remark that the tax is ~36 % of a 6 ms step and ~14 % of a 15 ms step
    assert round((e - c) / c, 2) == case["tax_frac"]


def test_step_ledger_configs():
    # 8B BF16: ~15.0 GB of weights streamed per step
    assert abs(ledger.weight_bytes(EIGHT_B) / 1e9 - 15.01) < 0.02
    # 70B FP8: ~69.5 GB including per-channel scales
    assert abs(ledger.weight_bytes(SEVENTY_B_FP8) / 1e9 - 69.53) < 0.02
    # FLOPs ~ 2 x params at batch 1 and short context
    p = ledger.matmul_params(ONE_B)
    assert abs(ledger.step_flops(ONE_B, [16]) / (2 * p) - 1) < 0.01
    assert ledger.step_bytes(EIGHT_B, [1000]) == ledger.weight_bytes(EIGHT_B) + 1000 * 32 * 2 * 8 * 128 * 2
