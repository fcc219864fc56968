"""Host logic: the byte/FLOP ledger against the numbers the pages print.

"GPU Inference Internals": machine balance 989e12 / 3.35e12 ~ 295 and
1979e12 / 3.35e12 ~ 590 ("The Hardware Ledger"); 2 x 70e9 = 140 GFLOP, intensity
2, 3.35 TB/s / 70 GB ~ 48 tokens/s, crossover of 2B/b_w with 295 at B ~ 295
("Roofline: Why Decode Is Memory-Bound"); 2 x 80 x 8 x 128 x 2 ~ 320 KB per
token and ~40 GB at 128K tokens ("The KV-Cache Ledger"); the naive 8192^2 BF16
score matrix ~ 134 MB ("Kernels: FlashAttention and the Memory Hierarchy").
"CUDA graphs & kernel fusion", "Code": 5.5 GiB -> 5.9 / 8.1 / 5.9 ms, 1.36x and
14.2 GiB -> 15.2 / 17.4 / 15.3 ms, 1.14x."""
import pytest

from memory_bound_transformer_gb300 import ledger
from synth import EIGHT_B, SEVENTY_B_FP8, ONE_B


def test_machine_balance():
    assert round(ledger.machine_balance(989e12, 3.35e12)) == 295
    assert round(ledger.machine_balance(1979e12, 3.35e12)) == 591     # printed as "~590"
    assert abs(ledger.machine_balance(1979e12, 3.35e12) - 590) < 1.5


def test_roofline_70b_example():
    assert 2 * 70e9 == 140e9
    assert 140e9 / 70e9 == 2
    assert round(ledger.single_stream_ceiling(3.35e12, 70e9)) == 48
    # 2B / b_w reaches 295 FLOP/B near B = 295 for BF16 (b_w = 2) ...
    assert abs(ledger.weight_intensity(295, 2) - 295) < 1e-9
    # ... and for FP8 (b_w = 1, balance 590) at the same B
    assert abs(ledger.weight_intensity(295, 1) - 590) < 1e-9


def test_kv_ledger():
    per_tok = ledger.kv_bytes_per_token(80, 8, 128, 2)
    assert per_tok == 327680
    assert round(per_tok / 1024) == 320
    assert abs(per_tok * 128 * 1024 / 2 ** 30 - 40) < 1e-9          # 40 GiB at 128K tokens
    assert abs(8192 ** 2 * 2 / 1e6 - 134) < 0.3


@pytest.mark.parametrize("gib,printed", [(5.5, (5.9, 8.1, 5.9, 1.36)), (14.2, (15.2, 17.4, 15.3, 1.14))])
def test_launch_tax_printed_outputs(gib, printed):
    c, e, g, s = ledger.launch_tax(gib)
    assert (round(c, 1), round(e, 1), round(g, 1), round(s, 2)) == printed
    # the remark that the tax is ~36 % of a 6 ms step and ~14 % of a 15 ms step
    assert round((e - c) / c, 2) in ((0.36,) if gib == 5.5 else (0.14,))


def test_step_ledger_configs():
    # 8B BF16: ~15.0 GB of weights streamed per step
    assert abs(ledger.weight_bytes(EIGHT_B) / 1e9 - 15.01) < 0.02
    # 70B FP8: ~69.5 GB including per-channel scales
    assert abs(ledger.weight_bytes(SEVENTY_B_FP8) / 1e9 - 69.53) < 0.02
    # FLOPs ~ 2 x params at batch 1 and short context
    p = ledger.matmul_params(ONE_B)
    assert abs(ledger.step_flops(ONE_B, [16]) / (2 * p) - 1) < 0.01
    assert ledger.step_bytes(EIGHT_B, [1000]) == ledger.weight_bytes(EIGHT_B) + 1000 * 32 * 2 * 8 * 128 * 2
