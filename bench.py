"""Decode-step benchmark: one JSON line on rank 0.

A step is one decode step (the whole per-layer kernel sequence, final norm, LM
head and greedy arg-max) for one batch of sequences, replayed from the captured
CUDA graph. The headline is the 8B-class BF16 decoder at batch 1 with a
per-sequence context drawn uniformly from [256, 2048] (random-init weights and
random cache contents), each step feeding back the previous step's token ids and
advancing every position by one; the same line carries batch 64 of that model
and the 70B-class FP8 decoder at batch 1 and 64 (context 2048).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 8b] [--batch 1]
                  [--also 70b_fp8,32b_fp8] [--impl reference]

Under torchrun every rank runs its own replica on its own GPU (the decode step
has no cross-sequence exchange, so there is no collective on the data path);
rank 0 prints the whole-job tokens/s over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from memory_bound_transformer_gb300 import blob as mblob  # noqa: E402
from memory_bound_transformer_gb300 import capi, ledger  # noqa: E402
from memory_bound_transformer_gb300.engine import Engine  # noqa: E402
from synth import WORKLOADS, SynthModel, random_contexts, random_kv_pool, seeded_block_tables  # noqa: E402

METRIC = "decode tokens/s at batch 1 and 64; achieved HBM GB/s as % of GB300 peak"
L2_BYTES = 126 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0
# dram__bytes_read.sum + dram__bytes_write.sum per launch of each workload's
# dominant batch-1 kernel (the gate/up projection with the norm prologue and
# SwiGLU epilogue) from one ncu capture of the current kernel; a workload
# without a capture of the current kernel reports null.
DRAM_TRAFFIC = {("8b", 1): 239_231_488, ("70b_fp8", 1): 474_587_904}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="8b", choices=sorted(WORKLOADS))
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--also", default="70b_fp8",
                    help="comma-separated workloads measured after the headline one at batch 1 and their "
                         "largest batch ('' for none)")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-kernel-timing", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--ladder", default=None, help="comma-separated graph ladder (default: the workload's)")
    ap.add_argument("--context", default=None,
                    help="LO,HI: per-sequence context range instead of the workload's (context sweeps)")
    ap.add_argument("--sweep", action="store_true",
                    help="batch sweep over the graph ladder: one JSON line per batch (tok/s, step p50/p99, GB/s)")
    ap.add_argument("--kernel-only", nargs="?", const="gemv_norm", default=None,
                    choices=["gemv", "gemv_norm", "attention", "tc"],
                    help="time one kernel alone for profiling: the gate/up GEMV over 4 layers' matrices (x "
                         "given, or with the step's norm prologue), the tensor-core gate/up, or one layer's "
                         "paged attention at the workload's contexts")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense BF16 tensor peak (TFLOP/s): measured burst, else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p))["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


class Clocks:
    """nvidia-smi sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
            out, _ = self.p.communicate()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def build_case(wl, B, steps_total, device="cuda", context=None):
    cfg = wl.model
    lo, hi = context or wl.context
    ctx = random_contexts(B, lo, hi, wl.seed + 2000)
    cap = ctx + steps_total + 1
    nb = int(sum(-(-int(c) // 16) for c in cap)) + 1
    tables = seeded_block_tables(cap, 16, nb, wl.seed + 3000)
    tables[tables < 0] = nb
    model = SynthModel(cfg, wl.seed, device=device, cache=False)
    blob = mblob.pack(cfg, model.tensors(), device=device)
    # the generator's tensors are not needed once packed: free them before the
    # engine allocates its own copy of the weights and the KV pool
    del model
    torch.cuda.empty_cache()
    eng = Engine(blob, nb)
    del blob
    torch.cuda.empty_cache()
    pool = random_kv_pool(cfg, nb, wl.seed + 4000, device=device)
    eng.pool().copy_(pool.view(torch.uint8).reshape(-1))
    del pool
    return cfg, ctx, tables, nb, eng


def job_rate(local_ms: float, local_tokens: int, world: int, device=None):
    """Whole-job throughput of N replicas: the tokens of all ranks over the
    slowest rank's time (replicas share nothing, so the job ends with the last
    one). Returns (tokens/s, max ms, total tokens); collective only for N > 1."""
    if world == 1:
        return local_tokens / (local_ms / 1e3), local_ms, local_tokens
    t = torch.tensor([local_ms], dtype=torch.float64, device=device)
    n = torch.tensor([float(local_tokens)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.all_reduce(n, op=torch.distributed.ReduceOp.SUM)
    return n.item() / (t.item() / 1e3), t.item(), int(n.item())


def timed_steps(eng, cfg, ctx, tables, B, K, W, dev, world, clocks_on):
    """W untimed then K timed decode steps at batch B (rows 0..B-1 of the case);
    each step feeds back the previous ids and advances every position by one."""
    S = torch.cuda.current_stream()
    total = K + W
    pos_all = torch.tensor(np.stack([ctx[:B] + t for t in range(total)]), dtype=torch.int32, device=dev)
    sl_all = pos_all + 1
    bt = torch.tensor(tables[:B], device=dev)
    ids = [torch.randint(0, cfg.vocab, (B,), dtype=torch.int32, device=dev) for _ in range(2)]

    def step(t):
        eng.step(ids[t % 2], pos_all[t], bt, sl_all[t], ids[(t + 1) % 2])

    for t in range(W):
        step(t)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = Clocks(dev.index) if clocks_on else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    torch.cuda.synchronize()
    ev[0].record(S)
    for t in range(K):
        step(W + t)
        ev[t + 1].record(S)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ck = clocks.stop() if clocks else None
    per_step = [ev[i].elapsed_time(ev[i + 1]) for i in range(K)]
    rate, total_ms, _ = job_rate(ev[0].elapsed_time(ev[K]), B * K, world, dev)
    byte_steps = [ledger.step_bytes(cfg, ctx[:B] + W + t + 1) for t in range(K)]
    kps, graph = eng.stats(B)
    return dict(B=B, total_ms=total_ms, rate=rate, per_step=per_step, avg_bytes=float(np.mean(byte_steps)),
                clocks=ck, kernels_per_step=kps, uses_graph=graph)


def measure_workload(wl, batches, args, world, head):
    """Build one workload (weights, random cache, graph ladder) and time its
    decode step at each batch; the headline workload also times the eager
    launch-tax ablation and the end-to-end path. Every workload times its
    dominant batch-1 kernel (gate/up with the norm prologue) and, when a batch
    runs on the tensor cores, the tensor-core gate/up at its largest batch."""
    Bmax = max(batches)
    K, W = args.steps, args.warmup
    dev = torch.device("cuda", torch.cuda.current_device())
    context = tuple(int(v) for v in args.context.split(",")) if (args.context and head) else None
    e2e_on = head and not args.no_e2e
    cfg, ctx, tables, nb, eng = build_case(wl, Bmax, K + W + (K + 2 if e2e_on else 0), context=context)
    mbs = tables.shape[1]
    ladder = [int(x) for x in args.ladder.split(",")] if (args.ladder and head) else list(wl.ladder)
    if Bmax > max(ladder):
        ladder = sorted(set(ladder) | {Bmax})
    eng.capture(ladder=ladder, max_blocks_per_seq=mbs)
    runs = [timed_steps(eng, cfg, ctx, tables, B, K, W, dev, world, clocks_on=(head and i == 0))
            for i, B in enumerate(batches)]
    eager = None
    if head:
        # launch-tax ablation ("CUDA graphs & kernel fusion", "Direct answer":
        # T_eager ~ T_compute + N tau, T_graph ~ T_compute + tau): the same
        # step, same kernels, launched one by one from the host
        eng.set_eager(True)
        eager = timed_steps(eng, cfg, ctx, tables, batches[0], K, W, dev, world, clocks_on=False)
        eng.set_eager(False)
    B0 = batches[0]
    e2e = None
    if e2e_on:
        bt0 = torch.tensor(tables[:B0], device=dev)
        e2e = time_e2e(eng, cfg, ctx[:B0] + W + K, bt0, B0, K, dev, tables[:B0])
    pf = None
    if head and not args.no_prefill:
        pf = [time_prefill(eng, cfg, n, nb, dev) for n in (512, 2048) if -(-n // 16) <= nb]
    eng.close()
    del eng
    torch.cuda.empty_cache()
    kern = kern_tc = None
    if not args.no_kernel_timing:
        kern = time_gemv_norm_swiglu(cfg, wl, B0, dev)
        if Bmax >= 16:
            kern_tc = time_tc_swiglu(cfg, wl, Bmax, dev)
    return dict(cfg=cfg, K=K, W=W, runs=runs, kern=kern, kern_tc=kern_tc, e2e=e2e, ctx=ctx, wl=wl, eager=eager,
                prefill=pf)


def batch_sweep(args):
    """Tokens/s against step latency across the graph ladder ("GPU Inference
    Internals", "Batching Economics": the weight bytes are shared by the batch,
    the KV bytes grow with it), one graph per rung, same contexts."""
    wl = WORKLOADS[args.workload]
    ladder = [int(x) for x in args.ladder.split(",")] if args.ladder else list(wl.ladder)
    K, W = args.steps, args.warmup
    dev = torch.device("cuda", torch.cuda.current_device())
    cfg, ctx, tables, nb, eng = build_case(wl, max(ladder), K + W)
    eng.capture(ladder=ladder, max_blocks_per_seq=tables.shape[1])
    peak, src = peaks()
    for B in ladder:
        r = timed_steps(eng, cfg, ctx, tables, B, K, W, dev, 1, clocks_on=False)
        ps = np.array(r["per_step"])
        gbs = r["avg_bytes"] / (np.mean(ps) / 1e3) / 1e9
        print(json.dumps({"sweep": wl.key, "batch": B, "tokens_per_s": round(r["rate"], 2),
                          "step_ms_p50": round(float(np.percentile(ps, 50)), 4),
                          "step_ms_p99": round(float(np.percentile(ps, 99)), 4),
                          "bytes_per_step": int(r["avg_bytes"]), "achieved_gbs": round(gbs, 1),
                          "frac_of_peak": round(gbs / peak, 4), "peak_source": src,
                          "kernels_per_step": r["kernels_per_step"], "graph": r["uses_graph"]}), flush=True)
    eng.close()


def _gate_up_mats(cfg, wl, dev, layers):
    """Gate/up matrices of a few layers (each larger than L2), enough distinct
    bytes that back-to-back launches read from HBM."""
    model = SynthModel(cfg, wl.seed + 17, device=dev, cache=False)
    w = 1 if cfg.weight_dtype == "fp8" else 2
    nl = min(cfg.n_layers, max(2, int(24e9 // (2 * cfg.ffn * cfg.hidden * w))))
    if layers:
        nl = min(nl, layers)
    return [model.get("w_gu", l) for l in range(nl)]


def time_gemv_swiglu(cfg, wl, B, dev, reps=3, layers=None):
    """Average duration of the gate/up GEMV (SwiGLU epilogue, x given) on its
    own stream with CUDA events, cycling through several layers' matrices."""
    mats = _gate_up_mats(cfg, wl, dev, layers)
    x = torch.randn((B, cfg.hidden), device=dev)
    act = torch.empty((B, cfg.ffn), device=dev)
    wdt = capi.DTYPE_E4M3 if cfg.weight_dtype == "fp8" else capi.DTYPE_BF16
    # the work-queue counters stay zeroed between launches: no memset between them
    sched = torch.zeros(max(1, capi.op_gemv_sched_ints(capi.EPI_SWIGLU, wdt, B, cfg.ffn, cfg.hidden)),
                        dtype=torch.int32, device=dev)
    torch.cuda.synchronize()     # the inputs are generated on other streams
    s = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(s):
        for m in mats[:2]:
            capi.op_gemv_ex(capi.EPI_SWIGLU, wdt, m["w"], m.get("s"), cfg.ffn, cfg.hidden, x, B, sched, act=act,
                            stream=s)
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        n = 0
        for _ in range(reps):
            for m in mats:
                capi.op_gemv_ex(capi.EPI_SWIGLU, wdt, m["w"], m.get("s"), cfg.ffn, cfg.hidden, x, B, sched,
                                act=act, stream=s)
                n += 1
        e1.record(s)
        s.synchronize()
    ms = e0.elapsed_time(e1) / n
    w = 1 if cfg.weight_dtype == "fp8" else 2
    nbytes = 2 * cfg.ffn * cfg.hidden * w + (2 * cfg.ffn * 4 if cfg.weight_dtype == "fp8" else 0) \
        + B * cfg.hidden * 4 + B * cfg.ffn * 4
    del mats
    torch.cuda.empty_cache()
    return {"ms": ms, "bytes": nbytes, "launches": n}


def time_gemv_norm_swiglu(cfg, wl, B, dev, reps=3, layers=None):
    """The step's dominant batch-1 kernel as the step launches it: the gate/up
    projection with the residual add + RMSNorm prologue (residual and two split
    partials in, new residual out) and the SwiGLU epilogue, CUDA events on its
    own stream over several layers' matrices. Algorithmic bytes per launch:
    weights (+ FP8 scales) + gain + residual and partials read + residual
    written + activation written."""
    mats = _gate_up_mats(cfg, wl, dev, layers)
    H, F = cfg.hidden, cfg.ffn
    r = torch.randn((B, H), device=dev)
    delta = torch.randn((2, B, H), device=dev) * 0.1
    r_out = torch.empty_like(r)
    gamma = (1.0 + 0.1 * torch.randn(H, device=dev)).to(torch.bfloat16)
    act = torch.empty((B, F), device=dev)
    wdt = capi.DTYPE_E4M3 if cfg.weight_dtype == "fp8" else capi.DTYPE_BF16
    sched = torch.zeros(max(1, capi.op_gemv_norm_sched_ints(capi.EPI_SWIGLU, wdt, B, F, H)),
                        dtype=torch.int32, device=dev)
    torch.cuda.synchronize()     # the inputs are generated on other streams
    s = torch.cuda.Stream(device=dev)

    def launch(m):
        capi.op_gemv_norm(capi.EPI_SWIGLU, wdt, m["w"], m.get("s"), F, H, r, delta, gamma, cfg.eps, r_out,
                          sched=sched, act=act, stream=s)

    with torch.cuda.stream(s):
        for m in mats[:2]:
            launch(m)
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        n = 0
        for _ in range(reps):
            for m in mats:
                launch(m)
                n += 1
        e1.record(s)
        s.synchronize()
    ms = e0.elapsed_time(e1) / n
    w = 1 if cfg.weight_dtype == "fp8" else 2
    nbytes = 2 * F * H * w + (2 * F * 4 if cfg.weight_dtype == "fp8" else 0) + H * 2 \
        + 3 * B * H * 4 + B * H * 4 + B * F * 4
    del mats
    torch.cuda.empty_cache()
    return {"ms": ms, "bytes": nbytes, "launches": n}


def time_tc_swiglu(cfg, wl, B, dev, reps=3, layers=4):
    """Average duration of the tensor-core gate/up projection with the SwiGLU
    epilogue (the e4m3 kernel for FP8 weights) at batch B over a few layers'
    matrices. The entry-point calls are captured once in a CUDA graph and the
    graph is replayed between CUDA events, so host-side work per call (tensor
    map encoding, argument marshalling) is not in the time; the entry point's
    activation split (BF16 high/low rows, or e4m3 term rows) and act
    read-back kernels are (a few us)."""
    model = SynthModel(cfg, wl.seed + 17, device=dev, cache=False)
    mats = [model.get("w_gu", l) for l in range(min(cfg.n_layers, layers))]
    x = torch.randn((B, cfg.hidden), device=dev)
    act = torch.empty((B, cfg.ffn), device=dev)
    fp8 = cfg.weight_dtype == "fp8"
    fn = capi.op_gemm_tc_e4m3 if fp8 else capi.op_gemm_tc
    torch.cuda.synchronize()     # the inputs are generated on other streams
    s = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(s):
        for m in mats[:2]:
            fn(capi.EPI_SWIGLU, m["w"], m.get("s"), cfg.ffn, cfg.hidden, x, B, act=act, stream=s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for m in mats:
                fn(capi.EPI_SWIGLU, m["w"], m.get("s"), cfg.ffn, cfg.hidden, x, B, act=act, stream=s)
        g.replay()
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(reps):
            g.replay()
        e1.record(s)
        s.synchronize()
    n = reps * len(mats)
    ms = e0.elapsed_time(e1) / n
    w = 1 if fp8 else 2
    nbytes = 2 * cfg.ffn * cfg.hidden * w + (2 * cfg.ffn * 4 if fp8 else 0) + B * cfg.hidden * 4 + B * cfg.ffn * 4
    flops = 2 * B * 2 * cfg.ffn * cfg.hidden
    del g, mats
    torch.cuda.empty_cache()
    return {"ms": ms, "bytes": nbytes, "flops": flops, "launches": n, "B": B}


def time_attention(wl, B, dev, reps=10):
    """One layer's paged attention at batch B over the workload's contexts (a
    one-layer cache of random values), timed with CUDA events on its stream."""
    cfg = wl.model
    lo, hi = wl.context
    ctx = random_contexts(B, lo, hi, wl.seed + 2000)
    nb = int(sum(-(-int(c) // 16) for c in ctx)) + 1
    tables = seeded_block_tables(ctx, 16, nb, wl.seed + 3000)
    tables[tables < 0] = nb
    one = cfg.replace(n_layers=1)
    pool = random_kv_pool(one, nb, wl.seed + 4000, device=dev).view(torch.uint8).reshape(2, -1)
    q = torch.randn((B, cfg.n_q_heads, cfg.head_dim), device=dev)
    out = torch.empty((B, cfg.n_q_heads * cfg.head_dim), device=dev)
    bt = torch.tensor(tables, device=dev)
    sl = torch.tensor(ctx, device=dev)
    kvd = capi.DTYPE_E4M3 if cfg.kv_dtype == "fp8" else capi.DTYPE_BF16
    torch.cuda.synchronize()     # the inputs are generated on other streams
    s = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(s):
        for _ in range(2):
            capi.op_paged_attention(q, cfg.n_kv_heads, pool[0], pool[1], kvd, 1.0, 1.0, bt, sl, nb, out, stream=s)
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(reps):
            capi.op_paged_attention(q, cfg.n_kv_heads, pool[0], pool[1], kvd, 1.0, 1.0, bt, sl, nb, out, stream=s)
        e1.record(s)
        s.synchronize()
    k = 1 if cfg.kv_dtype == "fp8" else 2
    nbytes = int(sum(int(c) for c in ctx)) * 2 * cfg.n_kv_heads * cfg.head_dim * k
    return {"ms": e0.elapsed_time(e1) / reps, "bytes": nbytes, "launches": reps}


def time_prefill(eng, cfg, n, nb, dev, reps=3):
    """Time to first token for an n-token prompt ("Kernel Fusion for
    Large-Scale LLM Inference", section 12: TTFT): one prefill call from
    position 0 over the first ceil(n / 16) blocks of the pool (their random
    contents are overwritten), CUDA events on the current stream, the best of
    `reps` after one warm-up. FLOPs: 2 x matmul params x n (the LM head once)
    + the causal attention products."""
    S = torch.cuda.current_stream()
    toks = torch.randint(0, cfg.vocab, (n,), dtype=torch.int32, device=dev)
    table = torch.arange(-(-n // 16), dtype=torch.int32, device=dev)
    nid = torch.zeros(1, dtype=torch.int32, device=dev)
    eng.prefill(toks, 0, table, nid)
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(S)
        eng.prefill(toks, 0, table, nid)
        e1.record(S)
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    per_tok = ledger.matmul_params(cfg) - cfg.vocab * cfg.hidden
    flops = 2 * per_tok * n + 2 * cfg.vocab * cfg.hidden + \
        2 * 2 * cfg.n_layers * cfg.n_q_heads * cfg.head_dim * (n * (n + 1) // 2)
    return {"tokens": n, "ttft_ms": round(best, 3), "tokens_per_s": round(n / (best / 1e3), 1),
            "flops": int(flops), "achieved_tflops": round(flops / (best / 1e3) / 1e12, 1)}


def time_e2e(eng, cfg, ctx0, bt, B, K, dev, tables):
    """Same metric through the public API with host buffers: every step copies
    its inputs from pinned host memory and reads the next ids back."""
    h_tok = torch.randint(0, cfg.vocab, (B,), dtype=torch.int32).pin_memory()
    h_pos = torch.zeros(B, dtype=torch.int32).pin_memory()
    h_sl = torch.zeros(B, dtype=torch.int32).pin_memory()
    h_bt = torch.tensor(tables).pin_memory()
    h_out = torch.zeros(B, dtype=torch.int32).pin_memory()
    d_tok = torch.empty(B, dtype=torch.int32, device=dev)
    d_pos, d_sl = torch.empty_like(d_tok), torch.empty_like(d_tok)
    d_bt = torch.empty_like(bt)
    d_out = torch.empty_like(d_tok)
    S = torch.cuda.current_stream()
    h2d = (3 * B + h_bt.numel()) * 4
    d2h = B * 4

    def one(t):
        h_pos.copy_(torch.from_numpy(ctx0 + t))
        h_sl.copy_(h_pos + 1)
        d_tok.copy_(h_tok, non_blocking=True)
        d_pos.copy_(h_pos, non_blocking=True)
        d_sl.copy_(h_sl, non_blocking=True)
        d_bt.copy_(h_bt, non_blocking=True)
        eng.step(d_tok, d_pos, d_bt, d_sl, d_out)
        h_out.copy_(d_out, non_blocking=True)
        S.synchronize()
        h_tok.copy_(h_out)

    one(0)
    one(1)
    t0 = time.perf_counter()
    for t in range(K):
        one(2 + t)
    dt = time.perf_counter() - t0
    return {"value": B * K / dt, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


def cpu_baseline(wl, B, budget_s=20.0):
    """The fp64 oracle on this host's cores, on a bounded sample of the workload:
    embedding + final norm + LM head, plus as many decoder layers as fit the
    budget, extrapolated to the full depth. Weights are copied to host memory
    before the clock starts."""
    from oracle.decode import OracleKV, decode_step
    from synth import raw_numpy

    cfg = wl.model
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    ctx = random_contexts(B, wl.context[0], wl.context[1], wl.seed + 2000)
    rows = min(B, 1)
    ctx_s = ctx[:rows]
    cap = ctx_s + 1
    nb = int(sum(-(-int(c) // 16) for c in cap)) + 1
    tables = seeded_block_tables(cap, 16, nb, wl.seed + 3000)
    model = SynthModel(cfg, wl.seed, device=dev, cache=False)
    cache = {}

    def W(name, layer):
        k = (name, layer)
        if k not in cache:
            cache[k] = {a: raw_numpy(v) for a, v in model.get(name, layer).items()}
        return cache[k]

    def run(nl):
        one = random_kv_pool(cfg.replace(n_layers=max(nl, 1)), nb, wl.seed + 4000, device="cpu")
        raw = one.numpy().view(np.uint16) if one.dtype == torch.int16 else one.numpy()
        kv = OracleKV(raw, np.ones(max(nl, 1)), np.ones(max(nl, 1)))
        t0 = time.perf_counter()
        decode_step(W, cfg, kv, [1] * rows, ctx_s, tables, ctx_s + 1, layers=range(nl))
        return time.perf_counter() - t0

    W("embed", -1), W("g_final", -1), W("lm_head", -1)
    t0 = run(0)
    nl = 1
    for n in ("g_attn", "w_qkv", "w_o", "g_ffn", "w_gu", "w_down"):
        W(n, 0)
    t1 = run(1)
    per_layer = max(t1 - t0, 1e-9)
    extra = int(max(0, min(cfg.n_layers - 1, (budget_s - t0 - t1) // max(per_layer, 1e-3))))
    if extra >= 1:
        nl = 1 + min(extra, 3)
        for l in range(1, nl):
            for n in ("g_attn", "w_qkv", "w_o", "g_ffn", "w_gu", "w_down"):
                W(n, l)
        tn = run(nl)
        per_layer = max((tn - t0) / nl, 1e-9)
    t_step = t0 + cfg.n_layers * per_layer
    threads = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
    cores = int(threads) if threads else (os.cpu_count() or 1)
    return {"value": rows / t_step, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"1 sequence of the {cfg.name} workload: embedding, final norm and LM head "
                      f"plus {nl} of {cfg.n_layers} layers timed, per-layer time extrapolated to "
                      f"the full depth; fp64 NumPy, {t_step:.2f} s per token-step"}


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        return main_reference(args)
    torch.cuda.set_device(local)
    if args.sweep:
        capi.load()
        batch_sweep(args)
        return
    if args.kernel_only:
        capi.load()
        wl = WORKLOADS[args.workload]
        B = args.batch or 1
        dev = torch.device("cuda", local)
        peak, src = peaks()
        if args.kernel_only == "attention":
            k = time_attention(wl, B, dev)
            name = "paged attention (split-K, tensor-core QK/PV, merge)"
        elif args.kernel_only == "tc":
            k = time_tc_swiglu(wl.model, wl, args.batch or 64, dev)
            B = args.batch or 64
            name = "tensor-core gate/up with SwiGLU epilogue (" + wl.model.weight_dtype + " weights)"
        elif args.kernel_only == "gemv":
            k = time_gemv_swiglu(wl.model, wl, B, dev, reps=1, layers=4)
            name = "gate/up GEMV with SwiGLU epilogue"
        else:
            k = time_gemv_norm_swiglu(wl.model, wl, B, dev, reps=1, layers=4)
            name = "gate/up GEMV with the norm prologue and SwiGLU epilogue"
        gbs = k["bytes"] / (k["ms"] / 1e3) / 1e9
        line = {"kernel": name, "workload": wl.key, "batch": B, "launches": k["launches"],
                "avg_ms": round(k["ms"], 5), "bytes": k["bytes"], "achieved_gbs": round(gbs, 1),
                "frac": round(gbs / peak, 4), "peak_source": src}
        if "flops" in k:
            line["achieved_tflops"] = round(k["flops"] / (k["ms"] / 1e3) / 1e12, 1)
        print(json.dumps(line))
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    capi.load()
    peak, src = peaks()
    wl = WORKLOADS[args.workload]
    batches = [args.batch] if args.batch else [b for b in wl.batches if b in (1, 64)] or [wl.batches[0]]
    r = measure_workload(wl, batches, args, world, head=True)
    extra = []
    if not args.batch and args.also:
        for key in [k for k in args.also.split(",") if k and k != wl.key]:
            wx = WORKLOADS[key]
            bx = sorted({wx.batches[0], max(wx.batches)})
            extra.append(measure_workload(wx, bx, args, world, head=False))
    cfg, K = r["cfg"], r["K"]

    def summary(run):
        step_ms = run["total_ms"] / K
        gbs = run["avg_bytes"] / (step_ms * 1e-3) / 1e9
        ps = sorted(run["per_step"])
        return {"batch": run["B"], "value": round(run["rate"], 2),
                "unit": "tokens/s", "ms_per_step": round(step_ms, 4),
                "latency_ms": {"p50": round(ps[len(ps) // 2], 4),
                               "p99": round(ps[min(len(ps) - 1, int(0.99 * len(ps)))], 4)},
                "step_roofline": {"bytes_per_step": int(run["avg_bytes"]), "achieved_gbs": round(gbs, 1),
                                  "frac_of_peak": round(gbs / peak, 4), "frac_of_8tbs": round(gbs / 8000, 4)},
                "kernels_per_step": run["kernels_per_step"], "graph": run["uses_graph"]}

    def roofline(res, B):
        k = res["kern"]
        if not k:
            return None
        gbs = k["bytes"] / (k["ms"] / 1e3) / 1e9
        wt = res["cfg"].weight_dtype
        return {"kernel": "gemv_kernel<NB=1,%s,EPI_SWIGLU,PRO_NORM> (residual add + RMSNorm prologue, fused "
                          "gate/up, SiLU x mul epilogue; as the step launches it)" % ("W_E4M3" if wt == "fp8" else "W_BF16"),
                "workload": res["wl"].key, "batch": B,
                "bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "peak_source": src,
                "unit": "GB/s", "frac": round(gbs / peak, 4), "traffic": DRAM_TRAFFIC.get((res["wl"].key, B)),
                "algorithmic_bytes_per_launch": k["bytes"], "avg_launch_ms": round(k["ms"], 5),
                "launches_timed": k["launches"]}

    def roofline_tc(res):
        k = res["kern_tc"]
        if not k:
            return None
        gbs = k["bytes"] / (k["ms"] / 1e3) / 1e9
        f8 = res["cfg"].weight_dtype == "fp8"
        return {"kernel": "tc_stream_kernel<%s, EPI_SWIGLU> (persistent stream-K tcgen05 gate/up at batch %d; "
                          "the entry point's row split and read-back kernels included)" % ("W_E4M3" if f8 else "W_BF16",
                                                                                         k["B"]),
                "bound": "hbm", "achieved": round(gbs, 1), "peak": peak,
                "unit": "GB/s", "frac": round(gbs / peak, 4),
                "achieved_tflops": round(k["flops"] / (k["ms"] / 1e3) / 1e12, 1),
                "algorithmic_bytes_per_launch": k["bytes"], "avg_launch_ms": round(k["ms"], 5)}

    head = summary(r["runs"][0])
    B = head["batch"]
    line = {
        "metric": METRIC,
        "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": r["W"],
        "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if cfg.weight_dtype == "bf16" else "fp8-e4m3 weights, fp32 math",
        "data": "synthetic (seeded random-init weights N(0,0.02), random KV contents and token ids)",
        "config": {"workload": f"{r['wl'].key}: {r['wl'].description}", "model": cfg.name, "batch": B,
                   "context_start": [int(c) for c in r["ctx"][:8]], "graph": head["graph"],
                   "l2": "weights of every step (%.1f GB) exceed L2; no flush needed"
                         % (head["step_roofline"]["bytes_per_step"] / 1e9),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "latency_ms": head["latency_ms"],
        "step_roofline": head["step_roofline"],
        "roofline": roofline(r, B),
        "kernels_per_step": head["kernels_per_step"],
    }
    for run in r["runs"][1:]:
        line["batch%d" % run["B"]] = summary(run)
        if run["B"] == max(batches) and roofline_tc(r):
            line["batch%d" % run["B"]]["roofline_tc"] = roofline_tc(r)
    for x in extra:
        obj = {"workload": f"{x['wl'].key}: {x['wl'].description}", "model": x["cfg"].name}
        for run in x["runs"]:
            obj["batch%d" % run["B"]] = summary(run)
        obj["roofline"] = roofline(x, x["runs"][0]["B"])
        if roofline_tc(x):
            obj["roofline_tc"] = roofline_tc(x)
        line[x["wl"].key] = obj
    ge, ee = r["runs"][0]["total_ms"] / K, r["eager"]["total_ms"] / K
    n_k = r["eager"]["kernels_per_step"]
    line["launch_tax"] = {"batch": head["batch"], "graph_ms": round(ge, 4), "eager_ms": round(ee, 4),
                          "eager_kernels_per_step": n_k, "tau_us": round((ee - ge) / max(n_k - 1, 1) * 1e3, 3),
                          "speedup": round(ee / ge, 4)}
    # kernels of this library launched inside the timed regions (graph replays:
    # the graph's kernel nodes plus the staging kernel per step)
    line["gpu_launches"] = int(sum(run["kernels_per_step"] * K for x in [r] + extra for run in x["runs"]))
    if r["prefill"]:
        tfl, tsrc = tensor_peak()
        line["prefill"] = {"what": "time to first token: one prompt through prefill() (tensor-core passes of "
                                   "128 tokens, BF16 high/low activations), best of 3",
                           "runs": r["prefill"], "peak_tflops": tfl, "peak_source": tsrc,
                           "frac_of_peak": [round(x["achieved_tflops"] / tfl, 4) for x in r["prefill"]]}
    if r["runs"][0]["clocks"]:
        line["clocks"] = r["runs"][0]["clocks"]
    if r["e2e"]:
        e = dict(r["e2e"])
        e["value"] = round(e["value"] * world, 2)
        line["e2e"] = e
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(r["wl"], B)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def main_reference(args):
    """The oracle, as it stands, on this host's cores, for the same workload.
    Each step is a bounded sample sized so that warm-up plus steps take about
    two minutes: the oracle's own row-chunked projection over a slice of one
    layer's gate/up rows, its cost per weight byte extrapolated to the whole
    step's algorithmic bytes (weights + KV read)."""
    from oracle.decode import matmul
    from synth import raw_numpy

    wl = WORKLOADS[args.workload]
    cfg = wl.model
    B = args.batch or wl.batches[0]
    n = max(1, args.steps + args.warmup)
    per_step_s = max(0.05, 120.0 / n)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = SynthModel(cfg, wl.seed, device=dev, cache=False).get("w_gu", 0)
    gu = {k: raw_numpy(v) for k, v in t.items()}
    x = np.random.default_rng(0).normal(size=(B, cfg.hidden))
    wbytes_row = cfg.hidden * (1 if cfg.weight_dtype == "fp8" else 2)
    rows = 64
    while True:                                   # size the slice to the per-step budget
        sl = {k: v[:rows] for k, v in gu.items()}
        t0 = time.perf_counter()
        matmul(sl, x)
        dt = time.perf_counter() - t0
        if dt > per_step_s / 2 or rows >= gu["w"].shape[0]:
            break
        rows = min(gu["w"].shape[0], rows * 2)
    ctx = random_contexts(B, wl.context[0], wl.context[1], wl.seed + 2000)
    step_b = ledger.step_bytes(cfg, ctx)
    sl = {k: v[:rows] for k, v in gu.items()}
    for _ in range(args.warmup):
        matmul(sl, x)
    vals = []
    t_all = time.perf_counter()
    for _ in range(args.steps):
        t0 = time.perf_counter()
        matmul(sl, x)
        dt = time.perf_counter() - t0
        vals.append(B / (dt / (rows * wbytes_row) * step_b))
    wall = time.perf_counter() - t_all
    v = float(np.mean(vals))
    threads = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
    cores = int(threads) if threads else (os.cpu_count() or 1)
    line = {"impl": "reference", "metric": METRIC,
            "value": round(v, 6), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(wall / max(args.steps, 1) * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{wl.key}: {wl.description}", "model": cfg.name, "batch": B},
            "cpu_baseline": {"value": round(v, 6), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"per step: the oracle's fp64 projection over {rows} rows of layer 0's "
                                       f"gate/up matrix for {B} row(s), cost per weight byte scaled to the "
                                       f"step's {step_b / 1e9:.2f} GB of algorithmic bytes"},
            "e2e": {"value": round(v, 6), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
