#!/usr/bin/env python3
"""Benchmark of the combined lookahead decode step (one JSON line on rank 0).

Workload (default ``7b``): a Llama-2-7B-shaped decoder (32 layers, d 4096,
32 heads x 128, SwiGLU FFN 11008, vocab 32000), random-init bf16 weights
N(0, 0.02), batch 1, a 512-token Zipf(1.1) prompt with planted repeated
16-token spans, lookahead W=15 N=5 G=15 (T = 121 rows per step), greedy.
The pages' own settings for 7B (Key points); synthetic data stands in for
their chat/code suites.

A "step" is one ``la_step``: one combined decode step (row assembly, the
32-layer forward over 121 rows, LM head + argmax, verification, n-gram
harvest, KV commit, token readback).  W warm-up steps, then exactly K timed
steps, each bracketed by CUDA events on the library's stream; when a
generation reaches its configured length (256 new tokens) the prompt is
prefilled again outside the step timers.  Weights (13.2 GB) exceed L2, so no
flush is needed between steps.

value      effective tokens/s = tokens emitted by the K steps / their device time
e2e        tokens/s of ``la_generate`` (host prompt -> host tokens, prefill and
           every step's token readback inside the wall-clock region)
roofline   the tcgen05 weight-streaming GEMM kernel: algorithmic bytes / its
           event-timed duration, vs the measured HBM copy bandwidth
speedup    vs the same library's plain greedy step (W = G = 0)
cpu_baseline / --impl reference: the CPU oracle, timed on a bounded sample
           (1-layer slice of the same model, full widths) and scaled to the
           full depth by the FLOP ratio.
N > 1: independent replicas (the path does not shard); value sums ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import la_inputs as I  # noqa: E402

GEN_TOKENS = {"tiny": 64, "7b": 256, "13b": 256, "34b": 512}
PRESEED = {"34b": True}
SAMPLE_SEED = 7  # uniform stream of the sampling verification (--sample)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="7b", choices=list(I.MODELS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="use only the first L decoder layers (small cases for profiler captures)")
    ap.add_argument("--wng", default="",
                    help="W,N,G to use instead of the workload's lookahead settings")
    ap.add_argument("--preseed", default="auto", choices=["auto", "on", "off"],
                    help="seed the n-gram pool with the prompt's n-grams (auto: the workload's setting)")
    ap.add_argument("--attn", default="auto", choices=["auto", "mma", "tc"],
                    help="the step's attention kernel: tc (tcgen05 + TMA, LA_ATTN_TC; needs W + N - 2 <= 31 and "
                         "max_seq <= 4096), mma (mma.sync, the library's default), or auto (tc where it applies, "
                         "else mma; the lookahead and greedy decoders always use the same one)")
    ap.add_argument("--micro", action="store_true",
                    help="instead of the benchmark line: the attention and n-gram pool micro-benchmarks")
    ap.add_argument("--sample", type=float, default=0.0,
                    help="sampling verification at this temperature (0: greedy verification); the "
                         "comparison decoder then samples too, and the output is lossless in distribution "
                         "instead of token for token")
    ap.add_argument("--top-k", type=int, default=0,
                    help="with --sample: restrict each row's distribution to its top-k tokens (0: all)")
    ap.add_argument("--top-p", type=float, default=1.0,
                    help="with --sample: then to the leading tokens holding this share of their weight (1: all)")
    ap.add_argument("--batch-sweep", action="store_true",
                    help="instead of the benchmark line: one JSON line per (W,N,G,batch) of batched decoding "
                         "(several sequences in one forward pass per step, batch x T <= 128 rows)")
    ap.add_argument("--batch-only", type=int, default=0,
                    help="with --batch-sweep: only the points of this many sequences (0: every point)")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the benchmark line: one JSON line per (W,N,G) of a sweep, plus "
                         "the prompt-lookup mode (W=0, G>0, pool seeded from the prompt) and greedy")
    return ap.parse_args()


def lookahead_of(args):
    """(W, N, G, preseed) of a run: the workload's, or the --wng / --preseed overrides."""
    W, N, G = I.LOOKAHEAD[args.workload]
    if args.wng:
        W, N, G = (int(x) for x in args.wng.split(","))
    pre = PRESEED.get(args.workload, False) if args.preseed == "auto" else args.preseed == "on"
    return W, N, G, pre


def attn_tc_applies(W, N, max_seq):
    """Whether the tcgen05 attention (LA_ATTN_TC) serves this window: every
    step row within 31 positions of P, max_seq <= 4096."""
    return (W + N - 2 if W > 0 else N - 1) <= 31 and max_seq <= 4096


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


def step_model(cfg, T, P):
    """Algorithmic bytes and FLOPs of one step at cache length P (bf16)."""
    w_bytes = cfg.streamed_params() * 2 + T * cfg.d_model * 2
    kv_read = 2 * cfg.n_layers * P * cfg.d_kv * 2
    kv_write = 2 * cfg.n_layers * cfg.d_kv * 2 * 5
    flops = 2 * cfg.streamed_params() * T + 4 * T * P * cfg.n_heads * cfg.head_dim * cfg.n_layers
    return w_bytes + kv_read + kv_write, flops


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None

    def stop(self):
        if not self.p:
            return None
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
            out, _ = self.p.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(n):
    rank, world = int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if n > 0 else "gloo"
        dist.init_process_group(backend)
    return rank, world


def aggregate(tokens: float, seconds: float, device=None):
    """Sum of tokens and max of seconds over ranks (replicas)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return tokens, seconds
    t = torch.tensor([tokens], dtype=torch.float64, device=device)
    s = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    dist.all_reduce(s, op=dist.ReduceOp.MAX)
    return float(t.item()), float(s.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------- GPU arm

def build_model(cfg, dtype):
    import torch
    import lossless_lookahead_decoding_gb300 as LA
    # fp32 draws, rounded to bf16 on the device (round-to-nearest-even, the
    # same values la_inputs.bf16_round gives on the host)
    return LA.device_weights(cfg, I.iter_weights(cfg, 0, bf16=False), dtype)


def timed_steps(dec, prompt, gen_tokens, warmup, steps):
    """W warm-up + K timed steps; returns (tokens, per-step device ms, wall s, accept list)."""
    import torch
    st = dec.stream
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    dec.prefill(prompt)
    emitted = 0
    for _ in range(warmup):
        if emitted >= gen_tokens:
            dec.prefill(prompt)
            emitted = 0
        emitted += len(dec.step())
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    tok, acc = 0, []
    t0 = time.perf_counter()
    for i in range(steps):
        if emitted >= gen_tokens:
            dec.prefill(prompt)
            emitted = 0
        ev[i][0].record(st)
        n = len(dec.step())
        ev[i][1].record(st)
        emitted += n
        tok += n
        acc.append(n)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier()
    return tok, [a.elapsed_time(b) for a, b in ev], wall, acc


def run_ours(args, rank, world):
    import torch
    import lossless_lookahead_decoding_gb300 as LA
    from lossless_lookahead_decoding_gb300 import build as B
    B.build()
    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    cfg = I.MODELS[args.workload]
    if args.layers:
        cfg = cfg.sliced(args.layers)
    W, N, G, pre = lookahead_of(args)
    T = 1 + (W + G) * (N - 1)
    gen = GEN_TOKENS[args.workload]
    prompt = I.make_prompt(args.workload)
    max_seq = len(prompt) + gen + W + N + 16
    flags = LA.LA_PRESEED_PROMPT if pre else 0
    attn = getattr(args, "attn", "mma")
    use_tc = attn == "tc" or (attn == "auto" and attn_tc_applies(W, N, max_seq))
    attn_flag = LA.LA_ATTN_TC if use_tc else 0
    flags |= attn_flag
    t_gen = time.perf_counter()
    dw = build_model(cfg, LA.LA_BF16)
    torch.cuda.synchronize()
    t_gen = time.perf_counter() - t_gen

    la = LA.Decoder(cfg, dw, LA.LA_BF16, W, N, G, max_seq, flags=flags)
    gr = LA.Decoder(cfg, dw, LA.LA_BF16, 0, 2, 0, max_seq, flags=attn_flag)
    sample = getattr(args, "sample", 0.0)
    if sample > 0:
        for d in (la, gr):
            d.set_sampling(sample, SAMPLE_SEED, top_k=getattr(args, "top_k", 0), top_p=getattr(args, "top_p", 1.0))
    clocks = Clocks(local)
    clocks.start()
    tok, step_ms_l, wall, acc = timed_steps(la, prompt, gen, args.warmup, args.steps)
    g_tok, g_step_ms_l, g_wall, _ = timed_steps(gr, prompt, gen, args.warmup, args.steps)
    ms, greedy_ms = sum(step_ms_l), sum(g_step_ms_l)
    clk = clocks.stop()
    kernels = la.stats()["kernels_per_step"]

    # losslessness on the benchmark workload: one full generation each way
    la_out = la.generate(prompt, gen)
    gr_out = gr.generate(prompt, gen)
    # under sampling the two decoders draw different uniforms: equal in
    # distribution, not token for token (checked by the tests, not here)
    lossless = bool(np.array_equal(la_out, gr_out)) if sample <= 0 else None
    full_steps = la.stats()["steps"]

    # e2e through la_generate (host prompt in, host tokens out)
    e2e = None
    if not args.no_e2e:
        reps = 3
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            out = la.generate(prompt, gen)
        torch.cuda.synchronize()
        e2e_s = time.perf_counter() - t0
        steps_e2e = la.stats()["steps"]
        e2e = {"value": reps * len(out) / e2e_s, "unit": "tokens/s",
               "h2d_bytes_per_step": round(4 * len(prompt) / max(steps_e2e, 1), 1),
               "d2h_bytes_per_step": 104,
               "what": f"la_generate({len(prompt)}-token host prompt, {gen} new tokens) incl. prefill"}
    la.close()
    gr.close()

    # per-kernel-class timing (separate profiled pass: events around launches)
    prof_dec = LA.Decoder(cfg, dw, LA.LA_BF16, W, N, G, max_seq, flags=flags | LA.LA_PROFILE | LA.LA_NO_GRAPH)
    if sample > 0:
        prof_dec.set_sampling(sample, SAMPLE_SEED, top_k=getattr(args, "top_k", 0),
                              top_p=getattr(args, "top_p", 1.0))
    prof_warm, prof_steps = 2, min(args.steps, 64)
    timed_steps(prof_dec, prompt, gen, prof_warm, prof_steps)
    prof = prof_dec.profile()
    prof_dec.close()
    n_prof = prof_warm + prof_steps  # every step of the pass is profiled (warm-up included)

    tot_tok, tot_s = aggregate(tok, ms / 1e3, device=torch.device("cuda", local))
    g_tot_tok, g_tot_s = aggregate(g_tok, greedy_ms / 1e3, device=torch.device("cuda", local))
    if rank != 0:
        return None
    peaks = load_peaks()
    gemm = [v for k, v in prof.items() if k.startswith("gemm_") and k != "gemm_epilogue"]
    g_bytes = sum(v["bytes"] for v in gemm)
    g_ms = sum(v["total_ms"] for v in gemm)
    g_launch = sum(v["launches"] for v in gemm)
    achieved = g_bytes / (g_ms / 1e3) / 1e9
    traffic = read_traffic(args.workload)
    roofline = {"bound": "hbm", "kernel": "k_gemm_tc (all projection/MLP/LM-head GEMMs)",
                "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_src": peaks["src"],
                "traffic": traffic, "algorithmic_bytes_per_launch": round(g_bytes / max(g_launch, 1)),
                "avg_launch_us": round(1e3 * g_ms / max(g_launch, 1), 2)}
    P_mid = len(prompt) - 1 + gen // 2
    sbytes, sflops = step_model(cfg, T, P_mid)
    t_roof = max(sbytes / (peaks["hbm_gbs"] * 1e9), sflops / (peaks["bf16_tflops"] * 1e12))
    step_ms = ms / args.steps
    g_step_ms = greedy_ms / args.steps
    acc_per_step = tok / args.steps
    value = tot_tok / tot_s
    g_value = g_tot_tok / g_tot_s
    out = {
        "metric": "effective tokens/s & step latency at batch 1 vs step roofline; accepted tok/step",
        "value": round(value, 2), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (random-init weights)",
        "config": {"workload": f"{args.workload}: {cfg.n_layers}L d{cfg.d_model} {cfg.n_heads}x{cfg.head_dim} "
                               f"(kv {cfg.n_kv_heads}) ffn{cfg.ffn} V{cfg.vocab} bf16, prompt {len(prompt)}, "
                               f"gen {gen}, W{W} N{N} G{G}, T={T} rows" + (", prompt-seeded pool" if pre else "")
                               + (", tcgen05 attention" if attn_flag else ""),
                   "global_batch": 1, "seq_len": max_seq, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2 (weights {cfg.streamed_params() * 2 / 1e9:.1f} GB stream every step)"},
        "accepted_tokens_per_step": round(acc_per_step, 4),
        "accept_hist": {str(k): acc.count(k) for k in range(1, N + 1)},
        "step_latency_ms": {"median": round(float(np.median(step_ms_l)), 4),
                            "p10": round(float(np.percentile(step_ms_l, 10)), 4),
                            "p90": round(float(np.percentile(step_ms_l, 90)), 4), "mean": round(step_ms, 4)},
        "wall_s_timed": round(wall, 3),
        "greedy": {"value": round(g_value, 2), "unit": "tokens/s", "ms_per_step": round(g_step_ms, 4)},
        "speedup_vs_greedy": round(value / g_value, 4),
        # the cost of the T - 1 extra rows: lookahead step time minus the
        # same library's greedy step time over the same prompt and steps
        "lookahead_premium_ms": round(step_ms - g_step_ms, 4),
        "lossless_vs_greedy": lossless, "full_generation_steps": full_steps,
        "verification": ({"mode": "sampling", "temperature": sample, "top_k": getattr(args, "top_k", 0),
                          "top_p": getattr(args, "top_p", 1.0)}
                         if sample > 0 else {"mode": "greedy"}),
        "step_roofline": {"t_roof_ms": round(t_roof * 1e3, 4), "frac": round(t_roof * 1e3 / step_ms, 4),
                          "bytes": sbytes, "flops": sflops, "P": P_mid, "peak_src": peaks["src"]},
        "kernel_profile_steps": n_prof,
        "kernel_profile": {k: {"launches": v["launches"], "ms_per_step": round(v["total_ms"] / n_prof, 4),
                               "GB/s": round(v["bytes"] / max(v["total_ms"], 1e-9) / 1e6, 1)}
                           for k, v in prof.items()},
        "gpu_launches": kernels * args.steps,
        "kernels_per_step": kernels,
        "roofline": roofline,
        "clocks": clk,
        "weights_gen_s": round(t_gen, 1),
    }
    if e2e:
        out["e2e"] = e2e
    if not args.no_cpu_baseline and world == 1:
        out["cpu_baseline"] = cpu_baseline(cfg, args.workload, W, N, G, prompt, steps=2, preseed=pre)
    return out


# (W, N, G, prompt-seeded pool, diagonal levels) of the sweep: T = 1 + (W+G)(N-1) <= 128 rows
SWEEP = [(0, 2, 0, False, False),                                            # greedy
         (0, 3, 4, True, False), (0, 5, 4, True, False),                      # prompt lookup: prompt n-grams
         (5, 5, 5, False, False), (7, 5, 7, False, False), (10, 5, 10, False, False), (15, 5, 15, False, False),
         (15, 3, 15, False, False), (31, 3, 31, False, False), (20, 4, 20, False, False),
         (10, 7, 10, False, False), (15, 5, 15, True, False),
         # branch balance at T = 121 (W + G = 30, N = 5): lopsided to balanced
         (28, 5, 2, False, False), (25, 5, 5, False, False), (20, 5, 10, False, False),
         (10, 5, 20, False, False), (5, 5, 25, False, False), (2, 5, 28, False, False),
         # the other mask reading (LA_MASK_DIAG) at the same shapes
         (5, 5, 5, False, True), (7, 5, 7, False, True), (10, 5, 10, False, True), (15, 5, 15, False, True),
         (15, 3, 15, False, True), (20, 4, 20, False, True), (10, 7, 10, False, True)]


def run_sweep(args, rank, world):
    """One JSON line per (W, N, G, mask): step latency, accepted tokens/step,
    tokens/s, speedup over greedy and losslessness (same library, same
    prompt).  W = 0 with a prompt-seeded pool is the prompt-lookup mode."""
    import torch
    import lossless_lookahead_decoding_gb300 as LA
    from lossless_lookahead_decoding_gb300 import build as B
    B.build()
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    cfg = I.MODELS[args.workload]
    if args.layers:
        cfg = cfg.sliced(args.layers)
    gen = GEN_TOKENS[args.workload]
    prompt = I.make_prompt(args.workload)
    max_seq = len(prompt) + gen + max(w + n for w, n, _, _, _ in SWEEP) + 16
    dw = build_model(cfg, LA.LA_BF16)
    lines, ref_out, greedy_tps = [], None, None
    for W, N, G, pre, diag in SWEEP:
        flags = (LA.LA_PRESEED_PROMPT if pre else 0) | (LA.LA_MASK_DIAG if diag else 0)
        dec = LA.Decoder(cfg, dw, LA.LA_BF16, W, N, G, max_seq, flags=flags)
        tok, step_ms_l, _, _ = timed_steps(dec, prompt, gen, args.warmup, args.steps)
        out = dec.generate(prompt, gen)
        dec.close()
        tps = tok / (sum(step_ms_l) / 1e3)
        if ref_out is None:
            ref_out, greedy_tps = out, tps
        T = 1 + (W + G) * (N - 1)
        lines.append({"sweep": args.workload, "mode": "greedy" if W == 0 and G == 0 else
                      ("prompt-lookup" if W == 0 else "lookahead"), "W": W, "N": N, "G": G, "T": T,
                      "prompt_seeded_pool": pre, "mask": "diagonal levels" if diag else "columns",
                      "ms_per_step": round(float(np.mean(step_ms_l)), 4),
                      "accepted_tokens_per_step": round(tok / args.steps, 4), "tokens_per_s": round(tps, 2),
                      "speedup_vs_greedy": round(tps / greedy_tps, 4),
                      "lossless_vs_greedy": bool(np.array_equal(out, ref_out)), "steps": args.steps})
    return lines if rank == 0 else None


# (W, N, G, batch) of the batch sweep: batch x (1 + (W+G)(N-1)) <= 128 rows
BATCH_SWEEP = [(0, 2, 0, 1), (0, 2, 0, 2), (0, 2, 0, 4), (0, 2, 0, 8), (0, 2, 0, 16), (0, 2, 0, 32),
               (0, 2, 0, 64), (0, 2, 0, 128),
               (15, 5, 15, 1), (7, 5, 7, 1), (7, 5, 7, 2), (5, 5, 5, 3), (3, 5, 3, 5), (3, 4, 3, 6)]


def batch_points(only: int = 0):
    """The --batch-sweep points, or those of `only` sequences."""
    return [p for p in BATCH_SWEEP if not only or p[3] == only]


def run_batch_sweep(args, rank, world):
    """Batched decoding: per (W, N, G, batch), the step latency and the
    tokens/s of all sequences together (prompts of the workload's recipe,
    seeds 1..batch), the same end to end through la_generate_batch (host
    prompts in, prefill included, host tokens out), and whether sequence 0's
    tokens equal a batch-1 greedy context's on the same prompt."""
    import torch
    import lossless_lookahead_decoding_gb300 as LA
    from lossless_lookahead_decoding_gb300 import build as B
    B.build()
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    cfg = I.MODELS[args.workload]
    if args.layers:
        cfg = cfg.sliced(args.layers)
    n_steps = args.warmup + args.steps
    points = batch_points(getattr(args, "batch_only", 0))
    if not points:
        raise SystemExit(f"no --batch-sweep point has {args.batch_only} sequences")
    prompts = [I.make_prompt(args.workload, seed=1 + b) for b in range(max(b for *_, b in points))]
    max_seq = len(prompts[0]) + n_steps * 8 + 32
    dw = build_model(cfg, LA.LA_BF16)
    ref = LA.Decoder(cfg, dw, LA.LA_BF16, 0, 2, 0, max_seq)
    want = ref.generate(prompts[0], n_steps)  # one token per greedy step: enough for every point
    ref.close()
    lines = []
    for W, N, G, bsz in points:
        dec = LA.Decoder(cfg, dw, LA.LA_BF16, W, N, G, max_seq, batch=bsz)
        for b in range(bsz):
            dec.prefill_seq(b, prompts[b])
        out0, tok = [], 0
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for i in range(n_steps):
            k = i - args.warmup
            if k >= 0:
                ev[k][0].record(dec.stream)
            got = dec.step_batch()
            if k >= 0:
                ev[k][1].record(dec.stream)
                tok += sum(len(t) for t in got)
            out0.extend(got[0].tolist())
        torch.cuda.synchronize()
        # end to end through la_generate_batch: host prompts in (prefill
        # included), host tokens out, n_steps tokens per sequence
        t0 = time.perf_counter()
        outs = dec.generate_batch(prompts[:bsz], n_steps)
        torch.cuda.synchronize()
        e2e_s = time.perf_counter() - t0
        dec.close()
        ms = [a.elapsed_time(b) for a, b in ev]
        T = 1 + (W + G) * (N - 1)
        lines.append({"batch_sweep": args.workload, "W": W, "N": N, "G": G, "batch": bsz, "T": T,
                      "rows_per_pass": bsz * T, "ms_per_step": round(float(np.mean(ms)), 4),
                      "tokens_per_step": round(tok / args.steps, 4),
                      "tokens_per_s": round(tok / (sum(ms) / 1e3), 2),
                      "tokens_per_s_per_sequence": round(tok / bsz / (sum(ms) / 1e3), 2),
                      "e2e_tokens_per_s": round(sum(len(o) for o in outs) / e2e_s, 2),
                      "seq0_equals_batch1_greedy": bool(np.array_equal(np.array(out0[:len(want)], np.int32),
                                                                       want[:len(out0)])),
                      "steps": args.steps, "warmup": args.warmup, "data": "synthetic prompts, random-init weights"})
    return lines if rank == 0 else None


def _event_times(fn, reps, stream, before=None):
    """Device time (µs) of fn() per rep on stream, CUDA events around each;
    before() (e.g. an L2 flush) runs outside the timed region."""
    import torch
    ts = []
    for _ in range(reps):
        if before:
            before()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b) * 1e3)
    return ts


def run_micro(args, rank, world):
    """Attention micro-benchmark (32 heads x 128, 2048 cached tokens ~ N(0,1),
    the 121 rows of W=15 N=5 G=15 under the lookahead mask), cold (L2 flushed
    by a 256 MB write before each rep) and warm; n-gram pool micro-benchmark
    (4096 Zipf(1.1) keys x 20 4-grams inserted, then a bulk lookup of the
    4096 keys and a bulk insert of 2048 further n-grams).  One JSON line each."""
    import torch
    import lossless_lookahead_decoding_gb300 as LA
    from lossless_lookahead_decoding_gb300 import build as B
    B.build()
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    peaks = load_peaks()
    st = torch.cuda.Stream()
    lines = []
    # ---- attention
    H, hd, P, W, N, G = 32, 128, 2048, 15, 5, 15
    T = 1 + (W + G) * (N - 1)
    max_seq = P + 64
    inp = I.attention_bench_inputs(heads=H, head_dim=hd, ctx=P, rows=T)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().to(torch.bfloat16)
    kc = torch.zeros((H, max_seq, hd), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    kc[:, :P] = bf(inp["k_cache"])
    vc[:, :P] = bf(inp["v_cache"])
    q, ks, vs = bf(inp["q"]), bf(inp["k_step"]), bf(inp["v_step"])
    out = torch.empty((T, H * hd), dtype=torch.bfloat16, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()

    def attn():
        rc = LA.la_attention(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), ks.data_ptr(), vs.data_ptr(),
                             out.data_ptr(), H, H, hd, max_seq, P, W, N, G, st.cuda_stream)
        assert rc == 0, rc

    def flush_l2():
        with torch.cuda.stream(st):
            flush.zero_()

    for _ in range(3):
        attn()
    op = _event_times(attn, 10, st)
    by = 2 * P * H * hd * 2 + T * (2 * H * hd + 2 * H * hd) * 2
    roof_us = by / (peaks["hbm_gbs"] * 1e3)
    # kernel time: the attention + split-merge launches of decode steps at
    # P = 2048 inside a decoder (event pairs around them, LA_PROFILE): the
    # 32-layer 7B-width model (each layer's 33.6 MB of KV is evicted by the
    # other layers' weights: cold) and a 1-layer slice of it (KV stays in L2:
    # warm); synthetic Zipf prompt, random-init weights
    # (the mma.sync kernel + split merge, and the tcgen05 pair, LA_ATTN_TC)
    kern = {}
    for name, layers in (("cold", 0), ("warm", 1)):
        cfg = I.MODELS["7b"] if not layers else I.MODELS["7b"].sliced(layers)
        dw = build_model(cfg, LA.LA_BF16)
        prompt = I.zipf_tokens(P + 1, cfg.vocab, 1.1, 21)
        for suffix, extra in (("", 0), ("_tc", LA.LA_ATTN_TC)):
            dec = LA.Decoder(cfg, dw, LA.LA_BF16, W, N, G, P + 1 + 64,
                             flags=LA.LA_PROFILE | LA.LA_NO_GRAPH | extra)
            dec.prefill(prompt)
            dec.step()
            p0 = dec.profile()["attention"]  # cumulative since creation: prefill blocks included
            for _ in range(8):
                dec.step()
            p1 = dec.profile()["attention"]
            kern[name + suffix] = 1e3 * (p1["total_ms"] - p0["total_ms"]) / (p1["launches"] - p0["launches"])
            dec.close()
        del dw
        torch.cuda.empty_cache()
    lines.append({"micro": "attention", "config": f"{H}x{hd} heads, {P} cached tokens, W{W} N{N} G{G} ({T} rows)",
                  "us_cold": round(kern["cold"], 2), "us_warm": round(kern["warm"], 2),
                  "us_cold_tcgen05": round(kern["cold_tc"], 2), "us_warm_tcgen05": round(kern["warm_tc"], 2),
                  "frac_cold_tcgen05": round(roof_us / kern["cold_tc"], 4),
                  "algorithmic_bytes": by, "roofline_us": round(roof_us, 2), "peak_gbs": peaks["hbm_gbs"],
                  "frac_cold": round(roof_us / kern["cold"], 4),
                  "la_attention_call_us": round(float(np.median(op)), 1),
                  "note": "us_cold/us_warm: the mma.sync attention + split merge per layer inside a decoder at "
                          "P=2048 (the decode steps' P grows by the accepted tokens); *_tcgen05: the same for the "
                          "tcgen05 + TMA pair (LA_ATTN_TC) that bench.py's step runs; la_attention_call_us: the "
                          "standalone ABI op (mma.sync) incl. its table uploads, scratch allocation and "
                          "synchronisation"})
    # ---- n-gram pool
    Np, Gp, V = 5, 15, 32000
    keys, grams = I.pool_bench_inserts(4096, 20, V, Np - 1)
    pool = LA.la_pool_create(2 * 4096 + 64, Np, Gp, st.cuda_stream)
    dk = torch.from_numpy(keys).cuda()
    dg = torch.from_numpy(np.ascontiguousarray(grams)).cuda()
    torch.cuda.synchronize()
    t_fill = _event_times(lambda: LA.la_pool_insert(pool, dk.data_ptr(), dg.data_ptr(), len(keys)), 1, st)[0]
    uq = torch.from_numpy(np.unique(keys)).cuda()
    lo = torch.empty((len(uq), Gp, Np - 1), dtype=torch.int32, device="cuda")
    lc = torch.empty(len(uq), dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()

    def lookup():
        assert LA.la_pool_lookup(pool, uq.data_ptr(), len(uq), lo.data_ptr(), lc.data_ptr()) == 0

    for _ in range(3):
        lookup()
    t_look = _event_times(lookup, 20, st)
    k2, g2 = I.pool_bench_ngrams(2048, V, Np - 1)
    dk2, dg2 = torch.from_numpy(k2).cuda(), torch.from_numpy(np.ascontiguousarray(g2)).cuda()
    torch.cuda.synchronize()
    t_ins = _event_times(lambda: LA.la_pool_insert(pool, dk2.data_ptr(), dg2.data_ptr(), len(k2)), 5, st)
    look_bytes = len(uq) * (4 + Gp * (Np - 1) * 4 + 4)
    lines.append({"micro": "ngram_pool", "config": f"{len(uq)} keys x {Gp} {Np - 1}-grams, vocab {V}, Zipf(1.1)",
                  "fill_us": round(t_fill, 1), "fill_inserts": int(len(keys)),
                  "lookup_us": round(float(np.median(t_look)), 2), "lookup_keys": int(len(uq)),
                  "lookup_bytes": look_bytes,
                  "insert_us": round(float(np.median(t_ins)), 2), "insert_ngrams": int(len(k2)),
                  "note": "insert times include the status read-back of la_pool_insert"})
    LA.la_pool_destroy(pool)
    return lines if rank == 0 else None


def read_traffic(workload):
    """DRAM bytes per GEMM launch from the committed ncu summary, if it was
    taken on the current kernel source (else null)."""
    p = os.path.join(ROOT, "profiles", f"gemm_tc_{workload}_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    src = open(os.path.join(ROOT, "lossless_lookahead_decoding_gb300", "csrc", "gemm_tc.cu"), "rb").read()
    if d.get("gemm_tc_sha1") != hashlib.sha1(src).hexdigest():
        return None
    return d.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- CPU oracle

def oracle_sample(cfg, W, N, G, prompt, n_steps, preseed=False, threads=0):
    """Run n_steps oracle lookahead steps on a 1-layer slice of the model (the
    same bytes as the full model's embedding, layer 0 and LM head, full widths
    and vocabulary) after prefilling the prompt with all cores; the steps run
    on `threads` threads (0: all).  Returns (per-step seconds, tokens emitted
    per step, full-depth/slice FLOP ratio, threads used).  The full 7B-shaped
    oracle step (~1.6 TFLOP of plain fp32 loops, ~17 s on 16 host cores, and a
    ~7 TFLOP prefill) does not fit a bounded sample, hence the slice."""
    import oracle as O
    sl = cfg.sliced(1)
    full = I.make_weights(cfg, 0, bf16=True, layers=[0])  # same bytes as the full model's layer 0
    w = {k: (v[:1] if isinstance(v, list) else v) for k, v in full.items()}
    m = O.Model(sl, w)
    all_cores = O.threads()
    O.set_threads(all_cores)
    seq = O.Seq(m, len(prompt) + 8 * n_steps + W + N + 8)
    seq.prefill(prompt[:-1])
    k = O.Controller(W, N, G, cfg.vocab)
    k.init(prompt, seed=2, preseed=preseed)
    c, P = int(prompt[-1]), len(prompt) - 1
    used = threads if threads > 0 else all_cores
    O.set_threads(used)
    times, toks = [], []
    for _ in range(n_steps):
        tok, pos, vis = k.rows(c, P)
        t0 = time.perf_counter()
        _, amax = seq.step(P, tok, pos, vis, want_logits=False)
        times.append(time.perf_counter() - t0)
        emit, rows, _ = k.advance(amax)
        seq.commit(P, rows)
        P += len(emit)
        c = int(emit[-1])
        toks.append(len(emit))
    O.set_threads(all_cores)
    per_layer = (cfg.n_heads * cfg.head_dim * cfg.d_model * 2 + 2 * cfg.d_kv * cfg.d_model + 3 * cfg.ffn * cfg.d_model)
    head = cfg.vocab * cfg.d_model
    ratio = (cfg.n_layers * per_layer + head) / (per_layer + head)
    return times, toks, ratio, used


def oracle_rate(times, toks, ratio):
    """The oracle's tokens/s on the full-depth model, one definition for the
    CPU baseline and the reference arm: the tokens its own lookahead steps
    emitted on the sample / their measured time scaled by the full-depth /
    slice FLOP ratio (the step is matrix-vector work over every weight, so its
    time scales with the weight FLOPs)."""
    return sum(toks) / (float(np.sum(times)) * ratio)


def cpu_baseline(cfg, workload, W, N, G, prompt, steps=2, preseed=False):
    t_all, k_all, ratio, cores = oracle_sample(cfg, W, N, G, prompt, steps, preseed)
    t_one, k_one, _, _ = oracle_sample(cfg, W, N, G, prompt, 1, preseed, threads=1)
    v_all, v_one = oracle_rate(t_all, k_all, ratio), oracle_rate(t_one, k_one, ratio)
    return {"value": round(v_all, 5), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "value_1_thread": round(v_one, 5),
            "sample": f"{steps} oracle lookahead steps on {cores} threads and 1 step on 1 thread (T="
                      f"{1 + (W + G) * (N - 1)} rows each) on a 1-layer slice of the {workload} model (full widths "
                      f"and vocabulary, the model's own layer-0 bytes) after prefilling the {len(prompt)}-token "
                      f"prompt; measured {1e3 * float(np.mean(t_all)):.0f} ms/step ({cores} threads) and "
                      f"{1e3 * float(np.mean(t_one)):.0f} ms/step (1 thread), scaled x{ratio:.2f} (full-depth/slice "
                      f"weight FLOPs); tokens/step = the oracle's own ({sum(k_all)}/{len(k_all)}); the full-depth "
                      f"oracle step (~{float(np.mean(t_all)) * ratio:.0f} s) does not fit a bounded sample"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    cfg = I.MODELS[args.workload]
    W, N, G, pre = lookahead_of(args)
    prompt = I.make_prompt(args.workload)
    # every step is one oracle lookahead step on the 1-layer slice (bounded sample)
    times, toks, ratio, cores = oracle_sample(cfg, W, N, G, prompt, args.warmup + args.steps, pre)
    t, k = times[args.warmup:], toks[args.warmup:]
    value = oracle_rate(t, k, ratio)
    sample_ms = 1e3 * float(np.mean(t))
    return {"impl": "reference", "metric": "effective tokens/s & step latency at batch 1 vs step roofline; "
            "accepted tok/step", "value": round(value, 5), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sample_ms * ratio, 1),
            "ms_per_step_measured_sample": round(sample_ms, 1), "extrapolation_x": round(ratio, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (random-init weights)",
            "config": {"workload": args.workload, "global_batch": 1, "seq_len": len(prompt) + GEN_TOKENS[args.workload],
                       "parallelism": "cpu"},
            "accepted_tokens_per_step": round(sum(k) / len(k), 4),
            "cpu_baseline": {"value": round(value, 5), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"each of the {args.warmup} + {args.steps} steps is one oracle lookahead step "
                                       f"on a 1-layer slice of the {args.workload} model ({cores} threads), measured "
                                       f"{sample_ms:.0f} ms/step; ms_per_step and value are that time scaled "
                                       f"x{ratio:.2f} to the full depth (weight FLOPs), tokens/step the oracle's "
                                       f"own ({sum(k)}/{len(k)})"},
            "e2e": {"value": round(value, 5), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank, world = dist_setup(args.gpus if args.impl == "ours" else 0)
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    elif args.sweep:
        out = run_sweep(args, rank, world)
    elif args.batch_sweep:
        out = run_batch_sweep(args, rank, world)
    elif args.micro:
        out = run_micro(args, rank, world)
    else:
        out = run_ours(args, rank, world)
    if rank == 0 and out is not None:
        for line in out if isinstance(out, list) else [out]:
            print(json.dumps(line), flush=True)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
