#!/usr/bin/env python
"""Decode / prefill throughput of the decode path on one GB300 (sm_103a), through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--workload llama8b_bf16_1seq] [--no-cpu-baseline]

Workload (default): the Llama-3-8B-shaped BF16 model (32 layers, d 4096, 32/8 heads, head_dim
128, n_ff 14336, vocab 128256, seeded synthetic weights), one sequence, a 512-token prompt
prefilled as one ubatch into an F16 KV cache of 4096 cells, then greedy decode steps from
context 513. A timed "step" is one decode step: one token through all 32 layers, the output
matrix and the device argmax, driven through llm_decode / llm_get_argmax_ith. `value` is decode
tokens/s (CUDA events on the library's stream around K steps); prefill tokens/s is reported
beside it. The weights (15 GB per step) exceed L2, so no flush is needed between steps.

N > 1 (torchrun): replicas only: every rank runs the same workload on its own GPU (independent
sequences, no collective on the data path); a gloo barrier brackets the timed region and the
slowest rank's time is used. value = tokens of all ranks / that time.

--impl reference times the CPU oracle (numpy float64) on a bounded sample of the same workload
on the host cores (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tok/s & prefill tok/s on 1×GB300; decode HBM GB/s vs ~8 TB/s peak"
GEMV_TRAFFIC = {"llama8b_bf16_1seq": 109.16e6}


def _env_int(k, d):
    try:
        return int(os.environ.get(k, d))
    except ValueError:
        return d


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.rows = []
        self.proc = None
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([s.strip() for s in line.split(",")])

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in self.rows if len(r) > 2 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) > 2 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in self.rows:
            for i, n in enumerate(names):
                if len(r) > 5 + i and r[5 + i].lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(self.rows)}


# ------------------------------------------------------------------------------- oracle sample
class OracleSampler:
    """Times the CPU oracle on a bounded sample of one decode step.

    Sample: the oracle's float64 projections of one token (rms_norm, then each of the seven
    matrices of layer 0 and the output matrix, dequantised from storage as the oracle does) over
    the first ceil(frac * rows) rows of every matrix. One decode step is extrapolated as
    (n_layer x layer sample + output sample) / frac."""

    def __init__(self, w, frac: float):
        import torch
        import synthetic as S
        self.w, self.frac = w, frac
        hp = w.hp
        self.mats = []
        specs = [n for n in S.tensor_specs(hp) if n[0].startswith("blk.0.")]
        for name, shape in specs + [("output.weight", (hp.n_embd, hp.n_vocab))]:
            if name.endswith("_norm.weight"):
                continue
            r = max(1, int(math.ceil(frac * shape[1])))
            wt = S.types_for(name, w.types)
            dev = "cuda" if torch.cuda.is_available() else "cpu"
            t = S.weight_bytes(w.weight_seed, name, shape, wt, dev)[:r].cpu()
            raw = t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()
            self.mats.append((name, wt, shape[0], raw))
        self.rng = np.random.default_rng(0)
        self.desc = (f"oracle float64 projections of one token over the first {frac:.4g} of the rows "
                     f"of layer 0's seven matrices and of the output matrix (dequantised from "
                     f"storage), extrapolated to {hp.n_layer} layers + output = one decode step")

    def step(self):
        """Returns (extrapolated seconds of one decode step, wall seconds of the sample)."""
        import oracle
        hp = self.w.hp
        g = np.ones(hp.n_embd)
        t_layer = t_out = 0.0
        for name, wt, ne0, raw in self.mats:
            x = self.rng.standard_normal((1, ne0))
            t0 = time.perf_counter()
            if ne0 == hp.n_embd:
                x = oracle.rms_norm(x, g, hp.rms_eps)
            y = oracle.linear(x, oracle.decode_weight(raw, wt, ne0))
            dt = time.perf_counter() - t0
            assert np.all(np.isfinite(y))
            if name == "output.weight":
                t_out += dt
            else:
                t_layer += dt
        return (hp.n_layer * t_layer + t_out) / self.frac, t_layer + t_out


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


# ------------------------------------------------------------------------------- GPU arm
def run_gpu(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    import synthetic as S
    from transformer_decode_kv_gb300 import Context, LIB_PATH
    from transformer_decode_kv_gb300 import build as B

    if not os.path.exists(LIB_PATH):
        B.build()
    torch.cuda.set_device(local_rank)
    w = S.WORKLOADS[args.workload]
    hp = w.hp
    stream = torch.cuda.Stream()
    NS = w.n_seq                                        # sequences decoded together
    ctx = Context(hp, n_ctx=w.n_ctx, n_seq_max=NS, type_k=w.type_kv, type_v=w.type_kv,
                  n_batch=max(w.n_batch, w.n_prompt) if NS == 1 else w.n_batch, n_ubatch=w.n_ubatch,
                  stream=stream.cuda_stream, fused_step=args.fused_step)
    for name, wt, shape, t in S.model_weights(hp, w.weight_seed, w.types, "cuda"):
        if ctx.load_weight(name, wt, shape, t) != 0:
            raise RuntimeError(ctx.last_error())
        del t
    if ctx.weights_ready() != 0:
        raise RuntimeError(ctx.last_error())
    torch.cuda.empty_cache()
    prompts = [S.prompt_tokens(w.prompt_seed_of(s) + 977 * rank if NS > 1 else w.prompt_seed + 97 * rank,
                               w.n_prompt, hp.n_vocab).numpy() for s in range(NS)]
    prompt = prompts[0]

    def prefill():
        """Every sequence's prompt, in calls of at most n_batch tokens; the last token of each
        sequence is the only output."""
        if NS == 1:
            return ctx.decode(prompt)
        for s in range(NS):
            for i0 in range(0, w.n_prompt, ctx.n_batch):
                chunk = prompts[s][i0:i0 + ctx.n_batch]
                flags = [0] * len(chunk)
                if i0 + len(chunk) == w.n_prompt:
                    flags[-1] = 1
                r = ctx.decode(chunk, seq_ids=[[s]] * len(chunk), logits=flags)
                if r != 0:
                    return r
        return 0

    def barrier():
        if world > 1:
            dist.barrier()

    # ---- prefill: the prompt as one batch (split into n_ubatch ubatches), timed with events
    pre_times = []
    for rep in range(3 if NS == 1 else 2):
        ctx.seq_rm(-1, -1, -1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        r = prefill()
        e1.record(stream)
        torch.cuda.synchronize()
        if r != 0:
            raise RuntimeError(f"prefill failed {r}: {ctx.last_error()}")
        if rep > 0:
            pre_times.append(e0.elapsed_time(e1) / 1e3)
    prefill_s = float(np.median(pre_times))
    tok0 = ctx.get_argmax_ith(-1) if NS == 1 else [ctx.get_argmax_ith(-1)] * NS

    seq_rows = [[s] for s in range(NS)]

    def decode_steps(n, tok):
        """n greedy steps: one token per sequence each, device argmax read back each step."""
        for _ in range(n):
            if NS == 1:
                if ctx.decode([tok]) != 0:
                    raise RuntimeError(ctx.last_error())
                tok = ctx.get_argmax_ith(-1)
            else:
                if ctx.decode(tok, seq_ids=seq_rows, logits=[1] * NS) != 0:
                    raise RuntimeError(ctx.last_error())
                tok = [ctx.get_argmax_ith(i) for i in range(NS)]
        return tok

    K, W = args.steps, args.warmup
    if NS * (w.n_prompt + max(K, W)) > ctx.n_ctx:
        raise SystemExit(f"--steps/--warmup exceed the cache ({ctx.n_ctx} cells)")
    decode_steps(W, tok0)
    ctx.seq_rm(-1, w.n_prompt, -1)                      # back to the prompt context
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        decode_steps(K, tok0)
        e1.record(stream)
        torch.cuda.synchronize()
    barrier()
    dec_s = e0.elapsed_time(e1) / 1e3
    if world > 1:
        t = torch.tensor([dec_s, prefill_s], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dec_s, prefill_s = float(t[0]), float(t[1])

    # ---- per-kernel timing over the same steps (roofline of the dominant kernel)
    ctx.seq_rm(-1, w.n_prompt, -1)
    ctx.kernel_timing(True)
    decode_steps(K, tok0)
    ctx.kernel_timing(False)
    ks = ctx.kernel_stats()

    # ---- end to end: host token in, host argmax out, wall clock around K steps
    ctx.seq_rm(-1, w.n_prompt, -1)
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    decode_steps(K, tok0)
    e2e_s = time.perf_counter() - t0
    if world > 1:
        t = torch.tensor([e2e_s], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_s = float(t[0])
    # ---- the device sampler chain on the last logits row (top-k 40, top-p 0.95, min-p 0.05,
    # temperature 0.8, repeat penalty 1.1 over the last 64 tokens): host call to token, per call
    n_s = 32
    pen = list(prompt[-64:])
    ctx.sample_ith(-1, top_k=40, top_p=0.95, min_p=0.05, temperature=0.8, repeat_penalty=1.1,
                   penalty_tokens=pen, u=0.5)
    t0 = time.perf_counter()
    for i in range(n_s):
        if ctx.sample_ith(-1, top_k=40, top_p=0.95, min_p=0.05, temperature=0.8, repeat_penalty=1.1,
                          penalty_tokens=pen, u=(i + 0.5) / n_s) < 0:
            raise RuntimeError(ctx.last_error())
    sample_us = (time.perf_counter() - t0) / n_s * 1e6
    perf = ctx.perf()
    ctx.free()
    return dict(w=w, dec_s=dec_s, prefill_s=prefill_s, e2e_s=e2e_s, ks=ks, clk=clk.summary(),
                perf=perf, sample_us=sample_us)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="llama8b_bf16_1seq")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fused-step", action="store_true",
                    help="one-token steps as the single persistent step kernel instead of the "
                         "per-op kernel sequence (for comparison)")
    ap.add_argument("--type-kv", default="", choices=["", "f32", "f16", "q8_0"],
                    help="KV cache type instead of the workload's own (f16 unless it says otherwise)")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling aid: run the workload's shape with only this many layers "
                         "(a small case for ncu captures; not a bench number)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank, world = _env_int("RANK", 0), _env_int("WORLD_SIZE", 1)
    local_rank = _env_int("LOCAL_RANK", 0)
    import dataclasses
    import synthetic as S
    w = S.WORKLOADS[args.workload]
    if args.layers:
        w = dataclasses.replace(w, hp=dataclasses.replace(w.hp, n_layer=args.layers))
        S.WORKLOADS[args.workload] = w
    if args.type_kv:
        w = dataclasses.replace(w, type_kv={"f32": 0, "f16": 1, "q8_0": 8}[args.type_kv])
        S.WORKLOADS[args.workload] = w
    config = {"workload": args.workload, "description": w.description, "sequences": w.n_seq,
              "prompt_tokens": w.n_prompt, "decode_steps_timed": args.steps,
              "n_ctx": w.n_ctx, "kv_cache": {0: "f32", 1: "f16", 8: "q8_0"}[w.type_kv],
              "l2": "inputs larger than L2: every decode step streams all weights (no flush)",
              "parallelism": "replicas" if args.gpus > 1 else "single",
              "decode_path": "persistent step kernel" if args.fused_step else "per-op kernels (graph)"}
    if args.layers:
        config["profiling_case_layers"] = args.layers

    if args.impl == "reference":
        if rank != 0:
            return
        budget = 150.0                                   # seconds for the whole run
        cal = OracleSampler(w, 1.0 / 256)
        cal.step()
        _, wall = cal.step()
        frac = budget / max(1, args.steps + args.warmup) / max(wall * 256.0, 1e-9)
        frac = min(1.0 / 4, max(1.0 / 1024, frac))
        smp = OracleSampler(w, frac)
        desc = smp.desc
        times = []
        for i in range(args.warmup + args.steps):
            s, _ = smp.step()
            if i >= args.warmup:
                times.append(s)
        step_s = float(np.mean(times))
        v = 1.0 / step_s
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tok/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "cpu_baseline": {"value": v, "unit": "tok/s", "cores": cpu_cores(), "kind": "oracle",
                                 "sample": desc},
                "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if args.gpus > 1 or world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo")
    res = run_gpu(args, rank, world, local_rank)
    if rank != 0:
        return
    hp = w.hp
    K = args.steps
    dec_tps = world * w.n_seq * K / res["dec_s"]
    pre_tps = world * w.n_seq * w.n_prompt / res["prefill_s"]
    hbm_peak, bf16_peak, peak_src = measured_peaks()
    ks = res["ks"]
    # decode step algorithmic bytes: every class's bytes over the K steps
    step_bytes = sum(v["bytes"] for v in ks.values()) / max(1, K)
    # the dominant kernel: the one-token step kernel, or the GEMV class of the per-op sequence
    dom = max((k for k in ks if ks[k]["launches"]), key=lambda k: ks[k]["ms"])
    g = ks[dom]
    # DRAM bytes (read + written) per launch of the per-layer decode GEMVs of this workload, from
    # one ncu capture of the current kernel (profiles/gemv_swiglu_llama8b_bf16.md: the mean of the
    # Q/K/V, output, gate/up and down launches of a layer)
    traffic = GEMV_TRAFFIC.get(args.workload) if dom == "linear_gemv" and not args.layers else None
    achieved = g["bytes"] / (g["ms"] / 1e3) / 1e9 if g["ms"] > 0 else 0.0
    lm = ks.get("lm_head", {"ms": 0, "bytes": 0})
    line = {
        "metric": METRIC, "value": dec_tps, "unit": "tok/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": res["dec_s"] / K * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 weights; decode f32 activations, prefill f16 GEMM operands; f32 accumulation",
        "data": "synthetic (seeded random weights and prompt)", "config": config,
        "prefill_tok_s": pre_tps, "prefill_ms": res["prefill_s"] * 1e3,
        "sampler_us_per_call": res["sample_us"],
        "decode_hbm_gbs": step_bytes * K / res["dec_s"] / 1e9,
        "decode_step_algorithmic_bytes": step_bytes,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm_peak,
                     "unit": "GB/s", "frac": achieved / hbm_peak, "traffic": traffic,
                     "algorithmic_bytes_per_launch": g["bytes"] / max(1, g["launches"]),
                     "peak_source": peak_src,
                     "launches": g["launches"], "avg_launch_us": g["ms"] * 1e3 / max(1, g["launches"])},
        "kernel_share": {k: v["ms"] / max(1e-9, sum(x["ms"] for x in ks.values())) for k, v in ks.items()
                         if v["launches"]},
        "clocks": res["clk"],
        "e2e": {"value": world * w.n_seq * K / res["e2e_s"], "unit": "tok/s",
                "h2d_bytes_per_step": 4 * w.n_seq, "d2h_bytes_per_step": 8 * w.n_seq},
        "gpu_launches": int(sum(v["launches"] for v in ks.values()) / max(1, K)) * K,
    }
    if not args.no_cpu_baseline:
        try:
            smp = OracleSampler(w, 1.0 / 8)
            s = min(smp.step()[0] for _ in range(2))
            line["cpu_baseline"] = {"value": 1.0 / s, "unit": "tok/s", "cores": cpu_cores(),
                                    "kind": "oracle", "sample": smp.desc}
        except Exception as e:  # the GPU number stands without it
            line["cpu_baseline"] = {"value": None, "unit": "tok/s", "cores": cpu_cores(),
                                    "kind": "oracle", "sample": f"failed: {e}"}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
