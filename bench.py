#!/usr/bin/env python
"""Decode / prefill throughput of the decode path on one GB300 (sm_103a), through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--workload llama8b_bf16_1seq] [--no-cpu-baseline] [--no-extra]

Workload (default): the Llama-3-8B-shaped BF16 model (32 layers, d 4096, 32/8 heads, head_dim
128, n_ff 14336, vocab 128256, seeded synthetic weights), one sequence, a 512-token prompt
prefilled as one ubatch into an F16 KV cache of 4096 cells, then greedy decode steps from
context 513. A timed "step" is one decode step: one token through all 32 layers, the output
matrix and the device argmax, driven through llm_decode / llm_get_argmax_ith. `value` is decode
tokens/s (CUDA events on the library's stream around K steps); prefill tokens/s is reported
beside it. The weights (15 GB per step) exceed L2, so no flush is needed between steps.

After the headline line's measurements, the default run also measures the two other 8B
workloads, each in a fresh context (nothing reused): the 8192-token Q8_0 prompt with its 128
decode steps, and the 32-sequence run (32 x 2048-token prompts, 256 steps of 32 tokens with the
seq_rm after step 128). Their figures go under "extra" in the same JSON line.

N > 1 (torchrun): replicas only: every rank runs the same workload on its own GPU (independent
sequences, no collective on the data path); a gloo barrier brackets the timed region and the
slowest rank's time is used. value = tokens of all ranks / that time.

--impl reference times the CPU oracle (numpy float64) on a bounded sample of the same workload
on the host cores (rank 0 only).
"""
from __future__ import annotations

import argparse
import dataclasses
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
NOMINAL_HBM_GBS = 8000.0
# DRAM bytes (read + written) per launch of the per-layer decode GEMVs of the 8B BF16 workload:
# the mean over the Q/K/V, output, gate/up and down launches of a layer, from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum) of the GEMV kernels as they are now
GEMV_TRAFFIC = {"llama8b_bf16_1seq": 109.16e6}
EXTRA_WORKLOADS = ("llama8b_q8_0_8k", "llama8b_bf16_32seq")


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
        return {"hbm_gbs": d.get("hbm_gbs", 6800.0), "bf16_tflops": d.get("bf16_tflops", 1900.0),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", 1700.0), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running; each row is kept
    with the host time it arrived, so a summary can be restricted to a time window."""
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
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.perf_counter(), [s.strip() for s in line.split(",")]))

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    @staticmethod
    def _stats(rows):
        sm = [float(r[1]) for r in rows if len(r) > 2 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) > 2 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for i, n in enumerate(names):
                if len(r) > 5 + i and r[5 + i].lower() == "active":
                    reasons.add(n)
        return sm, mx, sorted(reasons)

    def summary(self, window=None):
        """Median SM clock, max clock and throttle reasons over the whole sampling period, and the
        number of samples that fell inside `window` (host perf_counter seconds, start and end)."""
        rows = [r for _, r in self.rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm, mx, reasons = self._stats(rows)
        out = {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
               "reasons": reasons, "samples": len(rows),
               "sampled_over": "the whole decode phase: warm-up, timed region, kernel-share re-run, e2e run"}
        if window is not None:
            inside = [r for t, r in self.rows if window[0] - 0.1 <= t <= window[1] + 0.1]
            out["samples_in_timed_region"] = len(inside)
            if inside:
                s2, _, r2 = self._stats(inside)
                out["sm_mhz_in_timed_region"] = float(np.median(s2)) if s2 else None
                out["reasons_in_timed_region"] = r2
        return out


# ------------------------------------------------------------------------- algorithmic work
# "llama.cpp Architecture", Example 13: bytes read per decode token (every weight once) and
# FLOPs per prompt token (2 per weight, plus the causal attention).

def _row_bytes(wtype: int, ne0: int) -> float:
    return {0: 4.0 * ne0, 1: 2.0 * ne0, 2: 2.0 * ne0, 8: ne0 / 32 * 34.0}[wtype]


def linear_weight_bytes(w) -> float:
    """Bytes of every matrix a decode step reads whole: the per-layer projections and the output
    matrix (the embedding table is read one row per token)."""
    import synthetic as S
    tot = 0.0
    for name, shape in S.tensor_specs(w.hp):
        if len(shape) < 2 or name == "token_embd.weight":
            continue
        tot += shape[1] * _row_bytes(S.types_for(name, w.types), shape[0])
    return tot


def kv_value_bytes(type_kv: int) -> float:
    return {0: 4.0, 1: 2.0, 8: 34.0 / 32.0}[type_kv]


def decode_step_bytes(w, visible, n_out: int) -> float:
    """Algorithmic bytes of one decode ubatch whose tokens see `visible[t]` cells each: all linear
    weights once, the norms, one embedding row per token, the K/V rows of the visible cells of
    every layer, this step's K/V writes, and the logits rows written."""
    import synthetic as S
    hp = w.hp
    T = len(visible)
    kv_row = 2.0 * hp.n_head_kv * hp.head_dim * kv_value_bytes(w.type_kv) * hp.n_layer
    emb = _row_bytes(S.types_for("token_embd.weight", w.types), hp.n_embd)
    return (linear_weight_bytes(w) + (2 * hp.n_layer + 1) * hp.n_embd * 4.0 + T * emb
            + float(sum(visible)) * kv_row + T * kv_row + n_out * hp.n_vocab * 4.0)


def linear_params_per_layer(hp) -> float:
    d, qd, kvd = hp.n_embd, hp.n_head * hp.head_dim, hp.n_head_kv * hp.head_dim
    return d * (qd + 2 * kvd) + qd * d + 3.0 * d * hp.n_ff


def prefill_flops(hp, n_tokens: int, attn_pairs: float, n_out: int) -> float:
    """2 per weight per prompt token, 4 * n_head * head_dim per (token, visible cell) pair of the
    causal attention in every layer, and the output matrix for the flagged rows."""
    return (2.0 * linear_params_per_layer(hp) * hp.n_layer * n_tokens
            + 4.0 * hp.n_head * hp.head_dim * attn_pairs * hp.n_layer
            + 2.0 * hp.n_embd * hp.n_vocab * n_out)


def causal_pairs(n_prompt: int) -> float:
    """(token, visible cell) pairs of one sequence's causal prompt: sum over p of (p + 1)."""
    return n_prompt * (n_prompt + 1) / 2.0


# ------------------------------------------------------------------------------- oracle sample
class OracleBaseline:
    """Times the CPU oracle (numpy float64, as it stands) on a bounded sample of a workload.

    Sample: the first `n_layers` transformer layers of the model and the first `out_frac` of the
    output matrix's rows, on the workload's own prompt. prefill() runs one prompt ubatch
    (min(n_prompt, n_ubatch) tokens of sequence 0, causal attention, K/V kept) through the
    sampled layers and the output rows for its last token; decode() runs one greedy-step token
    through the sampled layers (attention over every cell the sequence holds, this step's K/V
    appended) and the sampled output rows. Each is extrapolated to the whole model as
    (layer time) * n_layer / n_layers + (output time) / out_frac."""

    def __init__(self, w, n_layers: int = 2, out_frac: float = 1.0 / 8, device: str = "cpu"):
        import torch
        import oracle
        import synthetic as S
        self.w, self.hp = w, w.hp
        self.n_layers, self.out_frac = n_layers, out_frac
        hp = w.hp
        # as the oracle runs the 8B shapes in the tests: every matrix decoded from its storage
        # format when used, in row blocks (no float64 copy of the model kept)
        self.ow = oracle.OracleWeights(cache=False)
        for name, shape in S.tensor_specs(hp):
            if not any(name.startswith(f"blk.{il}.") for il in range(n_layers)) and name != "output_norm.weight":
                continue
            t = S.weight_bytes(w.weight_seed, name, shape, S.types_for(name, w.types), device)
            self.ow.add(name, S.types_for(name, w.types), shape[0], self._raw(t))
        n_out = max(1, int(math.ceil(out_frac * hp.n_vocab)))
        wt = S.types_for("output.weight", w.types)
        t = S.weight_bytes(w.weight_seed, "output.weight", (hp.n_embd, n_out), wt, device)
        self.ow.add("output.weight", wt, hp.n_embd, self._raw(t))
        self.n_ub = min(w.n_prompt, w.n_ubatch)
        self.prompt = S.prompt_tokens(w.prompt_seed_of(0), w.n_prompt, hp.n_vocab).numpy()[:self.n_ub]
        et = S.types_for("token_embd.weight", w.types)
        self.emb_t = et
        self.dev = device
        self._emb = {}
        self.k = [None] * n_layers
        self.v = [None] * n_layers
        self.pos = 0
        self.torch = torch
        self.desc = (f"oracle float64 (numpy) forward on the first {n_layers} of {hp.n_layer} layers and the "
                     f"first {out_frac:.4g} of the output matrix's rows, extrapolated as layer time x "
                     f"{hp.n_layer}/{n_layers} + output time / {out_frac:.4g}; prefill = one "
                     f"{self.n_ub}-token prompt ubatch (causal attention), decode = one token at context "
                     f"{self.n_ub + 1} onward (attention over all its cells)")

    @staticmethod
    def _raw(t):
        import torch
        t = t.detach().cpu().contiguous()
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()

    def _embed(self, toks):
        import synthetic as S
        from oracle.formats import decode_weight
        rows = S.weight_rows(self.w.weight_seed, "token_embd.weight", (self.hp.n_embd, self.hp.n_vocab),
                             self.emb_t, list(toks), self.dev)
        return decode_weight(self._raw(rows), self.emb_t, self.hp.n_embd)

    def _run(self, toks):
        """Sampled layers + sampled output rows for the last token; returns (layer s, output s)."""
        import oracle
        from oracle.context import forward_layers, output_logits
        hp = self.hp
        x = self._embed(toks)
        n = len(toks)
        pos = np.arange(self.pos, self.pos + n)
        causal = np.arange(self.pos + n)[None, :] <= pos[:, None]

        def kv_write(il, k, v):
            k = oracle.round_to_type(k, self.w.type_kv)
            v = oracle.round_to_type(v, self.w.type_kv)
            self.k[il] = k if self.k[il] is None else np.concatenate([self.k[il], k])
            self.v[il] = v if self.v[il] is None else np.concatenate([self.v[il], v])

        def kv_read(il):
            return self.k[il], self.v[il], causal

        t0 = time.perf_counter()
        x = forward_layers(self.ow, hp, x, pos, kv_write, kv_read, layers=range(self.n_layers))
        t1 = time.perf_counter()
        lg = output_logits(self.ow, hp, x[-1:])
        t2 = time.perf_counter()
        assert np.all(np.isfinite(lg))
        self.pos += n
        self.last = int(np.argmax(lg[0]))
        return t1 - t0, t2 - t1

    def _scale(self, tl, to):
        return tl * self.hp.n_layer / self.n_layers + to / self.out_frac

    def prefill(self):
        """(extrapolated seconds of one prompt ubatch, wall seconds of the sample)."""
        self.k = [None] * self.n_layers
        self.v = [None] * self.n_layers
        self.pos = 0
        tl, to = self._run(self.prompt)
        return self._scale(tl, to), tl + to

    def decode(self):
        """(extrapolated seconds of one decode step, wall seconds of the sample)."""
        tl, to = self._run([self.last])
        return self._scale(tl, to), tl + to


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


# ------------------------------------------------------------------------------- GPU arm
def make_ctx(w, stream, n_batch=None, fused_step=False):
    import torch
    import synthetic as S
    from transformer_decode_kv_gb300 import Context
    ctx = Context(w.hp, n_ctx=w.n_ctx, n_seq_max=w.n_seq, type_k=w.type_kv, type_v=w.type_kv,
                  n_batch=n_batch or w.n_batch, n_ubatch=w.n_ubatch, stream=stream.cuda_stream,
                  fused_step=fused_step)
    for name, wt, shape, t in S.model_weights(w.hp, w.weight_seed, w.types, "cuda"):
        if ctx.load_weight(name, wt, shape, t) != 0:
            raise RuntimeError(ctx.last_error())
        del t
    if ctx.weights_ready() != 0:
        raise RuntimeError(ctx.last_error())
    torch.cuda.empty_cache()
    return ctx


class Driver:
    """Prompt and greedy decode steps of one workload through the C ABI."""

    def __init__(self, ctx, w, rank: int):
        import synthetic as S
        self.ctx, self.w, self.NS = ctx, w, w.n_seq
        self.prompts = [S.prompt_tokens(w.prompt_seed_of(s) + 977 * rank if w.n_seq > 1 else w.prompt_seed + 97 * rank,
                                        w.n_prompt, w.hp.n_vocab).numpy() for s in range(w.n_seq)]
        self.seq_rows = [[s] for s in range(w.n_seq)]

    def prefill(self):
        """Every sequence's prompt, in calls of at most n_batch tokens; the last token of each
        sequence is the only output."""
        ctx, w = self.ctx, self.w
        if self.NS == 1 and ctx.n_batch >= w.n_prompt:
            return ctx.decode(self.prompts[0])
        for s in range(self.NS):
            for i0 in range(0, w.n_prompt, ctx.n_batch):
                chunk = self.prompts[s][i0:i0 + ctx.n_batch]
                flags = [0] * len(chunk)
                if i0 + len(chunk) == w.n_prompt:
                    flags[-1] = 1
                r = ctx.decode(chunk, seq_ids=[[s]] * len(chunk), logits=flags)
                if r != 0:
                    return r
        return 0

    def first_tokens(self):
        if self.NS == 1:
            return self.ctx.get_argmax_ith(-1)
        return [self.ctx.get_argmax_ith(-1)] * self.NS

    def steps(self, n, tok, on_step=None):
        """n greedy steps: one token per sequence each, device argmax read back each step."""
        ctx = self.ctx
        for i in range(n):
            if self.NS == 1:
                if ctx.decode([tok]) != 0:
                    raise RuntimeError(ctx.last_error())
                tok = ctx.get_argmax_ith(-1)
            else:
                if ctx.decode(tok, seq_ids=self.seq_rows, logits=[1] * self.NS) != 0:
                    raise RuntimeError(ctx.last_error())
                tok = [ctx.get_argmax_ith(i) for i in range(self.NS)]
            if on_step is not None:
                on_step(i + 1)
        return tok


def visible_cells(w, n_steps: int):
    """Cells each token of every decode step sees: sequence s's token at position p sees its p + 1
    cells; after the seq_rm of step seq_rm_at, sequence 0 continues from half its length."""
    p = [w.n_prompt] * w.n_seq
    out = []
    for i in range(1, n_steps + 1):
        out.append([q + 1 for q in p])
        p = [q + 1 for q in p]
        if i == w.seq_rm_at:
            p[0] //= 2
    return out


def time_prefill(drv, stream, reps):
    import torch
    times = []
    for rep in range(reps + 1):
        drv.ctx.seq_rm(-1, -1, -1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        r = drv.prefill()
        e1.record(stream)
        torch.cuda.synchronize()
        if r != 0:
            raise RuntimeError(f"prefill failed {r}: {drv.ctx.last_error()}")
        if rep > 0:                                  # the first repetition is a warm-up
            times.append(e0.elapsed_time(e1) / 1e3)
    return float(np.median(times))


def max_over_ranks(times, world):
    """Each timing's maximum over the replicas (the job's time is its slowest replica's); every rank
    receives the same values. A single process returns its own."""
    if world <= 1:
        return [float(x) for x in times]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x) for x in times], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_rate(units_per_replica, world, seconds):
    """Whole-job throughput of N replicas that each processed units_per_replica in at most seconds
    (weak scaling: the work per GPU is fixed)."""
    return world * units_per_replica / seconds


def run_headline(args, rank, world, local_rank, stream):
    import torch
    import torch.distributed as dist
    w = args.w
    ctx = make_ctx(w, stream, n_batch=max(w.n_batch, w.n_prompt) if w.n_seq == 1 else w.n_batch,
                   fused_step=args.fused_step)
    drv = Driver(ctx, w, rank)
    NS = w.n_seq

    def barrier():
        if world > 1:
            dist.barrier()

    # ---- prefill: the prompt as one batch (split into n_ubatch ubatches), timed with events
    prefill_s = time_prefill(drv, stream, 2 if NS == 1 else 1)
    # per-class kernel times of one prompt (eager launches, events around each)
    ctx.seq_rm(-1, -1, -1)
    ctx.kernel_timing(True)
    drv.prefill()
    ctx.kernel_timing(False)
    ks_pre = ctx.kernel_stats()
    tok0 = drv.first_tokens()

    K, W = args.steps, args.warmup
    if NS * (w.n_prompt + max(K, W)) > ctx.n_ctx:
        raise SystemExit(f"--steps/--warmup exceed the cache ({ctx.n_ctx} cells)")
    with ClockSampler(local_rank) as clk:
        drv.steps(W, tok0)
        ctx.seq_rm(-1, w.n_prompt, -1)                  # back to the prompt context
        barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        tw0 = time.perf_counter()
        e0.record(stream)
        drv.steps(K, tok0)
        e1.record(stream)
        torch.cuda.synchronize()
        tw1 = time.perf_counter()
        barrier()
        dec_s = e0.elapsed_time(e1) / 1e3

        # ---- the same K steps again with an event pair around every kernel: per-class shares
        ctx.seq_rm(-1, w.n_prompt, -1)
        ctx.kernel_timing(True)
        drv.steps(K, tok0)
        ctx.kernel_timing(False)
        ks = ctx.kernel_stats()

        # ---- end to end: host token in, host argmax out, wall clock around K steps
        ctx.seq_rm(-1, w.n_prompt, -1)
        barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        drv.steps(K, tok0)
        e2e_s = time.perf_counter() - t0
    dec_s, prefill_s, e2e_s = max_over_ranks([dec_s, prefill_s, e2e_s], world)

    # ---- the device sampler chain on the last logits row (top-k 40, top-p 0.95, min-p 0.05,
    # temperature 0.8, repeat penalty 1.1 over the last 64 tokens): host call to token, per call
    n_s = 32
    pen = list(drv.prompts[0][-64:])
    ctx.sample_ith(-1, top_k=40, top_p=0.95, min_p=0.05, temperature=0.8, repeat_penalty=1.1,
                   penalty_tokens=pen, u=0.5)
    t0 = time.perf_counter()
    for i in range(n_s):
        if ctx.sample_ith(-1, top_k=40, top_p=0.95, min_p=0.05, temperature=0.8, repeat_penalty=1.1,
                          penalty_tokens=pen, u=(i + 0.5) / n_s) < 0:
            raise RuntimeError(ctx.last_error())
    sample_us = (time.perf_counter() - t0) / n_s * 1e6
    wdev = ctx.perf()["weight_device_bytes"]
    ctx.free()
    return dict(dec_s=dec_s, prefill_s=prefill_s, e2e_s=e2e_s, ks=ks, ks_pre=ks_pre,
                clk=clk.summary((tw0, tw1)), sample_us=sample_us, visible=visible_cells(w, K), wdev=wdev)


def run_extra(key, stream, peaks):
    """Prefill and the configured decode run of another 8B workload, in a fresh context."""
    import torch
    import synthetic as S
    w = S.WORKLOADS[key]
    hp = w.hp
    ctx = make_ctx(w, stream)
    drv = Driver(ctx, w, 0)
    prefill_s = time_prefill(drv, stream, 1)
    tok0 = drv.first_tokens()
    drv.steps(3, tok0)                                  # warm-up (graph capture of the step shape)
    ctx.seq_rm(-1, w.n_prompt, -1)
    torch.cuda.synchronize()

    def on_step(i):
        if i == w.seq_rm_at:                          # half of sequence 0 dropped, then reused
            ctx.seq_rm(0, (ctx.seq_pos_max(0) + 1) // 2, -1)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    drv.steps(w.n_decode, tok0, on_step=on_step)
    e1.record(stream)
    torch.cuda.synchronize()
    dec_s = e0.elapsed_time(e1) / 1e3
    wdev = ctx.perf()["weight_device_bytes"]
    ctx.free()
    torch.cuda.empty_cache()
    step_bytes = float(np.mean([decode_step_bytes(w, v, w.n_seq) for v in visible_cells(w, w.n_decode)]))
    pre_fl = prefill_flops(hp, w.n_seq * w.n_prompt, w.n_seq * causal_pairs(w.n_prompt), w.n_seq)
    pre_tf = pre_fl / prefill_s / 1e12
    dec_gbs = step_bytes * w.n_decode / dec_s / 1e9
    return {"description": w.description, "n_ctx": w.n_ctx,
            "decode_tok_s": w.n_seq * w.n_decode / dec_s, "decode_steps": w.n_decode,
            "decode_ms_per_step": dec_s / w.n_decode * 1e3,
            "decode_step_algorithmic_bytes": step_bytes, "decode_hbm_gbs": dec_gbs,
            "decode_hbm_frac": dec_gbs / peaks["hbm_gbs"],
            "prefill_tok_s": w.n_seq * w.n_prompt / prefill_s, "prefill_ms": prefill_s * 1e3,
            "prefill_flops": pre_fl, "prefill_tflops": pre_tf,
            "prefill_tensor_frac": pre_tf / peaks["bf16_tflops"],
            "seq_rm_after_step": w.seq_rm_at if w.seq_rm_at > 0 else None,
            "weight_device_bytes": wdev}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="llama8b_bf16_1seq")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other two 8B workloads' figures")
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
    import synthetic as S
    w = S.WORKLOADS[args.workload]
    if args.layers:
        w = dataclasses.replace(w, hp=dataclasses.replace(w.hp, n_layer=args.layers))
        S.WORKLOADS[args.workload] = w
    if args.type_kv:
        w = dataclasses.replace(w, type_kv={"f32": 0, "f16": 1, "q8_0": 8}[args.type_kv])
        S.WORKLOADS[args.workload] = w
    args.w = w
    hp = w.hp
    peaks = measured_peaks()
    config = {"workload": args.workload, "description": w.description, "sequences": w.n_seq,
              "prompt_tokens": w.n_prompt, "decode_steps_timed": args.steps,
              "n_ctx": w.n_ctx, "kv_cache": {0: "f32", 1: "f16", 8: "q8_0"}[w.type_kv],
              "l2": "inputs larger than L2: every decode step streams all weights (no flush)",
              "parallelism": "replicas" if args.gpus > 1 else "single",
              "decode_path": "persistent step kernel" if args.fused_step else "per-op kernels (graph)"}
    if args.workload in ("llama8b_q8_0_8k", "llama8b_bf16_32seq"):
        config["n_ctx_note"] = ("the configuration's n_ctx (8192 / 65536) cannot hold its prompt plus "
                                "its decode steps; the cache is enlarged to the cells needed, rounded to 256")
    if args.layers:
        config["profiling_case_layers"] = args.layers

    if args.impl == "reference":
        if rank != 0:
            return
        smp = OracleBaseline(w, n_layers=1, out_frac=1.0 / 32)
        pre_s, pre_wall = smp.prefill()
        times, walls = [], []
        for i in range(args.warmup + args.steps):
            s, wall = smp.decode()
            if i >= args.warmup:
                times.append(s)
                walls.append(wall)
        step_s = float(np.mean(times))
        v = 1.0 / step_s
        n_pre = min(w.n_prompt, w.n_ubatch)
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tok/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": float(np.mean(walls)) * 1e3,
                "ms_per_step_note": ("wall time of each sampled step actually run (one token through "
                                     "the sampled layer and output rows); value is extrapolated to "
                                     "the whole model: see cpu_baseline.sample"),
                "extrapolated_ms_per_full_step": step_s * 1e3,
                "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "prefill_tok_s": n_pre / pre_s, "prefill_sample_wall_s": pre_wall,
                "cpu_baseline": {"value": v, "unit": "tok/s", "cores": cpu_cores(), "kind": "oracle",
                                 "sample": smp.desc, "prefill_value": n_pre / pre_s},
                "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if args.gpus > 1 or world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo")
    import torch
    from transformer_decode_kv_gb300 import LIB_PATH
    from transformer_decode_kv_gb300 import build as B
    if not os.path.exists(LIB_PATH):
        B.build()
    torch.cuda.set_device(local_rank)
    stream = torch.cuda.Stream()
    res = run_headline(args, rank, world, local_rank, stream)
    extra = {}
    if rank == 0 and world == 1 and not args.no_extra and not args.layers and not args.fused_step \
            and not args.type_kv and args.workload == "llama8b_bf16_1seq":
        for key in EXTRA_WORKLOADS:
            try:
                extra[key] = run_extra(key, stream, peaks)
            except Exception as e:                   # the headline stands without them
                extra[key] = {"failed": str(e)[:300]}
    if rank != 0:
        return
    K = args.steps
    dec_s, ms_step = res["dec_s"], res["dec_s"] / K * 1e3
    dec_tps = job_rate(w.n_seq * K, world, dec_s)
    pre_tps = job_rate(w.n_seq * w.n_prompt, world, res["prefill_s"])
    hbm = peaks["hbm_gbs"]

    # ---- decode roofline: the GEMV class's share of the graph-replayed step
    ks = res["ks"]
    tot_ms = sum(v["ms"] for v in ks.values())
    share = {k: v["ms"] / tot_ms for k, v in ks.items() if v["launches"]}
    dom = max(share, key=share.get)
    g = ks[dom]
    launches_per_step = g["launches"] / K
    dom_bytes_step = g["bytes"] / K
    dom_ms_step = share[dom] * ms_step                 # that class's time inside the real step
    achieved = dom_bytes_step / (dom_ms_step / 1e3) / 1e9
    step_bytes = float(np.mean([decode_step_bytes(w, v, w.n_seq) for v in res["visible"]]))
    traffic = GEMV_TRAFFIC.get(args.workload) if dom == "linear_gemv" and not args.layers else None
    roofline = {
        "bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm, "unit": "GB/s",
        "frac": achieved / hbm, "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
        "peak_source": peaks["source"], "traffic": traffic,
        "traffic_source": ("ncu dram__bytes_read.sum + dram__bytes_write.sum per launch of these "
                           "kernels, one capture of the current code (not measured in this run)")
        if traffic else None,
        "algorithmic_bytes_per_launch": dom_bytes_step / launches_per_step,
        "launches_per_step": launches_per_step,
        "avg_launch_us": dom_ms_step * 1e3 / launches_per_step,
        "share_of_step": share[dom],
        "method": ("the class's share of the summed per-kernel CUDA-event times of the same K steps "
                   "re-run with an event pair around each kernel (live, this run), times the "
                   "graph-replayed ms_per_step; achieved = the class's algorithmic bytes per step / "
                   "that time"),
        "isolated_avg_launch_us": g["ms"] * 1e3 / max(1, g["launches"]),
    }
    # ---- prefill roofline: useful FLOPs of the prompt at the dense bf16 tensor peak
    pre_fl = prefill_flops(hp, w.n_seq * w.n_prompt, w.n_seq * causal_pairs(w.n_prompt), w.n_seq)
    pre_tf = pre_fl / res["prefill_s"] / 1e12
    kp = res["ks_pre"]
    lin = [k for k in kp if k.startswith("linear") and kp[k]["launches"]]
    gname = max(lin, key=lambda k: kp[k]["flops"]) if lin else "linear_tcgen05"
    gemm = kp.get(gname, {"ms": 0.0, "flops": 0.0, "launches": 0})
    pre_tot = sum(v["ms"] for v in kp.values())
    roofline_prefill = {
        "bound": "tensor", "achieved": pre_tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
        "frac": pre_tf / peaks["bf16_tflops"], "peak_source": peaks["source"] + " bf16 burst",
        "flops": pre_fl, "time_ms": res["prefill_s"] * 1e3,
        "flops_formula": "2 x linear params x tokens + 4 x n_head x head_dim x causal pairs x layers + 2 x d x vocab per output",
        "dominant_kernel": {
            "kernel": gname + " (the prompt's matrix products: token-major tcgen05 GEMMs)",
            "achieved": gemm["flops"] / (gemm["ms"] / 1e3) / 1e12 if gemm["ms"] else None,
            "frac": gemm["flops"] / (gemm["ms"] / 1e3) / 1e12 / peaks["bf16_tflops"] if gemm["ms"] else None,
            "launches": gemm["launches"], "share_of_prompt": gemm["ms"] / pre_tot if pre_tot else None,
            "method": "CUDA events around each launch of one prompt (eager launches)"},
        "kernel_share": {k: v["ms"] / pre_tot for k, v in kp.items() if v["launches"]} if pre_tot else {},
        "kernel_ms": {k: v["ms"] for k, v in kp.items() if v["launches"]},
    }
    line = {
        "metric": METRIC, "value": dec_tps, "unit": "tok/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 weights; decode f32 activations, prefill f16 GEMM operands; f32 accumulation",
        "data": "synthetic (seeded random weights and prompt)", "config": config,
        "prefill_tok_s": pre_tps, "prefill_ms": res["prefill_s"] * 1e3,
        "weight_device_bytes": res["wdev"],
        "sampler_us_per_call": res["sample_us"],
        "decode_step_algorithmic_bytes": step_bytes,
        "decode_hbm_gbs": step_bytes / (ms_step / 1e3) / 1e9,
        "decode_hbm_frac": step_bytes / (ms_step / 1e3) / 1e9 / hbm,
        "roofline": roofline,
        "roofline_prefill": roofline_prefill,
        "kernel_share": share,
        "clocks": res["clk"],
        "e2e": {"value": job_rate(w.n_seq * K, world, res["e2e_s"]), "unit": "tok/s",
                "h2d_bytes_per_step": 4 * w.n_seq, "d2h_bytes_per_step": 8 * w.n_seq},
        "gpu_launches": int(round(sum(v["launches"] for v in ks.values()) / K)) * K,
    }
    if extra:
        line["extra"] = extra
    if not args.no_cpu_baseline and world == 1:
        try:
            smp = OracleBaseline(w, n_layers=4, out_frac=1.0 / 4, device="cuda")
            pre_s, pre_wall = smp.prefill()
            dec = [smp.decode() for _ in range(2)]
            dec_step = min(d[0] for d in dec)
            n_pre = min(w.n_prompt, w.n_ubatch)
            line["cpu_baseline"] = {"value": w.n_seq / dec_step, "unit": "tok/s", "cores": cpu_cores(),
                                    "kind": "oracle", "sample": smp.desc,
                                    "prefill_value": n_pre / pre_s, "prefill_unit": "tok/s",
                                    "wall_s": pre_wall + sum(d[1] for d in dec)}
        except Exception as e:  # the GPU number stands without it
            line["cpu_baseline"] = {"value": None, "unit": "tok/s", "cores": cpu_cores(),
                                    "kind": "oracle", "sample": f"failed: {e}"}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
