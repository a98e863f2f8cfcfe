"""Shared harness of the GPU parity tests: synthetic models on the device, the library context,
the oracle context on the same weights, and the greedy-run comparison."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
import synthetic as S
from tests.helpers import to_numpy_raw

GAP = 1e-3          # greedy tokens are compared where the oracle's top-2 gap exceeds this


def rel_err(g: np.ndarray, o: np.ndarray) -> float:
    """max_v |g_v - o_v| / max_v |o_v| of one logits row."""
    return float(np.max(np.abs(g.astype(np.float64) - o)) / np.max(np.abs(o)))


@functools.lru_cache(maxsize=2)
def device_model(key: str):
    w = S.WORKLOADS[key]
    return [(n, wt, sh, t) for n, wt, sh, t in S.model_weights(w.hp, w.weight_seed, w.types, "cuda")]


def library_ctx(key: str, **over):
    from transformer_decode_kv_gb300 import Context
    w = S.WORKLOADS[key]
    kw = dict(n_ctx=w.n_ctx, n_seq_max=w.n_seq, type_k=w.type_kv, type_v=w.type_kv,
              n_batch=w.n_batch, n_ubatch=w.n_ubatch)
    kw.update(over)
    ctx = Context(w.hp, **kw)
    ctx.load_all(device_model(key))
    return ctx


@functools.lru_cache(maxsize=2)
def oracle_weights(key: str, cache: bool = True):
    ow = oracle.OracleWeights(cache=cache)
    for n, wt, sh, t in device_model(key):
        ow.add(n, wt, sh[0], to_numpy_raw(t))
    return ow


def oracle_ctx(key: str, **over):
    w = S.WORKLOADS[key]
    kw = dict(n_ctx=w.n_ctx, n_seq_max=w.n_seq, type_k=w.type_kv, type_v=w.type_kv,
              n_batch=w.n_batch, n_ubatch=w.n_ubatch)
    kw.update(over)
    return oracle.OracleContext(w.hp, oracle_weights(key), **kw)


def prompts(key: str):
    w = S.WORKLOADS[key]
    return [S.prompt_tokens(w.prompt_seed_of(s), w.n_prompt, w.hp.n_vocab).numpy()
            for s in range(w.n_seq)]


def prompt_batch(key: str):
    """Sequence-major prompt batch; the last prompt token of each sequence is flagged."""
    w = S.WORKLOADS[key]
    ps = prompts(key)
    toks = np.concatenate(ps)
    seqs = [[s] for s in range(w.n_seq) for _ in range(w.n_prompt)]
    flags = np.zeros(len(toks), dtype=np.int8)
    flags[[(s + 1) * w.n_prompt - 1 for s in range(w.n_seq)]] = 1
    return toks, seqs, flags


def greedy_compare(ctx, ora, n_seq: int, first_rows, n_steps: int, tol: float, report: dict):
    """Compare the flagged logits of the step just decoded, pick the next tokens and decode them
    in both. Tokens must match where the oracle's top-2 gap exceeds GAP; elsewhere both sides take
    the library's token (teacher forcing)."""
    rows = list(first_rows)
    for step in range(n_steps + 1):
        nxt = []
        for s, i in enumerate(rows):
            g = ctx.get_logits_ith(i)
            o = ora.get_logits_ith(i)
            assert g is not None and o is not None
            e = rel_err(g, o)
            report["max_rel_err"] = max(report.get("max_rel_err", 0.0), e)
            assert e <= tol, (step, s, e)
            top = np.argsort(o)[-2:]
            gap = o[top[1]] - o[top[0]]
            tg = ctx.get_argmax_ith(i)
            assert tg == int(np.argmax(g)), "device argmax disagrees with the logits it computed"
            if gap > GAP:
                assert tg == int(top[1]), (step, s, tg, int(top[1]), gap)
                report["tokens_checked"] = report.get("tokens_checked", 0) + 1
            else:
                report["tokens_teacher_forced"] = report.get("tokens_teacher_forced", 0) + 1
            nxt.append(tg)
        if step == n_steps:
            break
        seqs = [[s] for s in range(n_seq)]
        assert ctx.decode(nxt, seq_ids=seqs, logits=[1] * n_seq) == 0, ctx.last_error()
        assert ora.decode(nxt, seq_id=seqs, n_seq_id=[1] * n_seq, logits=[1] * n_seq) == 0
        rows = list(range(n_seq))
    return report
