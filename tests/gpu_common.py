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


# ---- full-size checks: one layer of the oracle on the library's own inputs ----

def layer_check(ow, hp, il: int, x_in: np.ndarray, x_out: np.ndarray, pos, slots, visible,
                kc: np.ndarray, vc: np.ndarray, type_kv: int) -> dict:
    """Layer il of the oracle for a few tokens, fed the library's residual stream before the layer
    (x_in [n, d]) and the library's layer-il K/V cache (kc, vc [n_head_kv][n_ctx][head_dim], float).

    Checks the K/V rows the library appended for these tokens (at cells `slots`) and the layer's
    update x_out - x_in, with attention over the cells `visible[t]` (a bool row over the first
    n_kv cells). At full size this is what the oracle can afford: every layer's input comes from
    the library, so each layer is checked on its own. Returns the largest relative errors
    (max |library - oracle| / max |oracle| per token row)."""
    H, Hkv, hd = hp.n_head, hp.n_head_kv, hp.head_dim
    n = x_in.shape[0]
    p = f"blk.{il}."
    x_in = x_in.astype(np.float64)
    h = oracle.rms_norm(x_in, ow.vector(p + "attn_norm.weight"), hp.rms_eps)
    q = oracle.rope(ow.matmul(h, p + "attn_q.weight").reshape(n, H, hd), np.asarray(pos),
                    hp.rope_freq_base)
    k = oracle.rope(ow.matmul(h, p + "attn_k.weight").reshape(n, Hkv, hd), np.asarray(pos),
                    hp.rope_freq_base)
    v = ow.matmul(h, p + "attn_v.weight").reshape(n, Hkv, hd)
    k = oracle.round_to_type(k, type_kv)
    v = oracle.round_to_type(v, type_kv)
    kc = kc.astype(np.float64)
    vc = vc.astype(np.float64)
    err = {"k": 0.0, "v": 0.0, "delta": 0.0}
    o = np.zeros((n, H * hd))
    for t in range(n):
        gk = kc[:, slots[t], :]
        gv = vc[:, slots[t], :]
        err["k"] = max(err["k"], rel_err(gk.reshape(-1), k[t].reshape(-1)))
        err["v"] = max(err["v"], rel_err(gv.reshape(-1), v[t].reshape(-1)))
        cells = np.nonzero(visible[t])[0]
        kt = kc[:, cells, :].transpose(1, 0, 2)
        vt = vc[:, cells, :].transpose(1, 0, 2)
        o[t] = oracle.attention(q[t:t + 1], kt, vt, np.ones((1, len(cells)), dtype=bool), Hkv)[0]
    x = x_in + ow.matmul(o, p + "attn_output.weight")
    h = oracle.rms_norm(x, ow.vector(p + "ffn_norm.weight"), hp.rms_eps)
    u = oracle.swiglu(ow.matmul(h, p + "ffn_gate.weight"), ow.matmul(h, p + "ffn_up.weight"))
    x = x + ow.matmul(u, p + "ffn_down.weight")
    for t in range(n):
        err["delta"] = max(err["delta"], rel_err(x_out[t] - x_in[t], x[t] - x_in[t]))
    return err


def logits_check(ow, hp, x_last: np.ndarray, g_logits, g_argmax) -> dict:
    """The oracle's final norm and output matrix on the library's last residual rows [n, d]
    against the library's logits rows and device argmax picks. Tokens must agree where the
    oracle's top-2 gap exceeds GAP."""
    from oracle.context import output_logits
    o = output_logits(ow, hp, x_last.astype(np.float64))
    out = {"logits": 0.0, "tokens_checked": 0}
    for t in range(len(o)):
        out["logits"] = max(out["logits"], rel_err(g_logits[t], o[t]))
        top = np.argsort(o[t])[-2:]
        if o[t][top[1]] - o[t][top[0]] > GAP:
            assert int(g_argmax[t]) == int(top[1]), (t, int(g_argmax[t]), int(top[1]))
            out["tokens_checked"] += 1
    return out


def kv_layer(ctx, il: int):
    return ctx.kv_cache(il, 0), ctx.kv_cache(il, 1)


def captured_rows(ctx, il: int, rows):
    """(x_in, x_out) rows of layer il from the library's capture of its last ubatch."""
    src = ctx.debug_tensor("embd") if il == 0 else ctx.debug_tensor("l_out", il - 1)
    d = ctx._hp.n_embd
    x_in = src.reshape(-1, d)[rows]
    x_out = ctx.debug_tensor("l_out", il).reshape(-1, d)[rows]
    return x_in, x_out


def mirror_ctx(w, **over):
    """The oracle's batch and cell bookkeeping alone (no forward pass), run beside the library."""
    kw = dict(n_ctx=w.n_ctx, n_seq_max=w.n_seq, type_k=w.type_kv, type_v=w.type_kv,
              n_batch=w.n_batch, n_ubatch=w.n_ubatch)
    kw.update(over)
    return oracle.OracleContext(w.hp, None, compute=False, **kw)


def mirror_slots(m):
    return np.concatenate([np.asarray(u["slots"], dtype=np.int32) for u in m.last_ubatches])


def check_layers(ctx, ow, w, layers, rows, bidx, pos, seqs, mirror, report, tag, tol):
    """layer_check for the captured rows `rows` of the library's last ubatch (batch indices bidx,
    positions pos, sequence ids seqs), with the mirror's visibility of the cells."""
    slots = ctx.last_slots()
    vis = mirror.cells.mask(pos, seqs, mirror.cells.n_kv())
    for il in layers:
        x_in, x_out = captured_rows(ctx, il, rows)
        kc, vc = kv_layer(ctx, il)
        e = layer_check(ow, w.hp, il, x_in, x_out, pos, slots[bidx], vis, kc, vc, w.type_kv)
        report[f"{tag}_layer{il}"] = e
        assert max(e.values()) <= tol, (tag, il, e)
