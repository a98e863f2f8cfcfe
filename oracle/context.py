"""The decode loop over a KV cache, mirroring llama_decode's steps one by one.

[P1] Крок 11 (llama_context::decode: balloc.init, init_batch, per-ubatch process_ubatch, logits
copied into the output buffer in batch order, return codes), Крок 12 (the whole batch is split and a
slot is found for every ubatch before any is committed; no room -> 1), Крок 13а-13в (apply, then the
graph: embeddings -> layers -> keep the requested rows -> final norm -> output matrix), Крок 14
(llama_get_logits_ith: i < 0 counts from the last output row; an unrequested index gives NULL);
[P4] エラーリカバリとステートロールバック (a failed ubatch is rolled back with seq_rm(s, pos_min, -1);
earlier ubatches stay).
"""
from __future__ import annotations

from typing import Callable, Dict, List, Optional

import numpy as np

from .formats import F16, F32, decode_weight, round_to_type
from .memory import (Cells, DecodeStatus, LLAMA_MAX_SEQ, derive_cparams, sanitize_batch,
                     split_simple, split_equal)
from .numerics import attention, linear, rms_norm, rope, swiglu


class OracleWeights:
    """Named weights kept in their storage format, decoded to float64 when used.

    raw: numpy array of the storage bytes (F32/F16/BF16 as 2-D element arrays, Q8_0 as uint8
    [rows, row_bytes]); ne0: row length in values. With cache=True the decoded float64 matrices
    are kept (small models)."""

    def __init__(self, cache: bool = True, row_chunk: int = 8192):
        self.raw: Dict[str, tuple] = {}
        self.cache = cache
        self.row_chunk = row_chunk
        self._dec: Dict[str, np.ndarray] = {}

    def add(self, name: str, wtype: int, ne0: int, raw: np.ndarray):
        self.raw[name] = (wtype, ne0, raw)
        self._dec.pop(name, None)

    def has(self, name: str) -> bool:
        return name in self.raw

    def get(self, name: str) -> np.ndarray:
        if name in self._dec:
            return self._dec[name]
        wtype, ne0, raw = self.raw[name]
        w = decode_weight(raw, wtype, ne0)
        if self.cache:
            self._dec[name] = w
        return w

    def vector(self, name: str) -> np.ndarray:
        return self.get(name).reshape(-1)

    def rows(self, name: str, idx) -> np.ndarray:
        """Rows idx of a weight (the GET_ROWS of an embedding lookup)."""
        wtype, ne0, raw = self.raw[name]
        return decode_weight(raw[np.asarray(idx)], wtype, ne0)

    def matmul(self, x: np.ndarray, name: str) -> np.ndarray:
        """linear(x, W) for a named weight; a large weight is decoded in row blocks (each output
        column is still one full dot product)."""
        if self.cache or name in self._dec:
            return linear(x, self.get(name))
        wtype, ne0, raw = self.raw[name]
        rows = raw.shape[0]
        out = np.empty((x.shape[0], rows), dtype=np.float64)
        for r0 in range(0, rows, self.row_chunk):
            r1 = min(rows, r0 + self.row_chunk)
            out[:, r0:r1] = linear(x, decode_weight(raw[r0:r1], wtype, ne0))
        return out


def forward_layers(w: OracleWeights, hp, x: np.ndarray, pos: np.ndarray, kv_write, kv_read,
                   layers=None):
    """The transformer blocks over the residual stream x [T, d] ([P2] Example 4, [P1] Крок 13б).

    kv_write(il, k, v) stores this ubatch's rounded K/V rows; kv_read(il) returns (K cells,
    V cells, visible mask) for the attention. Returns x after the last layer."""
    H, Hkv, hd = hp.n_head, hp.n_head_kv, hp.head_dim
    T = x.shape[0]
    for il in (range(hp.n_layer) if layers is None else layers):
        p = f"blk.{il}."
        h = rms_norm(x, w.vector(p + "attn_norm.weight"), hp.rms_eps)
        q = w.matmul(h, p + "attn_q.weight").reshape(T, H, hd)
        k = w.matmul(h, p + "attn_k.weight").reshape(T, Hkv, hd)
        v = w.matmul(h, p + "attn_v.weight").reshape(T, Hkv, hd)
        q = rope(q, pos, hp.rope_freq_base)
        k = rope(k, pos, hp.rope_freq_base)
        kv_write(il, k, v)
        kc, vc, visible = kv_read(il)
        o = attention(q, kc, vc, visible, Hkv)
        x = x + w.matmul(o, p + "attn_output.weight")
        h = rms_norm(x, w.vector(p + "ffn_norm.weight"), hp.rms_eps)
        u = swiglu(w.matmul(h, p + "ffn_gate.weight"), w.matmul(h, p + "ffn_up.weight"))
        x = x + w.matmul(u, p + "ffn_down.weight")
    return x


def output_logits(w: OracleWeights, hp, x_rows: np.ndarray) -> np.ndarray:
    """Final RMSNorm by output_norm.weight then the output matrix ([P1] Крок 13б, last item).
    reading: a model without output.weight reuses token_embd.weight (tied embeddings)."""
    xo = rms_norm(x_rows, w.vector("output_norm.weight"), hp.rms_eps)
    name = "output.weight" if w.has("output.weight") else "token_embd.weight"
    return w.matmul(xo, name)


class OracleContext:
    """A llama context: a KV cache of n_ctx cells, the batch allocator and the outputs.

    kv_unified (default) shares all n_ctx cells among the sequences (one stream); otherwise each
    sequence has a stream of its own of n_ctx // n_seq_max cells, and batches are split with
    split_equal instead of split_simple ([P1] Крок 12)."""

    def __init__(self, hp, weights: Optional[OracleWeights], n_ctx: int, n_seq_max: int = 1,
                 type_k: int = F16, type_v: int = F16, n_batch: int = 2048, n_ubatch: int = 512,
                 compute: bool = True, kv_unified: bool = True):
        cp = derive_cparams(n_ctx, n_batch, n_ubatch, n_seq_max)
        if cp is None:
            raise ValueError("invalid context parameters")
        self.n_ctx, self.n_batch, self.n_ubatch = cp
        self.hp, self.w = hp, weights
        self.n_seq_max = n_seq_max
        self.type_k, self.type_v = type_k, type_v
        self.kv_unified = kv_unified
        self.n_stream = 1 if kv_unified else n_seq_max
        self.cells = Cells(self.n_ctx, self.n_stream)
        self.compute = compute      # False: batch / cell bookkeeping only, no forward pass
        kvd = (hp.n_head_kv, hp.head_dim)
        n_k = hp.n_layer if compute else 0
        self.K = [np.zeros((self.n_ctx,) + kvd) for _ in range(n_k)]
        self.V = [np.zeros((self.n_ctx,) + kvd) for _ in range(n_k)]
        self.abort_callback: Optional[Callable[[], bool]] = None
        self.fail_at_ubatch: Optional[int] = None      # test hook: ubatch whose compute fails
        self.output_all = False
        self._reset_outputs(0)
        self.last_ubatches: List[dict] = []

    # ---- memory API ([P4] llama_memory_i) ----
    def seq_pos_max(self, s: int) -> int:
        return self.cells.seq_pos_max(s)

    def seq_pos_min(self, s: int) -> int:
        return self.cells.seq_pos_min(s)

    def seq_rm(self, s: int, p0: int, p1: int) -> bool:
        return self.cells.seq_rm(s, p0, p1)

    def memory_update(self, optimize: bool) -> bool:
        """llama_memory_i::update ([P4] KVキャッシュの詳細: with optimize=true the cache is
        defragmented, cells moved to close the gaps, the K/V rows moving with their cells).
        Returns True if any cell moved."""
        if not optimize:
            return False
        if self.cells.is_defragged():
            return False
        src = self.cells.defrag_order()
        keep = src >= 0
        self.cells.move(src)
        for il in range(len(self.K)):
            for X in (self.K, self.V):
                moved = np.zeros_like(X[il])
                moved[keep] = X[il][src[keep]]
                X[il] = moved
        return True

    # ---- outputs ([P1] Крок 14) ----
    def _reset_outputs(self, n_tokens: int):
        self.output_ids = np.full(n_tokens, -1, dtype=np.int64)
        self.logits = np.zeros((0, self.hp.n_vocab))

    @property
    def n_outputs(self) -> int:
        return self.logits.shape[0]

    def get_logits_ith(self, i: int) -> Optional[np.ndarray]:
        """i >= 0: the row of batch token i (None if its logits were not requested);
        i < 0: counted from the last output row (-1 = last)."""
        if i < 0:
            j = self.n_outputs + i
            if j < 0:
                return None
        else:
            if i >= len(self.output_ids) or self.output_ids[i] < 0:
                return None
            j = int(self.output_ids[i])
        return self.logits[j]

    def get_argmax_ith(self, i: int) -> int:
        """Greedy pick: index of the largest logit, lowest index on ties (reading); -1 if none."""
        row = self.get_logits_ith(i)
        return -1 if row is None else int(np.argmax(row))

    # ---- decode ([P1] Крок 11-13) ----
    def decode(self, token, pos=None, n_seq_id=None, seq_id=None, logits=None) -> int:
        b = sanitize_batch(token, pos, n_seq_id, seq_id, logits, n_vocab=self.hp.n_vocab,
                           n_seq_max=self.n_seq_max, n_batch=self.n_batch, cells=self.cells,
                           output_all=self.output_all)
        self._reset_outputs(0)
        if b is None:
            return int(DecodeStatus.INVALID_BATCH)
        if self.n_stream > 1:
            # reading: a token of a split cache lives in its sequence's stream, so it has one sequence
            if any(len(ss) != 1 for ss in b.seq_id):
                return int(DecodeStatus.INVALID_BATCH)
            ubatches = split_equal([ss[0] for ss in b.seq_id], self.n_ubatch)
        else:
            ubatches = split_simple(b.n_tokens, self.n_ubatch)
        # find a slot for every ubatch before committing any ([P1] Крок 12); if that fails, one
        # defrag and one more try ([P4] KVキャッシュの詳細: FAILED_PREPARE -> defrag -> retry)
        slots_all = self._prepare(b, ubatches)
        if slots_all is None and self.memory_update(True):
            slots_all = self._prepare(b, ubatches)
        if slots_all is None:
            return int(DecodeStatus.NO_KV_SLOT)
        self.last_ubatches = []
        rows, row_tok = [], []
        for k, ub in enumerate(ubatches):
            idx = list(ub)
            upos = b.pos[idx]
            useq = [b.seq_id[i] for i in idx]
            self.cells.apply(slots_all[k], upos, useq)           # mctx->apply()
            failed = None
            if self.abort_callback is not None and self.abort_callback():
                failed = DecodeStatus.ABORTED
            elif self.fail_at_ubatch == k:
                failed = DecodeStatus.COMPUTE_FAILED
            if failed is not None:
                self._rollback(upos, useq)
                self._reset_outputs(0)
                return int(failed)
            out_rows = [t for t, i in enumerate(idx) if b.output[i]]
            rows.append(self._process_ubatch(b.token[idx], upos, useq, slots_all[k], out_rows))
            row_tok.extend(idx[t] for t in out_rows)
        # output rows in batch order, whatever order the ubatches took the tokens in
        logits = np.concatenate(rows, axis=0) if rows else np.zeros((0, self.hp.n_vocab))
        self.logits = logits[np.argsort(row_tok, kind="stable")] if row_tok else logits
        self.output_ids = np.full(b.n_tokens, -1, dtype=np.int64)
        self.output_ids[np.nonzero(b.output)[0]] = np.arange(int(b.output.sum()))
        return int(DecodeStatus.OK)

    def _prepare(self, b, ubatches):
        work = self.cells.copy()
        slots_all = []
        for ub in ubatches:
            if self.n_stream == 1:
                sl = work.find_slots(len(ub))
            else:                            # each token takes the next free cell of its stream
                sl, need = [None] * len(ub), {}
                for t, i in enumerate(ub):
                    need.setdefault(b.seq_id[i][0], []).append(t)
                for s, ts in need.items():
                    got = work.find_slots(len(ts), s)
                    if got is None:
                        sl = None
                        break
                    for t, cell in zip(ts, got):
                        sl[t] = cell
            if sl is None:
                return None
            work.apply(sl, b.pos[list(ub)], [b.seq_id[i] for i in ub])
            slots_all.append(sl)
        return slots_all

    def _rollback(self, upos, useq):
        """[P4] エラーリカバリ: pos_min per sequence over the ubatch, then seq_rm(s, pos_min, -1)."""
        pos_min = {}
        for p, ss in zip(upos, useq):
            for s in ss:
                pos_min[s] = min(pos_min.get(s, int(p)), int(p))
        for s, p in pos_min.items():
            self.cells.seq_rm(s, p, -1)

    def _process_ubatch(self, tokens, upos, useq, slots, out_rows):
        hp = self.hp
        n_kv = self.cells.n_kv()
        visible = self.cells.mask(upos, useq, n_kv)
        self.last_ubatches.append({"slots": list(slots), "n_kv": n_kv, "mask": visible,
                                   "out_rows": list(out_rows), "pos": list(upos)})
        if not self.compute:
            return np.zeros((len(out_rows), hp.n_vocab))
        x = self.w.rows("token_embd.weight", tokens)                        # GET_ROWS
        slots = np.asarray(slots)

        def kv_write(il, k, v):                                             # SET_ROWS
            self.K[il][slots] = round_to_type(k, self.type_k)
            self.V[il][slots] = round_to_type(v, self.type_v)

        def kv_read(il):
            return self.K[il][:n_kv], self.V[il][:n_kv], visible

        x = forward_layers(self.w, hp, x, np.asarray(upos), kv_write, kv_read)
        if not out_rows:
            return np.zeros((0, hp.n_vocab))
        return output_logits(self.w, hp, x[out_rows])


def forward_no_cache(w: OracleWeights, hp, tokens, type_k: int = F16, type_v: int = F16):
    """Whole-sequence forward without a cache: positions 0..n-1, a lower-triangular mask, K/V
    rounded to the cache types. Returns logits for every position [n, n_vocab]. Used to check that
    cached, ubatched decoding gives the same result."""
    tokens = np.asarray(tokens)
    n = len(tokens)
    pos = np.arange(n)
    causal = np.tril(np.ones((n, n), dtype=bool))
    store = {}

    def kv_write(il, k, v):
        store[il] = (round_to_type(k, type_k), round_to_type(v, type_v))

    def kv_read(il):
        return store[il][0], store[il][1], causal

    x = forward_layers(w, hp, w.rows("token_embd.weight", tokens), pos, kv_write, kv_read)
    return output_logits(w, hp, x)
