"""Batch sanitising, ubatch splitting, KV cells, slot finding, masks and the context parameters.

[P1] Крок 10 (llama_batch_allocr::init), Крок 12 (llama_kv_cache::init_batch), Крок 13а (apply);
[P4] バッチパイプライン, KVキャッシュの詳細 (llama_kv_cells: pos, seq bitset, seq_pos), エラーリカバリ.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from enum import IntEnum
from typing import List, Optional, Sequence

import numpy as np

LLAMA_MAX_SEQ = 256   # reading: the pages name the limit LLAMA_MAX_SEQ without its value
N_CTX_PAD = 256       # [P2] Example 9: n_ctx is rounded up to a multiple of 256 (GGML_PAD)


class DecodeStatus(IntEnum):
    """llama_decode return values ([P1] Крок 11; [P4] エラーリカバリ)."""
    OK = 0
    NO_KV_SLOT = 1        # no room in the cache for the batch: warning, state unchanged
    ABORTED = 2           # the abort callback stopped the computation
    INVALID_BATCH = -1
    ALLOC_FAILED = -2     # also: internal error / no memory context
    COMPUTE_FAILED = -3


def derive_cparams(n_ctx: int, n_batch: int, n_ubatch: int, n_seq_max: int, causal: bool = True):
    """Context sizes ([P1] Крок 9-10 context constructor; [P2] Example 9):
    n_ctx rounded up to a multiple of 256; n_batch = min(n_ctx, n_batch) for a causal model;
    n_ubatch = min(n_batch, n_ubatch). Returns (n_ctx, n_batch, n_ubatch) or None if invalid."""
    if n_ctx <= 0 or n_batch <= 0 or n_ubatch <= 0 or not (1 <= n_seq_max <= LLAMA_MAX_SEQ):
        return None
    n_ctx = (n_ctx + N_CTX_PAD - 1) // N_CTX_PAD * N_CTX_PAD
    if causal:
        n_batch = min(n_ctx, n_batch)
    n_ubatch = min(n_batch, n_ubatch)
    return n_ctx, n_batch, n_ubatch


@dataclass
class Batch:
    """A sanitised batch: every field filled in ([P1] Крок 10 llama_batch)."""
    token: np.ndarray            # int32 [n]
    pos: np.ndarray              # int32 [n]
    seq_id: List[List[int]]      # per token, one or more sequence ids
    output: np.ndarray           # bool [n]

    @property
    def n_tokens(self) -> int:
        return len(self.token)


class Cells:
    """KV cells ([P4] KVキャッシュの詳細, llama_kv_cells): per cell a position (-1 = empty) and the
    set of sequences using it (a cell can be shared), held as a bool row seq[c, s].

    n_stream > 1 is a cache that is not shared by all sequences ([P1] Крок 9-10: n_ctx is then
    divided among the sequences, n_ctx_seq cells each; [P2] Example 9: kv_unified): stream s owns
    cells [s * n_ctx_seq, (s + 1) * n_ctx_seq), n_ctx_seq = n_ctx // n_stream (reading: the
    remainder of the division is left unused)."""

    def __init__(self, n_ctx: int, n_stream: int = 1):
        self.pos = np.full(n_ctx, -1, dtype=np.int64)
        self.seq = np.zeros((n_ctx, LLAMA_MAX_SEQ), dtype=bool)
        self.n_stream = n_stream
        self.n_ctx_seq = n_ctx // n_stream

    def stream_range(self, s: int):
        """Cells [lo, hi) of stream s (the whole cache when there is one stream)."""
        if self.n_stream == 1:
            return 0, len(self.pos)
        return s * self.n_ctx_seq, (s + 1) * self.n_ctx_seq

    @property
    def size(self) -> int:
        return len(self.pos)

    def copy(self) -> "Cells":
        c = Cells.__new__(Cells)
        c.pos = self.pos.copy()
        c.seq = self.seq.copy()
        c.n_stream, c.n_ctx_seq = self.n_stream, self.n_ctx_seq
        return c

    def seqs_of(self, c: int) -> set:
        """The sequence ids cell c holds."""
        return set(np.nonzero(self.seq[c])[0].tolist())

    def is_empty(self, c: int) -> bool:
        return self.pos[c] < 0

    def seq_pos_max(self, s: int) -> int:
        """Largest position held for sequence s, -1 if none ([P1] KV-cache section)."""
        ps = self.pos[self.seq[:, s]]
        return int(ps.max()) if len(ps) else -1

    def seq_pos_min(self, s: int) -> int:
        ps = self.pos[self.seq[:, s]]
        return int(ps.min()) if len(ps) else -1

    def seq_rm(self, s: int, p0: int, p1: int) -> bool:
        """Remove sequence s from the cells with p0 <= pos < p1 ([P4] エラーリカバリ, seq_rm).

        reading: p0 < 0 means 0 and p1 < 0 means no upper bound (the rollback calls
        seq_rm(s, pos_min, -1) to drop everything from pos_min on); s < 0 means every sequence.
        A cell whose sequence set becomes empty is freed (pos = -1)."""
        if p0 < 0:
            p0 = 0
        if p1 < 0:
            p1 = np.iinfo(np.int64).max
        sel = (self.pos >= 0) & (self.pos >= p0) & (self.pos < p1)
        if s < 0:
            self.seq[sel, :] = False
        else:
            self.seq[sel, s] = False
        self.pos[sel & ~self.seq.any(axis=1)] = -1
        return True

    def find_slots(self, n: int, stream: int = 0) -> Optional[List[int]]:
        """reading ("contiguous, or at least available" cells, [P4] KVキャッシュの詳細): the n
        lowest-index empty cells of the stream, in ascending order; None if fewer are empty."""
        lo, hi = self.stream_range(stream)
        free = lo + np.nonzero(self.pos[lo:hi] < 0)[0]
        return free[:n].tolist() if len(free) >= n else None

    def apply(self, slots: Sequence[int], pos: Sequence[int], seq_ids: Sequence[Sequence[int]]):
        """mctx->apply(): write each token's position and sequence ids into its cell
        ([P1] Крок 13а; [P4] process_ubatch: the only point where memory changes)."""
        for c, p, ss in zip(slots, pos, seq_ids):
            assert self.pos[c] < 0, "slot must be empty"
            self.pos[c] = int(p)
            self.seq[c, :] = False
            self.seq[c, [int(s) for s in ss]] = True

    def defrag_order(self) -> np.ndarray:
        """Where every cell's content comes from after a defrag ([P4] KVキャッシュの詳細:
        memory_update with optimize moves cells to close the gaps; the figure "After Defrag" shows
        the seven cells S0P0, S0P1, -, S1P0, S0P2, -, S1P1 becoming S0P0, S0P1, S0P2, S1P0, S1P1,
        -, -).

        reading (the figure's outcome): in each stream, the used cells packed from the stream's
        first cell, ordered by sequence then position; a cell shared by several sequences sorts
        under its lowest sequence id, and equal keys keep their cell order. Returns src [n_ctx]:
        new cell i takes old cell src[i] (-1: empty)."""
        src = np.full(len(self.pos), -1, dtype=np.int64)
        for s in range(self.n_stream):
            lo, hi = self.stream_range(s)
            used = lo + np.nonzero(self.pos[lo:hi] >= 0)[0]
            first_seq = np.array([int(np.argmax(self.seq[c])) for c in used], dtype=np.int64)
            src[lo:lo + len(used)] = used[np.lexsort((used, self.pos[used], first_seq))]
        return src

    def is_defragged(self) -> bool:
        src = self.defrag_order()
        return bool(np.all((src < 0) | (src == np.arange(len(src)))))

    def move(self, src: Sequence[int]):
        """Rewrite the cells so that cell i holds what old cell src[i] held (-1: empty)."""
        src = np.asarray(src, dtype=np.int64)
        keep = src >= 0
        pos = np.full_like(self.pos, -1)
        seq = np.zeros_like(self.seq)
        pos[keep] = self.pos[src[keep]]
        seq[keep] = self.seq[src[keep]]
        self.pos, self.seq = pos, seq

    def n_kv(self) -> int:
        """Cells the attention reads: highest used cell + 1 (reading of the 'recount' in apply)."""
        used = np.nonzero(self.pos >= 0)[0]
        return int(used[-1]) + 1 if len(used) else 0

    def mask(self, pos: Sequence[int], seq_ids: Sequence[Sequence[int]], n_kv: int) -> np.ndarray:
        """The KQ mask as booleans [T, n_kv] (True = visible).

        reading: token t may see cell c iff c holds a position, c shares a sequence with t, and
        c.pos <= pos(t) (causal); cells written by the same ubatch are included, because apply()
        and the K/V writes come before the attention ([P1] KV-cache section: K and V are appended
        first, then Q is multiplied by every key in the cache, including the current one)."""
        T = len(pos)
        m = np.zeros((T, n_kv), dtype=bool)
        cpos = self.pos[:n_kv]
        shares = {}                      # sequence set -> cells sharing one of its sequences
        for t in range(T):
            key = tuple(sorted(int(s) for s in seq_ids[t]))
            if key not in shares:
                shares[key] = self.seq[:n_kv][:, list(key)].any(axis=1)
            m[t] = shares[key] & (cpos >= 0) & (cpos <= pos[t])
        return m


def sanitize_batch(token, pos, n_seq_id, seq_id, logits, *, n_vocab: int, n_seq_max: int,
                   n_batch: int, cells: Optional[Cells], output_all: bool = False) -> Optional[Batch]:
    """llama_batch_allocr::init ([P1] Крок 10): validate, then fill the fields left as None.

    Invalid (returns None, which llama_decode turns into -1): no tokens; more than n_batch tokens;
    a token id outside [0, n_vocab); a sequence id outside [0, n_seq_max); a token with no
    sequence id.
    Defaults: seq_id None -> every token in sequence 0; pos None -> each sequence continues from
    seq_pos_max(s) + 1 in batch order (0 if there is no memory), and a token moves every one of its
    sequences past its position; logits None -> only the last token (all tokens if output_all).
    reading (the elided consistency checks): for each sequence, its positions in the batch must be
    consecutive in batch order and start at seq_pos_max(s) + 1; otherwise the batch is invalid.
    """
    n = 0 if token is None else len(token)
    if n <= 0 or n > n_batch:
        return None
    token = np.asarray(token, dtype=np.int64)
    if np.any(token < 0) or np.any(token >= n_vocab):
        return None
    if seq_id is None:
        sids = [[0] for _ in range(n)]
    else:
        sids = []
        for i in range(n):
            k = 1 if n_seq_id is None else int(n_seq_id[i])
            if k < 1:
                return None
            ss = [int(s) for s in seq_id[i][:k]]
            if any(s < 0 or s >= n_seq_max for s in ss):
                return None
            sids.append(ss)
    p0 = {}
    if pos is None:
        out_pos = np.zeros(n, dtype=np.int64)
        nxt = [0 if cells is None else cells.seq_pos_max(s) + 1 for s in range(n_seq_max)]
        for i in range(n):
            out_pos[i] = nxt[sids[i][0]]
            for s in sids[i]:
                nxt[s] = out_pos[i] + 1
    else:
        out_pos = np.asarray(pos, dtype=np.int64).copy()
    # consistency: per sequence, consecutive positions continuing the memory
    last = {}
    for i in range(n):
        for s in sids[i]:
            if s not in last:
                start = 0 if cells is None else cells.seq_pos_max(s) + 1
                if out_pos[i] != start:
                    return None
            elif out_pos[i] != last[s] + 1:
                return None
            last[s] = out_pos[i]
    if logits is None:
        out = np.zeros(n, dtype=bool)
        if output_all:
            out[:] = True
        else:
            out[-1] = True
    else:
        out = np.asarray(logits).astype(bool).copy()
        if output_all:
            out[:] = True
    return Batch(token.astype(np.int32), out_pos.astype(np.int32), sids, out)


def split_simple(n_tokens: int, n_ubatch: int) -> List[range]:
    """split_simple ([P1] Крок 12): the next at most n_ubatch unused tokens of the batch, in batch
    order, until the batch is used up. Returns the token ranges of the ubatches."""
    return [range(i, min(i + n_ubatch, n_tokens)) for i in range(0, n_tokens, n_ubatch)]


def split_equal(seq_of_token: Sequence[int], n_ubatch: int) -> List[List[int]]:
    """split_equal(n_ubatch, sequential = true) ([P1] Крок 12: the splitter of a cache with more
    than one stream; [P4] llama_ubatch: n_seq_tokens tokens per sequence set, n_seqs sets).

    reading (the pages give the call and the ubatch fields, not the steps): every token belongs
    to one sequence; a ubatch takes the sequences that still have unused tokens in ascending id,
    consecutive ids only ("sequential"), at most n_ubatch of them; each of the n_seqs sequences
    contributes the same number n_seq_tokens = min(n_ubatch // n_seqs, the fewest unused tokens
    among them) of its next unused tokens in batch order; the ubatch lists them sequence by
    sequence. Returns the batch indices of each ubatch."""
    queues = {}
    for i, s in enumerate(seq_of_token):
        queues.setdefault(int(s), []).append(i)
    heads = {s: 0 for s in queues}
    out = []
    while True:
        live = sorted(s for s in queues if heads[s] < len(queues[s]))
        if not live:
            return out
        sets = [live[0]]
        while len(sets) < n_ubatch and sets[-1] + 1 in live:
            sets.append(sets[-1] + 1)
        n_seq_tokens = min(n_ubatch // len(sets), min(len(queues[s]) - heads[s] for s in sets))
        ub = []
        for s in sets:
            ub.extend(queues[s][heads[s]:heads[s] + n_seq_tokens])
            heads[s] += n_seq_tokens
        out.append(ub)
