"""Model shapes and the five synthetic workloads (sizes, types, seeds), and the tensor-name list.

A workload is named by what it is. Seeds: workload k uses 1000+k for weights and 2000+k for
prompts; sequence s of workload k draws its prompt with seed (2000+k)*64+s.
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class HParams:
    n_layer: int
    n_embd: int
    n_head: int
    n_head_kv: int
    head_dim: int
    n_ff: int
    n_vocab: int
    rope_freq_base: float
    rms_eps: float
    rope_type: int = 0


# 4 layers, d 256, 8/2 heads, head_dim 32, n_ff 704, vocab 151936: ~80.6M parameters
TINY = HParams(4, 256, 8, 2, 32, 704, 151936, 10000.0, 1e-6)
# Llama-3-8B shape: 32 layers, d 4096, 32/8 heads, head_dim 128, n_ff 14336, vocab 128256
LLAMA8B = HParams(32, 4096, 32, 8, 128, 14336, 128256, 500000.0, 1e-5)


def tensor_specs(hp: HParams):
    """(name, ggml shape) of every llama tensor: ne0 is the row length, ne1 the row count."""
    d, qd, kvd = hp.n_embd, hp.n_head * hp.head_dim, hp.n_head_kv * hp.head_dim
    out = [("token_embd.weight", (d, hp.n_vocab)),
           ("output_norm.weight", (d,)),
           ("output.weight", (d, hp.n_vocab))]
    for il in range(hp.n_layer):
        p = f"blk.{il}."
        out += [(p + "attn_norm.weight", (d,)),
                (p + "attn_q.weight", (d, qd)),
                (p + "attn_k.weight", (d, kvd)),
                (p + "attn_v.weight", (d, kvd)),
                (p + "attn_output.weight", (qd, d)),
                (p + "ffn_norm.weight", (d,)),
                (p + "ffn_gate.weight", (d, hp.n_ff)),
                (p + "ffn_up.weight", (d, hp.n_ff)),
                (p + "ffn_down.weight", (hp.n_ff, d))]
    return out


@dataclass(frozen=True)
class Workload:
    key: str
    hp: HParams
    types: dict                 # storage type per tensor class
    type_kv: int                # 0 = F32, 1 = F16
    n_ctx: int
    n_seq: int
    n_prompt: int               # prompt tokens per sequence
    n_batch: int
    n_ubatch: int
    n_decode: int               # greedy decode steps (one token per sequence per step)
    weight_seed: int
    prompt_seed: int
    seq_rm_at: int = -1         # decode step after which seq 0 loses the upper half of its cache
    description: str = ""

    def prompt_seed_of(self, s: int) -> int:
        return self.prompt_seed * 64 + s if self.n_seq > 1 else self.prompt_seed


_F32, _F16, _BF16, _Q8 = 0, 1, 2, 8

WORKLOADS = {
    "tiny_f32_1seq": Workload(
        "tiny_f32_1seq", TINY, {"embd": _F32, "linear": _F32}, _F32,
        n_ctx=512, n_seq=1, n_prompt=32, n_batch=512, n_ubatch=512, n_decode=32,
        weight_seed=1001, prompt_seed=2001,
        description="tiny llama F32, 1 seq, 32-token prompt + 32 greedy steps, n_ctx 512, F32 KV"),
    "tiny_f32_8seq": Workload(
        "tiny_f32_8seq", TINY, {"embd": _F32, "linear": _F32}, _F16,
        n_ctx=4096, n_seq=8, n_prompt=128, n_batch=1024, n_ubatch=128, n_decode=128,
        weight_seed=1002, prompt_seed=2002,
        description="tiny llama F32, 8 seqs x 128-token prompts in one 1024 batch (ubatch 128), "
                    "unified F16 KV n_ctx 4096, 128 greedy steps of 8 tokens"),
    "llama8b_bf16_1seq": Workload(
        "llama8b_bf16_1seq", LLAMA8B, {"embd": _BF16, "linear": _BF16}, _F16,
        n_ctx=4096, n_seq=1, n_prompt=512, n_batch=512, n_ubatch=512, n_decode=256,
        weight_seed=1003, prompt_seed=2003,
        description="Llama-3-8B shape BF16, 512-token prompt (ubatch 512), n_ctx 4096, F16 KV, "
                    "256 greedy steps"),
    "llama8b_q8_0_8k": Workload(
        "llama8b_q8_0_8k", LLAMA8B, {"embd": _F32, "linear": _Q8}, _F16,
        n_ctx=8448, n_seq=1, n_prompt=8192, n_batch=8192, n_ubatch=512, n_decode=128,
        weight_seed=1004, prompt_seed=2004,
        description="Llama-3-8B shape, Q8_0 linear weights, F32 embeddings/norms, 8192-token "
                    "prompt in 512 ubatches, n_ctx 8448 (8192 + 128 decode cells, rounded to 256), "
                    "F16 KV, 128 greedy steps"),
    "llama8b_bf16_32seq": Workload(
        "llama8b_bf16_32seq", LLAMA8B, {"embd": _BF16, "linear": _BF16}, _F16,
        n_ctx=73728, n_seq=32, n_prompt=2048, n_batch=2048, n_ubatch=512, n_decode=256,
        weight_seed=1005, prompt_seed=2005, seq_rm_at=128,
        description="Llama-3-8B shape BF16, 32 seqs x 2048-token prompts (ubatch 512), unified "
                    "F16 KV n_ctx 73728, 256 steps of 32 tokens, seq_rm of half of seq 0 after "
                    "step 128"),
}
