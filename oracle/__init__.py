"""CPU oracle of llama_decode over a Llama GQA transformer with a KV cache.

TEST INFRASTRUCTURE ONLY. Nothing in the product package imports, calls or links this code; only
tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference legs use it.

The oracle is plain and slow on purpose: numpy float64 arithmetic (one library matmul per
projection), Python loops for the batch / KV-cell bookkeeping, a dense attention mask, and no
blocking, fusion or reordering beyond what the definitions state. It shares no code with the CUDA
path; the only common module is `synthetic` (seeded inputs, no method arithmetic).

Sources, cited by page title and section:
  [P1] "llama.cpp AI LLM Engine - Як це працює" (romankryvolapov.pages.dev/uk/llama-cpp/):
       Крок 10 (llama_batch, llama_batch_allocr::init), Крок 11 (llama_decode, decode loop,
       return codes), Крок 12 (llama_kv_cache::init_batch), Крок 13а-13в (process_ubatch,
       apply, graph layer scheme, set_inputs), Крок 14 (llama_get_logits_ith), KV-cache section.
  [P2] "llama.cpp Architecture" (codeloopback.dev/articles/llm-llama-cpp-architecture):
       Example 2 (tensor shapes/strides, Q8_0 blocks), Example 4 (the decode-step graph),
       Example 8-10 (hparams, context parameters, buffer sizes), Example 11 (compute buffer,
       non-fused attention nodes), Example 13 (bytes / FLOPs per token).
  [P4] "デコードループ：バッチ処理、KVキャッシュ、メモリ管理" (readoss.com): バッチパイプライン,
       KVキャッシュの詳細, エラーリカバリとステートロールバック.

Readings taken where the pages are silent are marked "reading:" in the docstrings. Whole-forward logits are "parity unpinned" by the pages (they print
no logits for a reproducible input); the forward pass is pinned by closed forms, analytic models
and invariants in tests/test_oracle_*.py.
"""
from .formats import (decode_weight, round_to_type, F32, F16, BF16, Q8_0)  # noqa: F401
from .numerics import (rms_norm, rope, attention, silu, swiglu, linear)    # noqa: F401
from .memory import (Cells, sanitize_batch, split_simple, derive_cparams,   # noqa: F401
                     LLAMA_MAX_SEQ, DecodeStatus)
from .context import OracleContext, OracleWeights                            # noqa: F401
from .sampling import SamplerParams, sample as sample_chain                   # noqa: F401
