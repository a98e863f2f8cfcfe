"""GB300-native (sm_103a) decode library for Llama-architecture GQA transformers with a KV cache.

The product is the C-ABI shared library libllm.so (include/llm.h, sources in csrc/); this package
holds its sources, its build script and a thin ctypes binding with the same call names.
"""
from .binding import (Context, LlmError, lib, F32, F16, BF16, Q8_0, LIB_PATH,  # noqa: F401
                      SIGNATURES)
