"""KV-cache byte arithmetic from the pages, as plain formulas.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

"DeepSeek V4 in vLLM", appendix "the arithmetic behind 8.7x":
* V3.2-style stack: per token per layer an MLA entry plus an indexer entry,
  61 layers, 1,048,576 tokens.
* V4: 30 c4a layers (shared KV entry per 4 tokens + indexer entry per 4
  tokens) and 31 c128a layers (shared KV entry per 128 tokens).
The page prints per-entry sizes (MLA 512*2 = 1024 B, indexer 64*2 = 128 B)
that do NOT reproduce its own totals (83.9 GiB, 9.62 GiB); the totals are
reproduced with MLA = (512+64)*2 = 1152 B and indexer = 128*2 = 256 B.  Both
variants are exposed so the tests can show which one the totals follow.
SGLang KV-pool article, section "DSA": indexer = 128 fp8 B + 4 B scale = 132 B;
section "DeepSeek-V4": 448 fp8 nope + 64 bf16 rope + 7 scale + 1 pad = 584 B.
"""
from __future__ import annotations

GIB = 2.0 ** 30
TOKENS_1M = 1 << 20


def v32_stack_bytes(mla_entry: int, indexer_entry: int, layers: int = 61,
                    tokens: int = TOKENS_1M) -> float:
    return (mla_entry + indexer_entry) * tokens * layers


def v4_stack_bytes(kv_entry: int, indexer_entry: int, c4a_layers: int = 30,
                   c128a_layers: int = 31, tokens: int = TOKENS_1M) -> float:
    c4a = c4a_layers * (kv_entry + indexer_entry) * tokens / 4
    c128a = c128a_layers * kv_entry * tokens / 128
    return c4a + c128a


def sglang_indexer_entry(head_dim: int = 128, quant_block: int = 128) -> int:
    return head_dim + (head_dim // quant_block) * 4


def sglang_dsv4_entry(nope: int = 448, rope_dims: int = 64, scale_block: int = 64) -> int:
    return nope + rope_dims * 2 + nope // scale_block + 1
