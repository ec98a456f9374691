"""KV-cache byte accounting: memory sizes and the algorithmic bytes of a step.

* "19.2 KV Cache 系统化管理" §19.2.1: KV bytes = 2 * L * B * S * Kh * bytes,
  with Kh the total KV width (heads * head_dim).
* "KV Cache：长上下文为什么吃显存" §02: logical KV bytes =
  B * L * S * H_kv * D * 2 * bytes; for ragged batches sum over sequences.
* "推理与 KV Cache 02", section "按整块分配,会多占多少空间": a request of N
  tokens takes ceil(N / K) blocks and reserves ceil(N / K) * K token slots.
"""

from __future__ import annotations

from typing import Iterable


def kv_cache_bytes(layers: int, batch: int, seq_len: int, kv_heads: int,
                   head_dim: int, elem_bytes: int) -> int:
    return batch * layers * seq_len * kv_heads * head_dim * 2 * elem_bytes


def kv_cache_bytes_kh(layers: int, batch: int, seq_len: int, kv_dim: int,
                      elem_bytes: int) -> int:
    return 2 * layers * batch * seq_len * kv_dim * elem_bytes


def blocks_needed(num_tokens: int, block_size: int) -> int:
    return -(-num_tokens // block_size)


def reserved_slots(num_tokens: int, block_size: int) -> int:
    return blocks_needed(num_tokens, block_size) * block_size


def unused_slots(num_tokens: int, block_size: int) -> int:
    return reserved_slots(num_tokens, block_size) - num_tokens


def shareable_prefix_tokens(shared_tokens: int, block_size: int) -> int:
    """Whole-block sharing only: the common prefix rounded down to blocks."""
    return (shared_tokens // block_size) * block_size


def attention_kv_bytes(context_lens: Iterable[int], num_kv_heads: int,
                       head_dim: int, elem_bytes: int) -> int:
    """Algorithmic bytes one decode-attention launch must read: every valid
    cached token's K and V rows for every KV head, each read once."""
    return sum(int(L) for L in context_lens) * num_kv_heads * head_dim * 2 * elem_bytes


def kv_write_bytes(num_tokens: int, num_kv_heads: int, head_dim: int,
                   elem_bytes: int) -> int:
    """Read the new K/V rows and write them into the pool."""
    return 2 * (num_tokens * num_kv_heads * head_dim * 2 * elem_bytes)


def block_copy_bytes(num_pairs: int, block_size: int, num_kv_heads: int,
                     head_dim: int, elem_bytes: int) -> int:
    """Read the source blocks and write the destination blocks, K and V."""
    return 2 * num_pairs * block_size * num_kv_heads * head_dim * 2 * elem_bytes
