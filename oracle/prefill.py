"""Multi-query paged attention (prefill of new tokens over a paged cache).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``.

Several new tokens of one sequence attend at once: the tail of a long prompt
processed in chunks ("KV Cache：长上下文为什么吃显存，PagedAttention 怎么救"
§06, Chunked Prefill: the prompt is cut into pieces interleaved with
decode), the suffix after a prefix-cache hit ("推理与 KV Cache 02:分页、共享
与回收如何协作", 前缀索引与 Block Table: a hit skips the prefix's prefill, yet
the new suffix still reads the prefix's KV), or several speculative candidate
tokens ("企业官网建设流程全解析" §8.2).  Every new token is an ordinary
query of the new-token attention of "KV Cache：长上下文为什么吃显存" §01 at
its own position: it sees the cached tokens and the new tokens up to and
including itself.

Reading (the pages give no layout for the batch): queries are packed as
``q[T, H_q, D]`` with ``cu_seqlens[s] .. cu_seqlens[s+1]`` the new tokens of
sequence ``s``; ``context_lens[s]`` counts every token of the sequence after
the new ones are stored, so new token ``i`` of ``n`` sits at position
``context_lens[s] - n + i`` and attends to positions ``0 .. context_lens[s]
- n + i``.  ``n = 1`` is the decode step.
"""

from __future__ import annotations

import numpy as np

from .paged_attention import decode, dense_attention, gather_kv

__all__ = ["query_positions", "paged_attention_prefill"]


def query_positions(cu_seqlens, context_lens) -> np.ndarray:
    """Position of every packed query token (int64 [T])."""
    cu = np.asarray(cu_seqlens, np.int64)
    pos = np.empty(int(cu[-1]), np.int64)
    for s in range(len(cu) - 1):
        n = int(cu[s + 1] - cu[s])
        L = int(context_lens[s])
        if n > L:
            raise ValueError(f"sequence {s}: {n} new tokens but context length {L}")
        pos[cu[s]:cu[s + 1]] = np.arange(L - n, L)
    return pos


def paged_attention_prefill(q, k_cache, v_cache, block_tables, cu_seqlens, context_lens,
                            scale: float, dtype: str) -> np.ndarray:
    """``out[t, h, :]`` (float64) for every packed query token and head: the
    dense definition over the sequence's gathered rows ``0 .. position``,
    with query head h reading KV head h // G."""
    T, H_q, D = q.shape
    H_kv, K = k_cache.shape[2], k_cache.shape[1]
    G = H_q // H_kv
    q64 = decode(q, dtype)
    pos = query_positions(cu_seqlens, context_lens)
    out = np.zeros((T, H_q, D))
    cu = np.asarray(cu_seqlens, np.int64)
    for s in range(len(cu) - 1):
        L = int(context_lens[s])
        for j in range(H_kv):
            Kj = gather_kv(k_cache, block_tables[s], L, j, K, dtype)
            Vj = gather_kv(v_cache, block_tables[s], L, j, K, dtype)
            for t in range(int(cu[s]), int(cu[s + 1])):
                p = int(pos[t])
                for h in range(j * G, (j + 1) * G):
                    out[t, h] = dense_attention(q64[t, h], Kj[:p + 1], Vj[:p + 1], scale)
    return out
