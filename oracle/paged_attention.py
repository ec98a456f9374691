"""Plain, slow, fp64 CPU oracle of the paged decode path.

TEST INFRASTRUCTURE ONLY (see the package docstring): only tests/, the smoke
check and bench.py's CPU-baseline legs may call this module.

Conventions (all numpy, row-major):

* ``k_cache`` / ``v_cache``: ``[num_blocks, block_size, num_kv_heads, head_dim]``,
  the pool layout of "19.2 KV Cache 系统化管理" §19.2.3 (``PhysicalBlockPool``:
  ``[num_blocks, block_size, num_heads, head_dim]``), with the head axis holding
  the KV heads.  Floating-point pools are passed as their raw storage: float32
  arrays for ``"f32"`` and uint16 bit patterns for ``"bf16"``; :func:`decode`
  turns them into exact float64.
* ``block_tables``: int ``[num_seqs, max_blocks_per_seq]``; row ``s`` maps
  logical block ``i`` of sequence ``s`` to a physical block id.  Entries past
  ``ceil(len_s / block_size)`` are never read.
* ``context_lens``: int ``[num_seqs]``, the number of cached tokens attention
  reads, counting the token appended in this decode step.
* ``q``: ``[num_seqs, num_q_heads, head_dim]``; query head ``h`` reads KV head
  ``h // G`` with ``G = num_q_heads // num_kv_heads``.

Readings taken where the pages leave a step open are stated inline.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "decode",
    "slot_mapping",
    "kv_write",
    "kv_block_copy",
    "kv_block_swap",
    "gather_kv",
    "dense_attention",
    "attention_rows",
    "paged_attention_decode",
    "paged_attention_decode_one",
    "paged_attention_streaming",
    "partial_state",
    "merge_partials",
]


# --------------------------------------------------------------------------
# storage decoding
# --------------------------------------------------------------------------

def decode(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact conversion of stored values to float64.

    ``"f32"``: IEEE binary32 values (float32, or their uint32 bit patterns),
    widened exactly.
    ``"bf16"``: bfloat16 bit patterns (uint16).  A bfloat16 number is the upper
    half of the binary32 number with the same sign, exponent and leading seven
    mantissa bits, so shifting the pattern into the high 16 bits of a 32-bit
    word gives that binary32 number exactly.
    """
    if dtype == "f32":
        a = np.asarray(x)
        if a.dtype == np.uint32:
            a = a.view(np.float32)
        return a.astype(np.float32).astype(np.float64)
    if dtype == "bf16":
        bits = np.asarray(x).view(np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


# --------------------------------------------------------------------------
# a1: slot mapping
# --------------------------------------------------------------------------

def slot_mapping(block_tables: np.ndarray, positions: np.ndarray,
                 block_size: int) -> np.ndarray:
    """Flattened token slot of each sequence's token at ``positions[s]``.

    "推理与 KV Cache 02", section "从一个位置找到缓存块": for position ``t``,
    logical block = floor(t / K), offset = t mod K, and the token slot is
    physical_block_id * K + offset.  Same arithmetic as ``append_token`` in
    "19.2 KV Cache 系统化管理" §19.2.3.

    Reading: a negative position marks a padding entry and maps to slot -1.
    """
    bt = np.asarray(block_tables)
    pos = np.asarray(positions)
    out = np.empty(pos.shape[0], dtype=np.int64)
    for s in range(pos.shape[0]):
        t = int(pos[s])
        if t < 0:
            out[s] = -1
            continue
        logical = t // block_size
        offset = t % block_size
        physical = int(bt[s, logical])
        out[s] = physical * block_size + offset
    return out


# --------------------------------------------------------------------------
# a2: slot-mapped KV append
# --------------------------------------------------------------------------

def kv_write(k_cache: np.ndarray, v_cache: np.ndarray, k: np.ndarray,
             v: np.ndarray, slots: np.ndarray):
    """Return copies of the pools with token ``i``'s K/V rows stored at ``slots[i]``.

    "19.2 KV Cache 系统化管理" §19.2.3, ``write_slot``: the pool entry
    ``[block, slot_in_block]`` (all heads) is overwritten by the token's key and
    value.  With the pool viewed as ``[num_blocks * K, heads, head_dim]`` the
    entry is indexed by the flattened token slot of "推理与 KV Cache 02".

    The copy is of raw storage (bit exact): pass the pools and rows as arrays
    of the same storage dtype.  Reading: slot -1 is a padding token and is
    skipped.  Tokens are applied in order.
    """
    nb, K = k_cache.shape[0], k_cache.shape[1]
    kc = k_cache.copy().reshape(nb * K, *k_cache.shape[2:])
    vc = v_cache.copy().reshape(nb * K, *v_cache.shape[2:])
    for i in range(len(slots)):
        s = int(slots[i])
        if s < 0:
            continue
        kc[s] = k[i]
        vc[s] = v[i]
    return kc.reshape(k_cache.shape), vc.reshape(v_cache.shape)


# --------------------------------------------------------------------------
# a5: copy-on-write block copy
# --------------------------------------------------------------------------

def kv_block_copy(k_cache: np.ndarray, v_cache: np.ndarray, pairs: np.ndarray):
    """Return copies of the pools with block ``dst`` holding block ``src``'s data.

    "19.2 KV Cache 系统化管理" §19.2.2 (写时复制): when a sequence must write
    into a physical block whose reference count is above one, a new block is
    allocated and the original contents are copied into it before the write.
    This is that copy, for K and for V, applied pair by pair in order.
    """
    kc = k_cache.copy()
    vc = v_cache.copy()
    for src, dst in np.asarray(pairs).reshape(-1, 2):
        kc[int(dst)] = kc[int(src)]
        vc[int(dst)] = vc[int(src)]
    return kc, vc


def kv_block_swap(src_k: np.ndarray, src_v: np.ndarray, dst_k: np.ndarray,
                  dst_v: np.ndarray, pairs: np.ndarray):
    """Return copies of the destination pools with block ``dst`` holding the
    source pool's block ``src``, for K and for V.

    Swap between GPU memory and host memory ("19.2 KV Cache 系统化管理",
    §19.2.6 调度与抢占, Swap: a preempted request's KV blocks are parked in
    CPU memory and brought back when GPU memory frees up;
    "企业官网建设流程全解析" §8.2: the oldest blocks move to CPU memory and
    return on demand while the block table keeps the logical view).  The two pools have the same block geometry but
    different block counts; the source is never written, so the pairs are
    independent of their order.
    """
    dk = dst_k.copy()
    dv = dst_v.copy()
    for src, dst in np.asarray(pairs).reshape(-1, 2):
        dk[int(dst)] = src_k[int(src)]
        dv[int(dst)] = src_v[int(src)]
    return dk, dv


# --------------------------------------------------------------------------
# a3 + a4: decode attention
# --------------------------------------------------------------------------

def gather_kv(cache: np.ndarray, block_table_row: np.ndarray, length: int,
              kv_head: int, block_size: int, dtype: str) -> np.ndarray:
    """Contiguous ``[length, head_dim]`` float64 rows of one sequence and KV head.

    Token ``t`` lives in physical block ``block_table_row[t // K]`` at offset
    ``t % K`` ("推理与 KV Cache 02", "从一个位置找到缓存块").
    """
    t = np.arange(length, dtype=np.int64)
    phys = np.asarray(block_table_row, dtype=np.int64)[t // block_size]
    off = t % block_size
    return decode(cache[phys, off, kv_head, :], dtype)


def dense_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray,
                    scale: float) -> np.ndarray:
    """softmax(scale * q K^T) V for one query row over contiguous K, V (fp64).

    "KV Cache：长上下文为什么吃显存" §01: the new token's query attends to all
    cached keys ``K_{1:t}`` and weights ``V_{1:t}``.  Two passes: the maximum
    score is subtracted before exponentiating (this changes nothing
    mathematically).  Reading: an empty context gives a zero output.
    """
    q = np.asarray(q, dtype=np.float64)
    if K.shape[0] == 0:
        return np.zeros(V.shape[1], dtype=np.float64)
    z = scale * (K @ q)
    w = np.exp(z - z.max())
    w /= w.sum()
    return w @ V


def attention_rows(Q: np.ndarray, K: np.ndarray, V: np.ndarray, limits,
                   scale: float) -> np.ndarray:
    """:func:`dense_attention` for several query rows over the same contiguous
    K, V (fp64): row ``i`` attends to keys ``0 .. limits[i]`` inclusive
    ("KV Cache：长上下文为什么吃显存" §01, the new token at position t sees
    ``K_{1:t}``).  All scores come from one matrix product; keys past a row's
    limit get weight zero; each row's maximum is subtracted before
    exponentiating.  A row with a negative limit sees no key and gives zeros.
    """
    Q = np.asarray(Q, dtype=np.float64)
    lim = np.asarray(limits, dtype=np.int64).reshape(-1)
    out = np.zeros((Q.shape[0], V.shape[1]), dtype=np.float64)
    if K.shape[0] == 0 or Q.shape[0] == 0:
        return out
    z = scale * (Q @ K.T)                                     # [rows, keys]
    visible = np.arange(K.shape[0])[None, :] <= lim[:, None]
    live = visible.any(axis=1)
    z = np.where(visible, z, -np.inf)
    m = np.where(live, z.max(axis=1), 0.0)
    w = np.where(visible, np.exp(z - m[:, None]), 0.0)
    tot = w.sum(axis=1)
    out[live] = (w[live] @ V) / tot[live, None]
    return out


def paged_attention_decode_one(q: np.ndarray, k_cache: np.ndarray,
                               v_cache: np.ndarray, block_tables: np.ndarray,
                               context_lens: np.ndarray, scale: float,
                               s: int, h: int, dtype: str) -> np.ndarray:
    """Output row ``out[s, h, :]`` (fp64): gather through the block table, then
    the dense definition.

    GQA reading ("KV Cache：长上下文为什么吃显存" §02 gives only the ratio
    H_kv / H_q and says query heads are grouped): query heads are grouped
    contiguously, query head ``h`` uses KV head ``h // G``.
    """
    H_q = q.shape[1]
    H_kv = k_cache.shape[2]
    G = H_q // H_kv
    K = k_cache.shape[1]
    L = int(context_lens[s])
    j = h // G
    Kj = gather_kv(k_cache, block_tables[s], L, j, K, dtype)
    Vj = gather_kv(v_cache, block_tables[s], L, j, K, dtype)
    return dense_attention(decode(q[s, h], dtype), Kj, Vj, scale)


def paged_attention_decode(q: np.ndarray, k_cache: np.ndarray,
                           v_cache: np.ndarray, block_tables: np.ndarray,
                           context_lens: np.ndarray, scale: float,
                           dtype: str) -> np.ndarray:
    """``out[s, h, :]`` for every sequence and query head, float64.

    For each sequence and KV head the rows are gathered once and shared by the
    ``G`` query heads of its group (same arithmetic as calling
    :func:`paged_attention_decode_one` per head).
    """
    S, H_q, D = q.shape
    H_kv = k_cache.shape[2]
    G = H_q // H_kv
    K = k_cache.shape[1]
    out = np.zeros((S, H_q, D), dtype=np.float64)
    q64 = decode(q, dtype)
    for s in range(S):
        L = int(context_lens[s])
        for j in range(H_kv):
            Kj = gather_kv(k_cache, block_tables[s], L, j, K, dtype)
            Vj = gather_kv(v_cache, block_tables[s], L, j, K, dtype)
            for h in range(j * G, (j + 1) * G):
                out[s, h] = dense_attention(q64[s, h], Kj, Vj, scale)
    return out


def paged_attention_streaming(q: np.ndarray, k_cache: np.ndarray,
                              v_cache: np.ndarray, block_table_row: np.ndarray,
                              length: int, scale: float, dtype: str) -> np.ndarray:
    """One sequence, all query heads, in the pages' block-by-block form (fp64).

    "19.2 KV Cache 系统化管理" §19.2.3, ``paged_attention``: walk the block
    table in logical order; in each block only ``min(K, remaining)`` slots are
    valid; scores are ``q . k * scale``; keep a running maximum, a running sum
    of exponentials and a running weighted sum of values, rescaling the old
    sum and output by ``exp(old_max - new_max)`` whenever the maximum grows;
    divide by the sum at the end.  Restated here in float64 with GQA.
    """
    H_q, D = q.shape
    H_kv = k_cache.shape[2]
    G = H_q // H_kv
    K = k_cache.shape[1]
    q64 = decode(q, dtype)
    run_max = np.full(H_q, -np.inf)
    run_sum = np.zeros(H_q)
    acc = np.zeros((H_q, D))
    remaining = int(length)
    n_blocks = -(-remaining // K)
    for i in range(n_blocks):
        phys = int(block_table_row[i])
        valid = min(K, remaining)
        remaining -= valid
        for h in range(H_q):
            j = h // G
            keys = decode(k_cache[phys, :valid, j, :], dtype)    # [valid, D]
            vals = decode(v_cache[phys, :valid, j, :], dtype)
            scores = (keys @ q64[h]) * scale                     # [valid]
            new_max = max(run_max[h], scores.max())
            old_scale = np.exp(run_max[h] - new_max)
            new_w = np.exp(scores - new_max)
            run_sum[h] = run_sum[h] * old_scale + new_w.sum()
            acc[h] = acc[h] * old_scale + new_w @ vals
            run_max[h] = new_max
    out = np.zeros((H_q, D))
    nz = run_sum > 0
    out[nz] = acc[nz] / run_sum[nz, None]
    return out


# --------------------------------------------------------------------------
# split-K partial states and their merge
# --------------------------------------------------------------------------

def partial_state(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """(m, l, o) of one query row over a subset of tokens (fp64).

    ``m`` = max score, ``l`` = sum of exp(score - m), ``o`` = unnormalised
    sum of exp(score - m) * v.  The same three running quantities that the
    block loop of §19.2.3 keeps; an empty subset gives (-inf, 0, 0).
    """
    q = np.asarray(q, dtype=np.float64)
    if K.shape[0] == 0:
        return -np.inf, 0.0, np.zeros(V.shape[1])
    z = scale * (K @ q)
    m = z.max()
    w = np.exp(z - m)
    return m, w.sum(), w @ V


def merge_partials(ms, ls, os_):
    """Merge split-K partials of one query row into the normalised output.

    Same rescaling identity as the online softmax of §19.2.3: with
    M = max_p m_p, the merged sum is sum_p l_p exp(m_p - M) and the merged
    output is sum_p o_p exp(m_p - M) divided by that sum.  Partials with
    m_p = -inf (empty subsets) contribute nothing; all-empty gives zeros.
    """
    ms = np.asarray(ms, dtype=np.float64)
    ls = np.asarray(ls, dtype=np.float64)
    os_ = np.asarray(os_, dtype=np.float64)
    live = np.isfinite(ms)
    if not live.any():
        return np.zeros(os_.shape[-1])
    M = ms[live].max()
    w = np.zeros_like(ms)
    w[live] = np.exp(ms[live] - M)
    L = (ls * w).sum()
    return (os_ * w[:, None]).sum(axis=0) / L
