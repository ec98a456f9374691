"""Seeded synthetic decode-step workloads.

Builds the inputs of one decode step of one attention layer: block tables,
context lengths, new-token positions and copy-on-write pairs (from the host
block manager), plus seeded N(0, 1) query / key / value data.  Nothing here
computes any part of the device path (no slot arithmetic, no attention): the
same inputs feed the CUDA library and the CPU oracle.

The five named configurations follow the decode shapes used throughout:

* ``tiny``        4 seqs, lens {10, 7, 16, 3}, H_q=4, H_kv=2, D=64, K=4,
                  pool of 32 blocks in seeded order, fp32.
* ``qwen3_0_6b``  64 seqs, lens U[512, 4096], H_q=16, H_kv=8, D=128, K=16, bf16.
* ``mistral_7b``  128 seqs, half at 8192 and half U[1024, 8192], H_q=32,
                  H_kv=8, D=128, K=16, bf16.
* ``llama31_70b`` 4 seqs at 131072, H_q=64, H_kv=8, D=128, K=32, bf16.
* ``prefix_cow``  256 seqs sharing a 2048-token prefix plus U[16, 1024]-token
                  suffixes, each forked 4 ways (parallel sampling) so that
                  the first three writers of a shared partial block copy it;
                  H_q=32, H_kv=8, D=128, K=16, bf16.

Lengths count the token appended this step; it sits at position len - 1.
Pools are 1.25x the blocks needed (the tiny pool is fixed at 32).  Lengths
are integers drawn uniformly from the inclusive range with numpy's PCG64 seeded
by ``seed``; values are float32 draws of ``torch.randn`` under a CPU generator
seeded by ``seed`` (rounded to bfloat16 to nearest-even for bf16 runs).
"""

from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, List, Optional

import numpy as np

from .blockmgr import BlockPool, SeqBlocks


@dataclass
class Workload:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    dtype: str                      # "bf16" | "f32"
    block_tables: np.ndarray        # int32 [S, max_blocks_per_seq]
    context_lens: np.ndarray        # int32 [S]
    positions: np.ndarray           # int32 [S] (new token; -1 = no token)
    copy_pairs: np.ndarray          # int64 [n, 2] (src, dst)
    history_mask: np.ndarray        # bool [num_blocks, block_size]: slots holding data before the step
    scale: float

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def gqa_group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4


def _pad_tables(rows: List[List[int]], pad, rng) -> np.ndarray:
    maxB = max([len(r) for r in rows] + [1])
    if pad == "garbage":
        bt = rng.integers(-2**31, 2**31 - 1, size=(len(rows), maxB), dtype=np.int64)
    else:
        bt = np.full((len(rows), maxB), int(pad), dtype=np.int64)
    for s, r in enumerate(rows):
        bt[s, :len(r)] = r
    return bt.astype(np.int32)


def _history_mask(num_blocks, K, tables, hist_lens) -> np.ndarray:
    mask = np.zeros((num_blocks, K), dtype=bool)
    for row, L in zip(tables, hist_lens):
        for i in range(-(-L // K)):
            n = min(K, L - i * K)
            mask[row[i], :n] = True
    return mask


def build_decode(name: str, lens, num_q_heads: int, num_kv_heads: int,
                 head_dim: int, block_size: int, dtype: str = "bf16",
                 num_blocks: Optional[int] = None, pool_factor: float = 1.25,
                 seed: int = 0, pad="garbage") -> Workload:
    """A plain decode step: sequence ``s`` holds ``lens[s] - 1`` cached tokens
    and appends one more (a length of 0 means an empty sequence with no new
    token)."""
    lens = [int(x) for x in lens]
    K = block_size
    need = sum(-(-L // K) for L in lens)
    if num_blocks is None:
        num_blocks = max(1, math.ceil(need * pool_factor))
    rng = np.random.default_rng(seed)
    pool = BlockPool(num_blocks, seed=int(rng.integers(2**31)))
    seqs, positions = [], []
    for L in lens:
        sb = SeqBlocks(pool, K)
        if L > 0:
            sb.grow_to(L - 1)
            pos, pair = sb.append_token()
            assert pair is None
        else:
            pos = -1
        seqs.append(sb)
        positions.append(pos)
    pool.check_invariants(seqs)
    rows = [list(sb.mapping) for sb in seqs]
    return Workload(
        name=name, num_seqs=len(lens), num_q_heads=num_q_heads,
        num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=K,
        num_blocks=num_blocks, dtype=dtype,
        block_tables=_pad_tables(rows, pad, rng),
        context_lens=np.array(lens, dtype=np.int32),
        positions=np.array(positions, dtype=np.int32),
        copy_pairs=np.zeros((0, 2), dtype=np.int64),
        history_mask=_history_mask(num_blocks, K, rows, [max(L - 1, 0) for L in lens]),
        scale=1.0 / math.sqrt(head_dim))


def build_prefix_cow(num_parents: int = 256, prefix_len: int = 2048,
                     suffix_range=(16, 1024), fork: int = 4, num_q_heads: int = 32,
                     num_kv_heads: int = 8, head_dim: int = 128, block_size: int = 16,
                     dtype: str = "bf16", pool_factor: float = 1.25, seed: int = 0,
                     pad="garbage") -> Workload:
    """Shared-prefix + parallel-sampling fork.

    One owner table prefills ``prefix_len`` tokens (whole blocks).  Each of
    ``num_parents`` sequences shares those blocks (count = number of users)
    and prefills its own suffix.  Each parent is forked ``fork`` ways; every
    sample then appends one token.  A sample whose last block is partial and
    still shared copies it first (the first ``fork - 1`` writers copy, the
    last writes in place); a sample whose last block is full opens a new one.
    The step's tables are the samples' tables, ``fork * num_parents`` rows.
    """
    K = block_size
    if prefix_len % K:
        raise ValueError("prefix must be whole blocks")
    rng = np.random.default_rng(seed)
    suffix = rng.integers(suffix_range[0], suffix_range[1] + 1, size=num_parents)
    pblocks = prefix_len // K
    need = pblocks + sum(-(-(prefix_len + int(x)) // K) - pblocks + fork for x in suffix)
    num_blocks = math.ceil(need * pool_factor)
    pool = BlockPool(num_blocks, seed=int(rng.integers(2**31)))
    owner = SeqBlocks(pool, K)
    owner.grow_to(prefix_len)
    parents = []
    for x in suffix:
        sb = SeqBlocks(pool, K)
        sb.share_prefix(owner, pblocks)
        sb.grow_to(prefix_len + int(x))
        parents.append(sb)
    owner.release_all()            # the prefix now lives only through its users
    hist_rows = [list(p.mapping) for p in parents]
    hist_lens = [p.num_tokens for p in parents]
    samples, positions, pairs = [], [], []
    for p in parents:
        kids = [p] + [p.fork() for _ in range(fork - 1)]
        # children 1..fork-1 write first, the original writes last
        order = list(range(1, fork)) + [0]
        got = {}
        for c in order:
            pos, pair = kids[c].append_token()
            got[c] = pos
            if pair is not None:
                pairs.append(pair)
        for c in range(fork):
            samples.append(kids[c])
            positions.append(got[c])
    pool.check_invariants(samples)
    rows = [list(sb.mapping) for sb in samples]
    lens = [sb.num_tokens for sb in samples]
    return Workload(
        name="prefix_cow", num_seqs=len(samples), num_q_heads=num_q_heads,
        num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=K,
        num_blocks=num_blocks, dtype=dtype,
        block_tables=_pad_tables(rows, pad, rng),
        context_lens=np.array(lens, dtype=np.int32),
        positions=np.array(positions, dtype=np.int32),
        copy_pairs=np.array(pairs, dtype=np.int64).reshape(-1, 2),
        history_mask=_history_mask(num_blocks, K, hist_rows, hist_lens),
        scale=1.0 / math.sqrt(head_dim))


def build(name: str, seed: int = 0, pad="garbage", block_size: Optional[int] = None) -> Workload:
    """The named workload; ``block_size`` replaces its block size (the same
    lengths and shapes, a pool re-cut into blocks of that many tokens), for
    block-size sweeps."""
    rng = np.random.default_rng(10_000 + seed)

    def K(default):
        return int(block_size) if block_size else default

    if name == "tiny":
        return build_decode("tiny", [10, 7, 16, 3], 4, 2, 64, K(4), "f32",
                            num_blocks=32 if not block_size else None, seed=seed, pad=pad)
    if name == "qwen3_0_6b":
        lens = rng.integers(512, 4096 + 1, size=64)
        return build_decode(name, lens, 16, 8, 128, K(16), "bf16", seed=seed, pad=pad)
    if name == "mistral_7b":
        lens = np.concatenate([np.full(64, 8192), rng.integers(1024, 8192 + 1, size=64)])
        lens = rng.permutation(lens)
        return build_decode(name, lens, 32, 8, 128, K(16), "bf16", seed=seed, pad=pad)
    if name == "llama31_70b":
        return build_decode(name, [131072] * 4, 64, 8, 128, K(32), "bf16", seed=seed, pad=pad)
    if name == "prefix_cow":
        return build_prefix_cow(seed=seed, pad=pad, block_size=K(16))
    raise KeyError(name)


CONFIG_NAMES = ("tiny", "qwen3_0_6b", "mistral_7b", "llama31_70b", "prefix_cow")


def swap_plan(w, seed: int):
    """Every other sequence of the workload is preempted by swap: its blocks
    (K and V) go to a host pool in a seeded shuffled order, and come back into
    a seeded permutation of the same GPU blocks (scattered placement)."""
    import numpy as np
    rng = np.random.default_rng(seed + 101)
    blocks = []
    for s in range(1, w.num_seqs, 2):
        n = -(-int(w.context_lens[s]) // w.block_size)
        blocks.extend(int(b) for b in w.block_tables[s, :n])
    blocks = np.array(blocks, np.int64)
    host = rng.permutation(len(blocks)).astype(np.int64)
    out_pairs = np.stack([blocks, host], 1)
    in_pairs = np.stack([host, rng.permutation(blocks)], 1)
    return out_pairs, in_pairs


# --------------------------------------------------------------------------
# tensors
# --------------------------------------------------------------------------

def _torch_dtype(dtype: str):
    import torch
    return {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]


def fill_normal_(t, gen, chunk_elems: int = 1 << 26):
    """Fill ``t`` (any float dtype, any device) with N(0, 1) float32 draws
    rounded to ``t``'s dtype, chunk by chunk (bounded host memory)."""
    import torch
    flat = t.view(-1)
    n = flat.numel()
    dev = gen.device
    for a in range(0, n, chunk_elems):
        b = min(n, a + chunk_elems)
        x = torch.randn(b - a, generator=gen, dtype=torch.float32, device=dev)
        flat[a:b].copy_(x.to(t.dtype))
    return t


def materialize(w: Workload, device="cpu", seed: int = 0, canary: bool = True,
                values_device: Optional[str] = None) -> Dict[str, "object"]:
    """Torch tensors for one step of ``w``.

    ``canary``: slots that hold no history before the step are set to NaN, so
    any read of them shows up in the output.  ``values_device``: where the
    random pool values are drawn ("cpu" by default; "cuda" draws them with a
    seeded CUDA generator, used only for large timing runs).
    """
    import torch
    td = _torch_dtype(w.dtype)
    vdev = values_device or "cpu"
    gen = torch.Generator(device=vdev)
    gen.manual_seed(seed)
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    k_cache = fill_normal_(torch.empty(shape, dtype=td, device=vdev), gen)
    v_cache = fill_normal_(torch.empty(shape, dtype=td, device=vdev), gen)
    if canary:
        m = torch.from_numpy(~w.history_mask).to(vdev)
        k_cache[m] = float("nan")
        v_cache[m] = float("nan")
    q = fill_normal_(torch.empty(w.num_seqs, w.num_q_heads, w.head_dim, dtype=td, device=vdev), gen)
    k_new = fill_normal_(torch.empty(w.num_seqs, w.num_kv_heads, w.head_dim, dtype=td, device=vdev), gen)
    v_new = fill_normal_(torch.empty(w.num_seqs, w.num_kv_heads, w.head_dim, dtype=td, device=vdev), gen)
    out = dict(
        k_cache=k_cache, v_cache=v_cache, q=q, k_new=k_new, v_new=v_new,
        block_tables=torch.from_numpy(w.block_tables.copy()),
        context_lens=torch.from_numpy(w.context_lens.copy()),
        positions=torch.from_numpy(w.positions.copy()),
        copy_pairs=torch.from_numpy(w.copy_pairs.copy()),
    )
    return {k: v.to(device) for k, v in out.items()}


# --------------------------------------------------------------------------
# multi-query (prefill) workloads
# --------------------------------------------------------------------------

@dataclass
class PrefillWorkload:
    """Sequences with ``prefix[s]`` cached tokens and ``news[s]`` new tokens
    (queries packed by ``cu_seqlens``); ``context_lens = prefix + news``."""
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    prefix: np.ndarray
    news: np.ndarray
    block_tables: np.ndarray
    scale: float

    @property
    def context_lens(self) -> np.ndarray:
        return (self.prefix + self.news).astype(np.int32)

    @property
    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.news)]).astype(np.int32)

    @property
    def num_seqs(self) -> int:
        return len(self.news)

    @property
    def num_tokens(self) -> int:
        return int(self.news.sum())


def build_prefill(name: str, seed: int = 0) -> PrefillWorkload:
    """``suffix_prefill``: 32 requests that hit a cached prefix of U[1024, 4096]
    tokens and prefill a 512-token suffix ("推理与 KV Cache 02", 前缀索引与
    Block Table), Mistral-7B attention shape.  ``chunked_prefill``: 64
    requests with U[1024, 4096] tokens already cached, each prefilling its
    next 32-token chunk ("KV Cache：长上下文为什么吃显存，PagedAttention 怎么救"
    §06: a long prompt's prefill cut into small chunks interleaved with decode
    steps), Mistral-7B attention shape.  ``speculative_decode``: the
    Qwen3-0.6B decode batch (64 sequences, U[512, 4096] cached tokens) with 4
    candidate tokens each ("企业官网建设流程全解析" §8.2)."""
    rng = np.random.default_rng(20_000 + seed)
    if name == "suffix_prefill":
        prefix = rng.integers(1024, 4096 + 1, size=32)
        news = np.full(32, 512)
        H_q, H_kv, D, K = 32, 8, 128, 16
    elif name == "chunked_prefill":
        prefix = rng.integers(1024, 4096 + 1, size=64)
        news = np.full(64, 32)
        H_q, H_kv, D, K = 32, 8, 128, 16
    elif name == "speculative_decode":
        prefix = rng.integers(512, 4096 + 1, size=64)
        news = np.full(64, 4)
        H_q, H_kv, D, K = 16, 8, 128, 16
    else:
        raise KeyError(name)
    lens = prefix + news
    need = int(sum(-(-int(L) // K) for L in lens))
    nb = math.ceil(need * 1.25)
    pool = BlockPool(nb, seed=int(rng.integers(2**31)))
    rows = []
    for L in lens:
        sb = SeqBlocks(pool, K)
        sb.grow_to(int(L))
        rows.append(list(sb.mapping))
    return PrefillWorkload(name=name, num_q_heads=H_q, num_kv_heads=H_kv, head_dim=D,
                           block_size=K, num_blocks=nb, prefix=prefix.astype(np.int64),
                           news=news.astype(np.int64),
                           block_tables=_pad_tables(rows, "garbage", rng),
                           scale=1.0 / math.sqrt(D))


PREFILL_NAMES = ("suffix_prefill", "chunked_prefill", "speculative_decode")
