"""Host block manager, workload generator and byte accounting (CPU only)."""

import numpy as np
import pytest

from paged_kv_cache_115_gb300 import accounting as acc
from paged_kv_cache_115_gb300.blockmgr import (BlockPool, PoolExhausted, SeqBlocks, swap_in,
                                              swap_out)
from paged_kv_cache_115_gb300 import workloads as wl


def test_p1_selfcheck_block_accounting(golden):
    g = golden("p1_selfcheck.json")
    pool = BlockPool(g["num_blocks"])          # page order: pop from list(range(n))
    t = SeqBlocks(pool, g["block_size"])
    for _ in range(g["num_tokens"]):
        t.append_token()
    assert len(t.mapping) == g["blocks_used"]
    assert t.mapping == [15, 14, 13]
    t.release_all()
    assert pool.num_free == g["free_after_release"]


def test_p3_table_from_free_list(golden):
    g = golden("p3_block_table_example.json")
    pool = BlockPool(8)
    pool.free_list = [b for b in range(8) if b not in g["block_table"]] + g["block_table"][::-1]
    t = SeqBlocks(pool, g["block_size"])
    for _ in range(g["num_tokens"]):
        t.append_token()
    assert t.mapping == g["block_table"]
    assert acc.unused_slots(g["num_tokens"], g["block_size"]) == \
        g["block_size"] - g["used_slots_in_last_block"]


def test_p1_lifecycle(golden):
    g = golden("p1_lifecycle_example.json")
    pool = BlockPool(8)
    order = g["final_block_table"]
    pool.free_list = [b for b in range(8) if b not in order] + order[::-1]
    t = SeqBlocks(pool, g["block_size"])
    t.grow_to(g["prompt_tokens"])
    assert t.mapping == g["prefill_blocks"]
    for step in g["decode"]:
        before = len(t.mapping)
        pos, pair = t.append_token()
        assert pos == step["position"] and pair is None
        assert (len(t.mapping) > before) == step["allocates"]
        assert t.mapping[pos // g["block_size"]] == step["physical_block"]
    assert t.mapping == g["final_block_table"]


def test_exhaustion_raises():
    pool = BlockPool(2)
    pool.allocate(), pool.allocate()
    with pytest.raises(PoolExhausted):
        pool.allocate()


def test_refcount_lifecycle_and_cow():
    # two users of one block: count 2 -> 1 -> 0 ("推理与 KV Cache 02", recycling section)
    pool = BlockPool(4)
    a = SeqBlocks(pool, 4)
    a.grow_to(3)
    b = a.fork()
    blk = a.mapping[0]
    assert pool.ref_counts[blk] == 2
    # B writes into the shared partial block: copy-on-write
    pos, pair = b.append_token()
    assert pos == 3 and pair is not None and pair[0] == blk
    assert pool.ref_counts[blk] == 1 and pool.ref_counts[pair[1]] == 1
    # A is now the only user and writes in place
    pos, pair = a.append_token()
    assert pair is None
    a.release_all()
    assert pool.ref_counts[blk] == 0 and blk in pool.free_list
    b.release_all()
    assert pool.num_free == 4
    pool.check_invariants([])


def test_random_ops_keep_invariants():
    rng = np.random.default_rng(3)
    pool = BlockPool(200, seed=1)
    live = []
    for step in range(400):
        op = rng.integers(0, 4)
        try:
            if op == 0 or not live:
                s = SeqBlocks(pool, 8)
                try:
                    s.grow_to(int(rng.integers(0, 40)))
                except PoolExhausted:
                    s.release_all()           # give back a partial prefill
                    raise
                live.append(s)
            elif op == 1:
                live.append(live[int(rng.integers(len(live)))].fork())
            elif op == 2:
                live[int(rng.integers(len(live)))].append_token()
            else:
                live.pop(int(rng.integers(len(live)))).release_all()
        except PoolExhausted:
            for _ in range(len(live) // 2):   # preempt half the requests
                live.pop(0).release_all()
        pool.check_invariants(live)
        for s in live:
            assert len(s.mapping) == acc.blocks_needed(s.num_tokens, 8)
            assert acc.unused_slots(s.num_tokens, 8) <= 7   # tail waste <= K - 1
    for s in live:
        s.release_all()
    assert pool.num_free == 200


def test_invariant_checker_catches_leak_and_undercount():
    pool = BlockPool(4)
    s = SeqBlocks(pool, 2)
    s.grow_to(3)
    pool.free_list.pop()                         # leak a free block
    with pytest.raises(AssertionError):
        pool.check_invariants([s])
    pool = BlockPool(4)
    s = SeqBlocks(pool, 2)
    s.grow_to(3)
    t = SeqBlocks(pool, 2, list(s.mapping), 3)   # shared without counting
    with pytest.raises(AssertionError):
        pool.check_invariants([s, t])


def test_tail_waste_table(golden):
    g = golden("p3_tail_waste.json")
    for r in g["rows"]:
        assert acc.blocks_needed(r["num_tokens"], r["block_size"]) == r["blocks"]
        assert acc.unused_slots(r["num_tokens"], r["block_size"]) == r["unused_slots"]
    b = g["bytes_example"]
    per_tok = b["bytes_per_token_kib"] * 1024
    assert b["num_tokens"] * per_tok / 2**20 == b["useful_mib"]
    assert acc.reserved_slots(b["num_tokens"], b["block_size"]) == b["reserved_slots"]
    assert b["reserved_slots"] * per_tok / 2**20 == b["reserved_mib"]
    p = g["prefix_sharing_example"]
    assert acc.shareable_prefix_tokens(p["shared_tokens"], p["block_size"]) == p["shareable_tokens"]


def test_kv_sizes(golden):
    g = golden("kv_sizes.json")
    c0 = g["cases"][0]
    assert acc.kv_cache_bytes_kh(c0["layers"], c0["batch"], c0["seq_len"], c0["kv_dim"],
                                 c0["bytes_per_elem"]) == c0["exact_bytes"]
    for c in g["cases"][1:]:
        got = acc.kv_cache_bytes(c["layers"], c["batch"], c["seq_len"], c["kv_heads"],
                                 c["head_dim"], c["bytes_per_elem"])
        assert got == c["exact_bytes"], c
    q = g["cases"][-1]
    assert acc.kv_cache_bytes(q["layers"], 1, 1, q["kv_heads"], q["head_dim"], 2) == \
        q["exact_bytes_per_token"]
    r = g["gqa_ratio"]
    assert acc.kv_cache_bytes(32, 1, 100, r["num_kv_heads"], 128, 2) / \
        acc.kv_cache_bytes(32, 1, 100, r["num_q_heads"], 128, 2) == r["ratio"]


def test_attention_bytes():
    assert acc.attention_kv_bytes([1, 2], 8, 128, 2) == 3 * 8 * 128 * 2 * 2


@pytest.mark.parametrize("name", ["tiny", "qwen3_0_6b", "mistral_7b", "llama31_70b", "prefix_cow"])
def test_configs_build(name):
    w = wl.build(name, seed=0)
    S = w.num_seqs
    assert w.block_tables.shape[0] == S and w.context_lens.shape == (S,)
    for s in range(S):
        L = int(w.context_lens[s])
        n = acc.blocks_needed(L, w.block_size)
        row = w.block_tables[s, :n]
        assert np.all((row >= 0) & (row < w.num_blocks))
        assert w.positions[s] == L - 1
    if name == "tiny":
        assert list(w.context_lens) == [10, 7, 16, 3]
        assert w.num_blocks == 32 and w.dtype == "f32"
        assert sum(acc.blocks_needed(int(L), 4) for L in w.context_lens) == 10
    if name == "mistral_7b":
        assert (w.context_lens == 8192).sum() >= 64
        assert w.context_lens.min() >= 1024
    if name == "llama31_70b":
        assert list(w.context_lens) == [131072] * 4 and w.block_size == 32
    if name == "prefix_cow":
        assert S == 1024
        pre = w.block_tables[0, :128]
        assert all(np.array_equal(w.block_tables[s, :128], pre) for s in range(0, S, 97))
        # pairs: distinct destinations, sources are blocks that samples shared
        dst = w.copy_pairs[:, 1]
        assert len(set(dst.tolist())) == len(dst)
        partial = sum(1 for s in range(0, S, 4) if (int(w.context_lens[s]) - 1) % 16 != 0)
        assert len(w.copy_pairs) == 3 * partial
        assert 600 < len(w.copy_pairs) <= 768


def test_tiny_materialize_canaries():
    import torch
    w = wl.build("tiny", seed=0)
    t = wl.materialize(w, seed=0)
    hist = torch.from_numpy(w.history_mask)
    assert torch.isnan(t["k_cache"][~hist]).all()
    assert torch.isfinite(t["k_cache"][hist]).all()
    assert hist.sum().item() == sum(int(L) - 1 for L in w.context_lens)


def test_swap_out_and_in_all_or_nothing():
    gpu, host = BlockPool(16, seed=1), BlockPool(8, seed=2)
    a = SeqBlocks(gpu, 4)
    a.grow_to(13)                                  # 4 blocks
    b = a.fork()                                   # shares all 4
    c = SeqBlocks(gpu, 4)
    c.grow_to(20)                                  # 5 blocks
    old = list(a.mapping)
    pairs = swap_out(a, host)
    assert [p[0] for p in pairs] == old and a.pool is host
    assert a.mapping == [p[1] for p in pairs] and len(set(a.mapping)) == 4
    assert all(gpu.ref_counts[x] == 1 for x in old)     # b still holds them
    assert a.num_tokens == 13
    gpu.check_invariants([b, c])
    host.check_invariants([a])
    # not enough host room for c (5 blocks, 4 free): nothing changes
    before = (list(c.mapping), host.num_free, gpu.num_free)
    with pytest.raises(PoolExhausted):
        swap_out(c, host)
    assert (list(c.mapping), host.num_free, gpu.num_free) == before
    # back in: fresh GPU blocks, host blocks freed
    hosts = list(a.mapping)
    pairs = swap_in(a, gpu)
    assert [p[0] for p in pairs] == hosts and a.pool is gpu and host.num_free == 8
    assert not set(a.mapping) & set(b.mapping)      # a now owns private copies
    gpu.check_invariants([a, b, c])
    for t in (a, b, c):
        t.release_all()
    assert gpu.num_free == 16
