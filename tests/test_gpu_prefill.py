"""GPU parity of multi-query paged attention (prefill of new tokens) and of the
packed KV append, against the oracle (oracle/prefill.py, oracle.slot_mapping,
oracle.kv_write).

Pools hold NaN in every slot without history before the step and block-table
rows carry garbage past their last used entry, so stray reads show up.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import prefill as P
from paged_kv_cache_115_gb300.blockmgr import BlockPool, SeqBlocks
from tests._helpers import as_f64, check_attention, storage

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def ops():
    from paged_kv_cache_115_gb300 import build
    build.build()
    from paged_kv_cache_115_gb300 import ops as o
    o.get_device_error()
    return o


def prefill_problem(prefix, news, H_q, H_kv, D, K, seed=0):
    """Sequence s has prefix[s] cached tokens and news[s] new ones."""
    rng = np.random.default_rng(seed)
    lens = [int(a) + int(b) for a, b in zip(prefix, news)]
    need = sum(-(-L // K) for L in lens)
    nb = max(4, math.ceil(need * 1.25) + 2)
    pool = BlockPool(nb, seed=int(rng.integers(2**31)))
    rows = []
    for L in lens:
        sb = SeqBlocks(pool, K)
        sb.grow_to(L)
        rows.append(list(sb.mapping))
    maxb = max(1, max(len(r) for r in rows)) + 2
    bt = rng.integers(-5, nb + 50, size=(len(lens), maxb)).astype(np.int32)
    for s, r in enumerate(rows):
        bt[s, :len(r)] = r
    g = torch.Generator().manual_seed(seed)
    kc = torch.randn((nb, K, H_kv, D), generator=g).to(torch.bfloat16)
    vc = torch.randn((nb, K, H_kv, D), generator=g).to(torch.bfloat16)
    hist = np.zeros(nb * K, bool)
    for s, r in enumerate(rows):
        for t in range(int(prefix[s])):
            hist[r[t // K] * K + t % K] = True
    m = torch.from_numpy(~hist.reshape(nb, K))
    kc[m] = float("nan")
    vc[m] = float("nan")
    cu = np.concatenate([[0], np.cumsum(news)]).astype(np.int32)
    T = int(cu[-1])
    q = torch.randn((T, H_q, D), generator=g).to(torch.bfloat16)
    k_new = torch.randn((T, H_kv, D), generator=g).to(torch.bfloat16)
    v_new = torch.randn((T, H_kv, D), generator=g).to(torch.bfloat16)
    return dict(lens=lens, bt=bt, cu=cu, kc=kc, vc=vc, q=q, k_new=k_new, v_new=v_new, K=K,
                scale=1.0 / math.sqrt(D), max_q=max(int(x) for x in news) if len(news) else 0)


def oracle_pools(pb):
    pos = P.query_positions(pb["cu"], pb["lens"])
    seq = np.repeat(np.arange(len(pb["lens"])), np.diff(pb["cu"]))
    slots = oracle.slot_mapping(pb["bt"][seq], pos, pb["K"])
    kc, vc = oracle.kv_write(storage(pb["kc"]), storage(pb["vc"]), storage(pb["k_new"]),
                             storage(pb["v_new"]), slots)
    return slots, kc, vc


def run_gpu(ops, pb, kernel=0, num_splits=0):
    d = {k: pb[k].to(DEV) for k in ("kc", "vc", "q", "k_new", "v_new")}
    bt = torch.from_numpy(pb["bt"]).to(DEV)
    cu = torch.from_numpy(pb["cu"]).to(DEV)
    lens = torch.tensor(pb["lens"], dtype=torch.int32, device=DEV)
    slots = torch.empty(d["q"].shape[0], dtype=torch.int64, device=DEV)
    ops.paged_kv_append_varlen(d["k_new"], d["v_new"], cu, lens, bt, d["kc"], d["vc"], slots)
    out = ops.paged_attention_prefill(d["q"], d["kc"], d["vc"], bt, cu, lens, pb["scale"],
                                      max_query_len=max(pb["max_q"], 1),
                                      max_context_len=max(max(pb["lens"]), 1), kernel=kernel,
                                      num_splits=num_splits)
    torch.cuda.synchronize()
    return slots, d, out


def full_check(ops, pb, what="", kernel=0, num_splits=0):
    slots, d, out = run_gpu(ops, pb, kernel, num_splits)
    assert ops.get_device_error() == 0
    eslots, ekc, evc = oracle_pools(pb)
    assert np.array_equal(slots.cpu().numpy(), eslots), what
    assert np.array_equal(storage(d["kc"]), ekc) and np.array_equal(storage(d["vc"]), evc), what
    ref = P.paged_attention_prefill(storage(pb["q"]), ekc, evc, pb["bt"], pb["cu"], pb["lens"],
                                    pb["scale"], "bf16")
    return check_attention(as_f64(out), ref, "bf16", what)


@pytest.mark.parametrize("kernel", [1, 2])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("K", [8, 16, 32])
def test_prefill_shapes(ops, kernel, D, G, K):
    H_kv = 2
    prefix = [0, 5, 100, 0, 33, 600, 17]
    news = [1, 3, 16, 70, 0, 9, 129]
    pb = prefill_problem(prefix, news, G * H_kv, H_kv, D, K, seed=D + G + K)
    full_check(ops, pb, f"kernel={kernel} D={D} G={G} K={K}", kernel)


@pytest.mark.parametrize("kernel", [1, 2])
def test_fresh_prompts_and_long_chunks(ops, kernel):
    # whole prompts (no prefix), one long enough for several query tiles and key tiles
    pb = prefill_problem([0, 0, 0, 0], [1, 15, 300, 513], 32, 8, 128, 16, seed=3)
    full_check(ops, pb, "fresh prompts", kernel)


@pytest.mark.parametrize("kernel", [1, 2])
def test_prefix_hit_suffix(ops, kernel):
    # a long cached prefix and a suffix of new tokens (prefix-cache hit)
    pb = prefill_problem([2048, 1000, 4096], [256, 64, 100], 32, 8, 128, 16, seed=4)
    full_check(ops, pb, "suffix prefill", kernel)


@pytest.mark.parametrize("kernel", [0, 1])
@pytest.mark.parametrize("n", [2, 4, 8])
def test_speculative_tokens_long_context(ops, n, kernel):
    # a few candidate tokens per sequence over long contexts (automatic: one
    # consumer warp; tcgen05: a 128-row tile mostly of padding rows)
    prefix = [3000, 1, 777, 5000, 64]
    pb = prefill_problem(prefix, [n] * len(prefix), 16, 4, 128, 16, seed=n)
    full_check(ops, pb, f"speculative n={n}", kernel)


def test_one_new_token_matches_decode(ops):
    rng = np.random.default_rng(6)
    prefix = [int(x) for x in rng.integers(0, 900, size=9)]
    pb = prefill_problem(prefix, [1] * 9, 32, 8, 128, 16, seed=6)
    slots, d, out = run_gpu(ops, pb)
    lens = torch.tensor(pb["lens"], dtype=torch.int32, device=DEV)
    dec = ops.paged_attention_decode(d["q"], d["kc"], d["vc"], torch.from_numpy(pb["bt"]).to(DEV),
                                     lens, pb["scale"], max_context_len=max(pb["lens"]))
    _, ekc, evc = oracle_pools(pb)
    ref = oracle.paged_attention_decode(storage(pb["q"]), ekc, evc, pb["bt"], pb["lens"],
                                        pb["scale"], "bf16")
    check_attention(as_f64(out), ref, "bf16", "prefill n=1")
    check_attention(as_f64(dec), ref, "bf16", "decode")
    assert ops.get_device_error() == 0


def test_chunked_prefill_matches_one_shot(ops):
    """A 700-token prompt in chunks of 256, 256, 188 (each chunk's K/V stored
    before its attention) gives the rows of the one-shot prefill."""
    H_q, H_kv, D, K = 16, 4, 128, 16
    pb = prefill_problem([0], [700], H_q, H_kv, D, K, seed=8)
    _, _, one = run_gpu(ops, pb)
    d = {k: pb[k].to(DEV) for k in ("kc", "vc", "q", "k_new", "v_new")}
    bt = torch.from_numpy(pb["bt"]).to(DEV)
    parts, done = [], 0
    for n in (256, 256, 188):
        cu = torch.tensor([0, n], dtype=torch.int32, device=DEV)
        lens = torch.tensor([done + n], dtype=torch.int32, device=DEV)
        sl = slice(done, done + n)
        ops.paged_kv_append_varlen(d["k_new"][sl].contiguous(), d["v_new"][sl].contiguous(), cu,
                                   lens, bt, d["kc"], d["vc"])
        parts.append(ops.paged_attention_prefill(d["q"][sl].contiguous(), d["kc"], d["vc"], bt, cu,
                                                 lens, pb["scale"], max_query_len=n,
                                                 max_context_len=700))
        done += n
    chunked = torch.cat(parts)
    _, ekc, evc = oracle_pools(pb)
    ref = P.paged_attention_prefill(storage(pb["q"]), ekc, evc, pb["bt"], pb["cu"], pb["lens"],
                                    pb["scale"], "bf16")
    check_attention(as_f64(chunked), ref, "bf16", "chunked")
    check_attention(as_f64(one), ref, "bf16", "one shot")
    assert ops.get_device_error() == 0


def test_empty_sequences_and_bad_counts(ops):
    # sequences with no new tokens produce no rows; the others are unaffected
    pb = prefill_problem([40, 0, 300, 7], [0, 0, 33, 5], 8, 2, 64, 16, seed=9)
    for kernel in (1, 2):
        full_check(ops, pb, "empty members", kernel)
    # more new tokens than the context holds: skipped and reported
    d = {k: pb[k].to(DEV) for k in ("kc", "vc", "q")}
    bt = torch.from_numpy(pb["bt"]).to(DEV)
    cu = torch.from_numpy(pb["cu"]).to(DEV)
    bad = torch.tensor([40, 0, 20, 12], dtype=torch.int32, device=DEV)     # 33 new > 20
    for kernel in (1, 2):
        ops.paged_attention_prefill(d["q"], d["kc"], d["vc"], bt, cu, bad, pb["scale"],
                                    max_query_len=33, max_context_len=333, kernel=kernel)
        assert ops.get_device_error() == 4


def test_unsupported_shapes_refused(ops):
    q = torch.zeros((4, 4, 96), dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros((8, 16, 2, 96), dtype=torch.bfloat16, device=DEV)
    cu = torch.tensor([0, 4], dtype=torch.int32, device=DEV)
    lens = torch.tensor([4], dtype=torch.int32, device=DEV)
    bt = torch.zeros((1, 2), dtype=torch.int32, device=DEV)
    with pytest.raises(ops.PagedKVError):
        ops.paged_attention_prefill(q, kc, kc, bt, cu, lens, 0.1, 4, 4)


@pytest.mark.parametrize("num_splits", [1, 2, 3, 7, 100])
def test_key_range_splits(ops, num_splits):
    """The mma.sync kernel with its keys cut into ranges merged by the split-K
    reduce: any number of ranges gives the oracle's rows (ranges past a tile's
    last key are empty and merge as zero weight)."""
    prefix = [3000, 1, 777, 5000, 64, 0]
    news = [4, 4, 4, 4, 4, 37]
    pb = prefill_problem(prefix, news, 16, 4, 128, 16, seed=31 + num_splits)
    full_check(ops, pb, f"splits={num_splits}", kernel=2, num_splits=num_splits)


def test_split_workspace_refusals(ops):
    pb = prefill_problem([3000, 10], [4, 4], 16, 4, 128, 16, seed=5)
    d = {k: pb[k].to(DEV) for k in ("kc", "vc", "q")}
    bt = torch.from_numpy(pb["bt"]).to(DEV)
    cu = torch.from_numpy(pb["cu"]).to(DEV)
    lens = torch.tensor(pb["lens"], dtype=torch.int32, device=DEV)
    need = ops.prefill_workspace_bytes(2, 8, 4, 3004, 16, 4, 128, 16, pb["scale"],
                                       torch.bfloat16, kernel=2, num_splits=6)
    assert need > 0
    small = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(ops.PagedKVError):
        ops.paged_attention_prefill(d["q"], d["kc"], d["vc"], bt, cu, lens, pb["scale"], 4, 3004,
                                    kernel=2, num_splits=6, workspace=small)
    # the tcgen05 kernel takes no split
    with pytest.raises(ops.PagedKVError):
        ops.paged_attention_prefill(d["q"], d["kc"], d["vc"], bt, cu, lens, pb["scale"], 4, 3004,
                                    kernel=1, num_splits=3)
    assert ops.prefill_workspace_bytes(2, 8, 4, 3004, 16, 4, 128, 16, pb["scale"],
                                       torch.bfloat16, kernel=1) == 0


@pytest.mark.parametrize("K", [8, 16, 32])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G,n", [(1, 8), (2, 4), (4, 2), (8, 1), (2, 3), (1, 5)])
def test_multi_token_decode_kernel(ops, K, D, G, n):
    """Several query tokens per sequence through the stream-K decode kernel
    (queries as the score columns of its tiles, a causal limit per column):
    short and long contexts, sequences with fewer or no new tokens."""
    H_kv = 2
    prefix = [0, 3, 40, 700, 16, 1500, 9, 250]
    news = [n, n, max(n - 1, 0), n, 0, n, 1, n]
    news[0] = n                         # a fresh prompt of n tokens
    pb = prefill_problem(prefix, news, G * H_kv, H_kv, D, K, seed=K + D + 3 * G + n)
    full_check(ops, pb, f"decode kernel K={K} D={D} G={G} n={n}", kernel=3)


def test_multi_token_decode_kernel_counts(ops):
    # more new tokens than the context holds: skipped and reported
    pb = prefill_problem([40, 10], [2, 2], 8, 2, 128, 16, seed=2)
    d = {k: pb[k].to(DEV) for k in ("kc", "vc", "q")}
    bt = torch.from_numpy(pb["bt"]).to(DEV)
    cu = torch.from_numpy(pb["cu"]).to(DEV)
    bad = torch.tensor([42, 1], dtype=torch.int32, device=DEV)
    ops.paged_attention_prefill(d["q"], d["kc"], d["vc"], bt, cu, bad, pb["scale"], 2, 42,
                                kernel=3)
    assert ops.get_device_error() == 4
    # more than 8 rows per KV head is refused for this kernel
    with pytest.raises(ops.PagedKVError):
        ops.paged_attention_prefill(d["q"], d["kc"], d["vc"], bt, cu, bad, pb["scale"], 5, 42,
                                    kernel=3)


@pytest.mark.parametrize("D,K", [(128, 16), (64, 8), (128, 32)])
@pytest.mark.parametrize("n", [3, 4, 16])
def test_few_rows_many_pairs_automatic(ops, n, D, K):
    # 9 .. 64 query rows per KV head with at least as many (sequence, KV head)
    # pairs as SMs: the automatic plan takes one tcgen05 tile per CTA (mostly
    # padding rows); the result must match the oracle and the mma.sync kernel
    S, H_kv, G = 40, 4, 4
    rng = np.random.default_rng(60 + n)
    prefix = [int(x) for x in rng.integers(0, 300, size=S)]
    pb = prefill_problem(prefix, [n] * S, G * H_kv, H_kv, D, K, seed=70 + n + D + K)
    full_check(ops, pb, f"automatic n={n} D={D} K={K}")
    _, _, out_tc = run_gpu(ops, pb, kernel=1)
    _, _, out_ms = run_gpu(ops, pb, kernel=2)
    check_attention(as_f64(out_tc), as_f64(out_ms), "bf16", f"tcgen05 vs mma.sync n={n} D={D} K={K}")
