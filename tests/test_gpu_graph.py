"""CUDA-graph capture of the decode step (append + attention) and block sizes.

"19.2 KV Cache 系统化管理" §19.2.3 (closing remarks): production kernels are
fused and captured in CUDA graphs to remove launch overhead.  One graph holds
the fused slot mapping + KV append and the attention call (partition +
reduce); it is replayed for several decode steps whose inputs change in place
(new q, new K/V rows, positions and lengths one further).  Each replay must
equal eager launches bit for bit and the oracle within tolerance.

"企业官网建设流程全解析" §7.3: block sizes 8, 16, 32 and 64 are all served by
the tensor-core kernel; the output for one set of lengths and values must not
depend on the block size beyond fp32 reassociation.
"""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_115_gb300 import workloads as wl
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


def _lens_with_room(rng, n, K, steps):
    """Lengths whose last block has room for `steps` more tokens."""
    out = []
    while len(out) < n:
        L = int(rng.integers(1, 900))
        if 1 <= L % K <= K - steps:
            out.append(L)
    return out


@pytest.mark.parametrize("fmt", ["bf16", "fp8"])
@pytest.mark.parametrize("K", [8, 16])
def test_graph_replay_matches_eager_and_oracle(ops, fmt, K):
    steps = 3
    rng = np.random.default_rng(21 + K)
    lens0 = _lens_with_room(rng, 12, K, steps + 1)
    w = wl.build_decode("graph", lens0, 32, 8, 128, K, "bf16", seed=K)
    c = wl.materialize(w, seed=K)
    d = {k: v.to(DEV) for k, v in c.items()}
    S = w.num_seqs
    bound = w.max_context_len + steps
    if fmt == "fp8":
        gen = torch.Generator().manual_seed(K)
        codes = torch.randint(0, 256, d["k_cache"].shape, generator=gen, dtype=torch.int32)
        codes = torch.where((codes & 0x7F) == 0x7F, codes - 1, codes).to(torch.uint8)
        d["k_cache"], d["v_cache"] = codes.to(DEV), codes.flip(0).contiguous().to(DEV)
        qd = ops.kv_quant("fp8", 0.05, 0.07)
        ws_bytes = ops.attention_quant_workspace_bytes(S, 32, 8, 128, K, bound, torch.bfloat16, qd)
    else:
        qd = None
        ws_bytes = ops.attention_workspace_bytes(S, 32, 8, 128, K, bound, torch.bfloat16)
    out = torch.empty_like(d["q"])
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=DEV)
    slots = torch.empty(S, dtype=torch.int64, device=DEV)

    def step(t, o):
        if qd is None:
            ops.paged_kv_append(t["k_new"], t["v_new"], t["block_tables"], t["positions"],
                                t["k_cache"], t["v_cache"], slots)
            ops.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                                       t["context_lens"], w.scale, out=o,
                                       max_context_len=bound, workspace=ws)
        else:
            ops.paged_kv_append_quant(t["k_new"], t["v_new"], t["block_tables"], t["positions"],
                                      t["k_cache"], t["v_cache"], qd, slots)
            ops.paged_attention_decode_quant(t["q"], t["k_cache"], t["v_cache"],
                                             t["block_tables"], t["context_lens"], w.scale, qd,
                                             out=o, max_context_len=bound, workspace=ws)

    # eager warm-up on a throw-away copy (kernel attributes are set once)
    scratch = {k: v.clone() for k, v in d.items()}
    step(scratch, torch.empty_like(out))
    torch.cuda.synchronize()
    del scratch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            step(d, out)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    gen = torch.Generator().manual_seed(99)
    for it in range(steps):
        # the decode step `it`: every sequence appends its next token
        for name in ("q", "k_new", "v_new"):
            d[name].copy_(torch.randn(d[name].shape, generator=gen).to(torch.bfloat16))
        d["positions"].copy_(torch.tensor([L - 1 + it for L in lens0], dtype=torch.int32))
        d["context_lens"].copy_(torch.tensor([L + it for L in lens0], dtype=torch.int32))
        eager = {k: v.clone() for k, v in d.items()}
        eager_out = torch.empty_like(out)
        step(eager, eager_out)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager_out.view(torch.int16)), it
        assert torch.equal(d["k_cache"].view(torch.uint8), eager["k_cache"].view(torch.uint8))
        assert ops.get_device_error() == 0
        if qd is None:
            lens = [L + it for L in lens0]
            ref = oracle.paged_attention_decode(storage(d["q"]), storage(d["k_cache"]),
                                                storage(d["v_cache"]), w.block_tables, lens,
                                                w.scale, "bf16")
            check_attention(as_f64(out), ref, "bf16", f"replay {it}")


def test_block_sizes_give_the_same_attention(ops):
    """One set of lengths and token values, pools cut into 8-, 16-, 32- and
    64-token blocks: every output matches the oracle, and the outputs agree
    with one another within fp32 reassociation."""
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(1, 1500, size=10)] + [8, 9, 16, 64, 65]
    H_q, H_kv, D = 32, 8, 128
    gen = torch.Generator().manual_seed(5)
    q = torch.randn((len(lens), H_q, D), generator=gen).to(torch.bfloat16)
    rows_k = [torch.randn((L, H_kv, D), generator=gen).to(torch.bfloat16) for L in lens]
    rows_v = [torch.randn((L, H_kv, D), generator=gen).to(torch.bfloat16) for L in lens]
    outs = {}
    for K in (8, 16, 32, 64):
        w = wl.build_decode("bs", lens, H_q, H_kv, D, K, "bf16", seed=K)
        kc = torch.full((w.num_blocks, K, H_kv, D), float("nan"), dtype=torch.bfloat16)
        vc = kc.clone()
        for s, L in enumerate(lens):
            t = np.arange(L)
            slots = w.block_tables[s][t // K].astype(np.int64) * K + t % K
            kc.view(-1, H_kv, D)[torch.from_numpy(slots)] = rows_k[s]
            vc.view(-1, H_kv, D)[torch.from_numpy(slots)] = rows_v[s]
        out = ops.paged_attention_decode(q.to(DEV), kc.to(DEV), vc.to(DEV),
                                         torch.from_numpy(w.block_tables).to(DEV),
                                         torch.tensor(lens, dtype=torch.int32, device=DEV),
                                         w.scale, max_context_len=max(lens), kernel=1)
        assert ops.get_device_error() == 0
        ref = oracle.paged_attention_decode(storage(q), storage(kc), storage(vc), w.block_tables,
                                            lens, w.scale, "bf16")
        check_attention(as_f64(out), ref, "bf16", f"K={K}")
        outs[K] = as_f64(out)
    for K in (16, 32, 64):
        check_attention(outs[K], outs[8], "bf16", f"K={K} vs K=8")


@pytest.mark.parametrize("news", [[3, 3, 2, 3], [40, 200, 7, 130]])
def test_graph_replay_multi_query(ops, news):
    """A packed multi-query step (KV append of the new tokens + attention)
    captured once and replayed: speculative tokens take the stream-K decode
    kernel, longer chunks the tcgen05 kernel; replay equals eager launches."""
    import math
    from paged_kv_cache_115_gb300.blockmgr import BlockPool, SeqBlocks
    H_q, H_kv, D, K = 16, 8, 128, 16
    prefix = [500, 33, 1200, 64]
    lens = [a + b for a, b in zip(prefix, news)]
    pool = BlockPool(sum(-(-L // K) for L in lens) + 4, seed=7)
    rows = []
    for L in lens:
        sb = SeqBlocks(pool, K)
        sb.grow_to(L)
        rows.append(sb.mapping)
    bt = np.zeros((4, max(len(r) for r in rows)), np.int32)
    for i, r in enumerate(rows):
        bt[i, :len(r)] = r
    g = torch.Generator().manual_seed(1)
    nb = pool.num_blocks
    T = sum(news)
    t = dict(kc=torch.randn((nb, K, H_kv, D), generator=g).to(torch.bfloat16),
             vc=torch.randn((nb, K, H_kv, D), generator=g).to(torch.bfloat16),
             q=torch.randn((T, H_q, D), generator=g).to(torch.bfloat16),
             k=torch.randn((T, H_kv, D), generator=g).to(torch.bfloat16),
             v=torch.randn((T, H_kv, D), generator=g).to(torch.bfloat16))
    d = {k_: v_.to(DEV) for k_, v_ in t.items()}
    bt_d = torch.from_numpy(bt).to(DEV)
    cu = torch.tensor([0] + list(np.cumsum(news)), dtype=torch.int32, device=DEV)
    cl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    scale = 1.0 / math.sqrt(D)
    need = ops.prefill_workspace_bytes(4, T, max(news), max(lens), H_q, H_kv, D, K, scale,
                                       torch.bfloat16)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=DEV)
    out = torch.empty_like(d["q"])

    def step(x, o):
        ops.paged_kv_append_varlen(x["k"], x["v"], cu, cl, bt_d, x["kc"], x["vc"])
        ops.paged_attention_prefill(x["q"], x["kc"], x["vc"], bt_d, cu, cl, scale, max(news),
                                    max(lens), out=o, workspace=ws)

    scratch = {k_: v_.clone() for k_, v_ in d.items()}
    step(scratch, torch.empty_like(out))
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            step(d, out)
    torch.cuda.current_stream().wait_stream(side)
    gen = torch.Generator().manual_seed(2)
    for it in range(2):
        for name in ("q", "k", "v"):
            d[name].copy_(torch.randn(d[name].shape, generator=gen).to(torch.bfloat16))
        eager = {k_: v_.clone() for k_, v_ in d.items()}
        eager_out = torch.empty_like(out)
        step(eager, eager_out)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager_out.view(torch.int16)), it
        assert torch.equal(d["kc"].view(torch.int16), eager["kc"].view(torch.int16))
    assert ops.get_device_error() == 0
