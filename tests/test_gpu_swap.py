"""GPU parity of the block swap between GPU pools and pinned host pools.

Byte movement must be bit-exact against the oracle's ``kv_block_swap``; a
request swapped out and back into other GPU blocks must give bit-identical
attention output (the kernels' work split depends only on lengths).
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_115_gb300.blockmgr import BlockPool, SeqBlocks, swap_in, swap_out
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


def _pool(shape, dtype, gen, fill=None):
    if dtype in (torch.uint8, torch.int8):
        t = torch.randint(-128 if dtype == torch.int8 else 0, 128 if dtype == torch.int8 else 256,
                          shape, generator=gen, dtype=torch.int32).to(dtype)
    else:
        t = torch.randn(shape, generator=gen).to(dtype)
    if fill is not None:
        t.fill_(fill)
    return t


def _pairs(rng, n, src_nb, dst_nb):
    src = rng.choice(src_nb, size=n, replace=False)
    dst = rng.choice(dst_nb, size=n, replace=False)
    return np.stack([src, dst], 1).astype(np.int64)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32, torch.uint8])
@pytest.mark.parametrize("pairs_on", ["cuda", "pinned"])
def test_swap_out_then_in_bit_exact(ops, dtype, pairs_on):
    g = torch.Generator().manual_seed(5)
    rng = np.random.default_rng(5)
    K, H, D = 16, 8, 128
    gk = _pool((40, K, H, D), dtype, g)
    gv = _pool((40, K, H, D), dtype, g)
    hk = _pool((24, K, H, D), dtype, g, fill=7).pin_memory()      # canary contents
    hv = _pool((24, K, H, D), dtype, g, fill=3).pin_memory()
    out_pairs = _pairs(rng, 17, 40, 24)
    dgk, dgv = gk.to(DEV), gv.to(DEV)

    def put(p):
        t = torch.from_numpy(p)
        return t.to(DEV) if pairs_on == "cuda" else t.pin_memory()

    p1 = put(out_pairs)
    ops.kv_block_swap(dgk, dgv, hk, hv, p1)
    torch.cuda.synchronize()
    ek, ev = oracle.kv_block_swap(storage(gk), storage(gv), storage(hk.clone().fill_(7)),
                                  storage(hv.clone().fill_(3)), out_pairs)
    assert np.array_equal(storage(hk), ek) and np.array_equal(storage(hv), ev)
    # back into other GPU blocks (device pool pre-filled with different data)
    in_pairs = np.stack([out_pairs[:, 1], rng.choice(40, size=17, replace=False)], 1)
    before_k, before_v = storage(dgk), storage(dgv)
    p2 = put(in_pairs)
    ops.kv_block_swap(hk, hv, dgk, dgv, p2)
    torch.cuda.synchronize()
    ek2, ev2 = oracle.kv_block_swap(ek, ev, before_k, before_v, in_pairs)
    assert np.array_equal(storage(dgk), ek2) and np.array_equal(storage(dgv), ev2)
    assert ops.get_device_error() == 0


def test_swap_device_to_device_and_scale_arrays(ops):
    g = torch.Generator().manual_seed(6)
    rng = np.random.default_rng(6)
    a = _pool((30, 32, 2, 64), torch.bfloat16, g).to(DEV)
    b = _pool((30, 32, 2, 64), torch.bfloat16, g).to(DEV)
    c = _pool((11, 32, 2, 64), torch.bfloat16, g).to(DEV)
    d = _pool((11, 32, 2, 64), torch.bfloat16, g).to(DEV)
    pairs = _pairs(rng, 9, 30, 11)
    ek, ev = oracle.kv_block_swap(storage(a), storage(b), storage(c), storage(d), pairs)
    ops.kv_block_swap(a, b, c, d, torch.from_numpy(pairs).to(DEV))
    assert np.array_equal(storage(c), ek) and np.array_equal(storage(d), ev)
    # INT8 slot scales: one float32 per slot, a block is K of them (64 bytes)
    sk = torch.rand((50, 16), generator=g).to(DEV)
    hs = torch.full((20, 16), -1.0).pin_memory()
    pairs = _pairs(rng, 13, 50, 20)
    ops.kv_block_swap(sk, None, hs, None, torch.from_numpy(pairs).to(DEV))
    torch.cuda.synchronize()
    want = storage(torch.full((20, 16), -1.0))
    want, _ = oracle.kv_block_swap(storage(sk), storage(sk), want, want.copy(), pairs)
    assert np.array_equal(storage(hs), want)
    # odd block sizes take the narrow vector paths
    e = _pool((7, 3, 1, 5), torch.bfloat16, g).to(DEV)     # 30-byte blocks
    f = _pool((5, 3, 1, 5), torch.bfloat16, g).pin_memory()
    pairs = _pairs(rng, 4, 7, 5)
    want, _ = oracle.kv_block_swap(storage(e), storage(e), storage(f), storage(f), pairs)
    ops.kv_block_swap(e, None, f, None, torch.from_numpy(pairs).to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(storage(f), want)
    assert ops.get_device_error() == 0


def test_swap_refusals_and_bad_pairs(ops):
    g = torch.Generator().manual_seed(7)
    a = _pool((4, 16, 2, 64), torch.bfloat16, g).to(DEV)
    b = _pool((4, 16, 2, 64), torch.bfloat16, g).to(DEV)
    pageable = torch.zeros((4, 16, 2, 64), dtype=torch.bfloat16)
    pairs = torch.tensor([[0, 1]], dtype=torch.int64, device=DEV)
    with pytest.raises(ValueError):
        ops.kv_block_swap(a, None, pageable, None, pairs)
    # the library itself refuses pageable host memory (no launch)
    blk = 16 * 2 * 64 * 2
    st = ops._block_swap(ctypes.c_void_p(a.data_ptr()), None, 4,
                         ctypes.c_void_p(pageable.data_ptr()), None, 4, blk,
                         ctypes.c_void_p(pairs.data_ptr()), 1,
                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == ops.PKV_ERR_INVALID_ARGUMENT
    assert b"pageable" in ops._last_msg()
    # out-of-range ids: pair skipped, device error 3, others still move
    before = storage(b)
    bad = torch.tensor([[0, 4], [1, 2], [-1, 0]], dtype=torch.int64, device=DEV)
    ops.kv_block_swap(a, None, b, None, bad)
    assert ops.get_device_error() == 3
    want = before.copy()
    want[2] = storage(a)[1]
    assert np.array_equal(storage(b), want)


def test_preempt_swap_resume_attention_bit_identical(ops):
    """Three requests are preempted by swap, their GPU blocks are handed to a
    newcomer and overwritten, then the requests resume in fresh blocks: the
    attention output is bit-identical to the output before preemption and
    matches the oracle."""
    K, H_q, H_kv, D = 16, 16, 8, 128
    lens = [700, 33, 1, 517, 260, 96, 1024, 15]
    rng = np.random.default_rng(8)
    gpu = BlockPool(200, seed=1)
    host = BlockPool(160, seed=2)
    seqs = []
    for L in lens:
        s = SeqBlocks(gpu, K)
        s.grow_to(L)
        seqs.append(s)
    g = torch.Generator().manual_seed(8)
    kc = torch.randn((200, K, H_kv, D), generator=g).to(torch.bfloat16).to(DEV)
    vc = torch.randn((200, K, H_kv, D), generator=g).to(torch.bfloat16).to(DEV)
    q = torch.randn((len(lens), H_q, D), generator=g).to(torch.bfloat16).to(DEV)
    maxb = max(len(s.mapping) for s in seqs)

    def tables():
        t = np.full((len(lens), maxb), -5, np.int32)
        for i, s in enumerate(seqs):
            t[i, :len(s.mapping)] = s.mapping
        return torch.from_numpy(t).to(DEV)

    cl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    scale = D ** -0.5
    out1 = ops.paged_attention_decode(q, kc, vc, tables(), cl, scale, max_context_len=max(lens))
    bt1 = tables().cpu().numpy()
    ref = oracle.paged_attention_decode(storage(q), storage(kc), storage(vc), bt1, lens, scale,
                                        "bf16")
    check_attention(as_f64(out1), ref, "bf16", "before preemption")

    hk = torch.zeros((160, K, H_kv, D), dtype=torch.bfloat16).pin_memory()
    hv = torch.zeros((160, K, H_kv, D), dtype=torch.bfloat16).pin_memory()
    victims = [0, 3, 6]
    for i in victims:
        p = torch.tensor(swap_out(seqs[i], host), dtype=torch.int64).to(DEV)
        ops.kv_block_swap(kc, vc, hk, hv, p)
    gpu.check_invariants([s for i, s in enumerate(seqs) if i not in victims])
    # a newcomer takes freed blocks and writes over them
    newcomer = SeqBlocks(gpu, K)
    newcomer.grow_to(K * min(gpu.num_free, 60))
    taken = torch.tensor(newcomer.mapping, dtype=torch.int64, device=DEV)
    kc[taken] = float("nan")
    vc[taken] = float("nan")
    newcomer.release_all()
    for i in victims:
        p = torch.tensor(swap_in(seqs[i], gpu), dtype=torch.int64).to(DEV)
        ops.kv_block_swap(hk, hv, kc, vc, p)
    gpu.check_invariants(seqs)
    bt2 = tables()
    assert not np.array_equal(bt2.cpu().numpy(), bt1)
    out2 = ops.paged_attention_decode(q, kc, vc, bt2, cl, scale, max_context_len=max(lens))
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert ops.get_device_error() == 0
