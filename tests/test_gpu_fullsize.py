"""Full-size parity of the rows past the decode step, in the launch plans
bench.py times: every output element against the oracle.

* FP8 / INT8 pools at the Mistral-7B-shaped decode size (quantizing append +
  attention, automatic kernel choice);
* the multi-query workloads suffix_prefill (two-tile tcgen05 kernel),
  chunked_prefill (tcgen05 kernel, one query tile per CTA) and speculative_decode
  (stream-K decode kernel with several query rows);
* the block swap workload (every other sequence out to pinned host memory and
  back into a permutation of the blocks).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import prefill as OP
from oracle import quant as Q
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


@pytest.mark.parametrize("fmt", ["fp8", "int8", "k16v8"])
def test_quant_full_size(ops, fmt):
    w = wl.build("mistral_7b")
    rng = np.random.default_rng(17)
    nb, K, H, D = w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim
    shape = (nb, K, H, D)
    if fmt in ("fp8", "k16v8"):
        kc = rng.integers(0, 256, size=shape, dtype=np.uint8)
        vc = rng.integers(0, 256, size=shape, dtype=np.uint8)
        kc[(kc & 0x7F) == 0x7F] -= 1                    # no NaN codes
        vc[(vc & 0x7F) == 0x7F] -= 1
        kts = vts = None
        if fmt == "k16v8":    # K: bf16 patterns of N(0, 1) draws
            kc = (rng.standard_normal(shape, dtype=np.float32).view(np.uint32) >> 16).astype(
                np.uint16)
    else:
        kc = rng.integers(-127, 128, size=shape, dtype=np.int8)
        vc = rng.integers(-127, 128, size=shape, dtype=np.int8)
        kts = (rng.random(nb * K, dtype=np.float32) * 0.02 + 0.001).astype(np.float32)
        vts = (rng.random(nb * K, dtype=np.float32) * 0.02 + 0.001).astype(np.float32)
    g = torch.Generator().manual_seed(17)
    q = torch.randn((w.num_seqs, w.num_q_heads, D), generator=g).to(torch.bfloat16)
    k_new = torch.randn((w.num_seqs, H, D), generator=g).to(torch.bfloat16)
    v_new = torch.randn((w.num_seqs, H, D), generator=g).to(torch.bfloat16)
    dk, dv = torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV)
    if fmt == "fp8":
        qd = ops.kv_quant("fp8", 0.05, 0.07)
    elif fmt == "k16v8":
        dk = torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16).to(DEV)
        qd = ops.kv_quant("k16v8", v_scale=0.07)
    else:
        dkt, dvt = torch.from_numpy(kts.copy()).to(DEV), torch.from_numpy(vts.copy()).to(DEV)
        qd = ops.kv_quant("int8", k_token_scales=dkt, v_token_scales=dvt)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    ops.paged_kv_append_quant(k_new.to(DEV), v_new.to(DEV), bt,
                              torch.from_numpy(w.positions).to(DEV), dk, dv, qd)
    out = ops.paged_attention_decode_quant(q.to(DEV), dk, dv, bt,
                                           torch.from_numpy(w.context_lens).to(DEV), w.scale, qd,
                                           max_context_len=w.max_context_len)
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    # the appended rows, bit-exact, through the oracle's quantized write
    slots = oracle.slot_mapping(w.block_tables, w.positions, K)
    kf, vf = k_new.float().numpy(), v_new.float().numpy()
    idx = np.arange(w.num_seqs)
    if fmt == "fp8":
        sk = np.zeros((w.num_seqs, 1, H, D), np.uint8)
        okc, ovc = Q.kv_write_fp8(sk, sk.copy(), kf, vf, idx, 0.05, 0.07)
    elif fmt == "k16v8":
        okc, ovc = Q.kv_write_k16v8(np.zeros((w.num_seqs, 1, H, D), np.uint16),
                                    np.zeros((w.num_seqs, 1, H, D), np.uint8), kf, vf, idx, 0.07)
    else:
        sk = np.zeros((w.num_seqs, 1, H, D), np.int8)
        okc, ovc, okts, ovts = Q.kv_write_int8(sk, sk.copy(), np.zeros(w.num_seqs, np.float32),
                                               np.zeros(w.num_seqs, np.float32), kf, vf, idx)
    got_k = storage(dk.view(-1, H, D)[torch.from_numpy(slots).to(DEV)])
    got_v = dv.view(-1, H, D)[torch.from_numpy(slots).to(DEV)].cpu().numpy()
    assert np.array_equal(got_k, okc[:, 0]) and np.array_equal(got_v, ovc[:, 0])
    # the pool as the oracle's own write leaves it (the rows just checked)
    kc_now, vc_now = kc.copy(), vc.copy()
    kc_now.reshape(-1, H, D)[slots] = okc[:, 0]
    vc_now.reshape(-1, H, D)[slots] = ovc[:, 0]
    if fmt == "int8":
        assert np.array_equal(dkt.cpu().numpy()[slots], okts)
        assert np.array_equal(dvt.cpu().numpy()[slots], ovts)
        kts_now, vts_now = kts.copy(), vts.copy()
        kts_now[slots], vts_now[slots] = okts, ovts
    outf = as_f64(out)
    assert np.all(np.isfinite(outf))
    # every output row against the oracle over the pool as it now stands
    qn = storage(q)
    if fmt == "fp8":
        ref = Q.paged_attention_decode_quant(qn, kc_now, vc_now, w.block_tables, w.context_lens,
                                             w.scale, "bf16", "fp8", k_scale=0.05, v_scale=0.07)
    elif fmt == "k16v8":
        ref = Q.paged_attention_decode_quant(qn, kc_now, vc_now, w.block_tables, w.context_lens,
                                             w.scale, "bf16", "k16v8", v_scale=0.07)
    else:
        ref = Q.paged_attention_decode_quant(qn, kc_now, vc_now, w.block_tables, w.context_lens,
                                             w.scale, "bf16", "int8", k_tok_scales=kts_now,
                                             v_tok_scales=vts_now)
    check_attention(outf, ref, "bf16", f"{fmt} full size")


@pytest.mark.parametrize("name", ["suffix_prefill", "chunked_prefill", "speculative_decode"])
def test_prefill_full_size(ops, name):
    w = wl.build_prefill(name)
    K, H, D, H_q = w.block_size, w.num_kv_heads, w.head_dim, w.num_q_heads
    G = H_q // H
    g = torch.Generator().manual_seed(23)
    kc = torch.randn((w.num_blocks, K, H, D), generator=g).to(torch.bfloat16)
    vc = torch.randn((w.num_blocks, K, H, D), generator=g).to(torch.bfloat16)
    T = w.num_tokens
    q = torch.randn((T, H_q, D), generator=g).to(torch.bfloat16)
    k_new = torch.randn((T, H, D), generator=g).to(torch.bfloat16)
    v_new = torch.randn((T, H, D), generator=g).to(torch.bfloat16)
    dk, dv = kc.to(DEV), vc.to(DEV)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    cu = torch.from_numpy(w.cu_seqlens).to(DEV)
    lens = torch.from_numpy(w.context_lens).to(DEV)
    slots = torch.empty(T, dtype=torch.int64, device=DEV)
    ops.paged_kv_append_varlen(k_new.to(DEV), v_new.to(DEV), cu, lens, bt, dk, dv, slots)
    out = ops.paged_attention_prefill(q.to(DEV), dk, dv, bt, cu, lens, w.scale,
                                      int(w.news.max()), int(w.context_lens.max()))
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    pos = OP.query_positions(w.cu_seqlens, w.context_lens)
    seq = np.repeat(np.arange(w.num_seqs), w.news)
    oslots = oracle.slot_mapping(w.block_tables[seq], pos, K)
    assert np.array_equal(slots.cpu().numpy(), oslots)
    okc, ovc = oracle.kv_write(storage(kc), storage(vc), storage(k_new), storage(v_new), oslots)
    assert np.array_equal(storage(dk), okc) and np.array_equal(storage(dv), ovc)
    outf = as_f64(out)
    assert np.all(np.isfinite(outf))
    # every output row: per (sequence, KV head) the rows are gathered once and
    # each query row (new token i, head of the group) sees keys 0 .. its position
    qn = oracle.decode(storage(q), "bf16")
    ref = np.zeros_like(outf)
    for s_ in range(w.num_seqs):
        L = int(w.context_lens[s_])
        t0, t1 = int(w.cu_seqlens[s_]), int(w.cu_seqlens[s_ + 1])
        for j in range(H):
            Kj = oracle.gather_kv(okc, w.block_tables[s_], L, j, K, "bf16")
            Vj = oracle.gather_kv(ovc, w.block_tables[s_], L, j, K, "bf16")
            rows = qn[t0:t1, j * G:(j + 1) * G].reshape(-1, D)
            lim = np.repeat(pos[t0:t1], G)
            ref[t0:t1, j * G:(j + 1) * G] = oracle.attention_rows(
                rows, Kj, Vj, lim, w.scale).reshape(t1 - t0, G, D)
    check_attention(outf, ref, "bf16", name)


def test_swap_full_size(ops):
    w = wl.build("qwen3_0_6b")
    out_np, in_np = wl.swap_plan(w, 0)
    n = len(out_np)
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    g = torch.Generator().manual_seed(29)
    kc = torch.randn(shape, generator=g).to(torch.bfloat16)
    vc = torch.randn(shape, generator=g).to(torch.bfloat16)
    dk, dv = kc.to(DEV), vc.to(DEV)
    hk = torch.zeros((n,) + shape[1:], dtype=torch.bfloat16).pin_memory()
    hv = torch.zeros((n,) + shape[1:], dtype=torch.bfloat16).pin_memory()
    ops.kv_block_swap(dk, dv, hk, hv, torch.from_numpy(out_np).to(DEV))
    torch.cuda.synchronize()
    ek, ev = oracle.kv_block_swap(storage(kc), storage(vc), storage(torch.zeros_like(hk)),
                                  storage(torch.zeros_like(hv)), out_np)
    assert np.array_equal(storage(hk), ek) and np.array_equal(storage(hv), ev)
    # the GPU blocks are reused meanwhile; swap back into a permutation of them
    dk.fill_(float("nan"))
    dv.fill_(float("nan"))
    before_k, before_v = storage(dk), storage(dv)
    ops.kv_block_swap(hk, hv, dk, dv, torch.from_numpy(in_np).to(DEV))
    torch.cuda.synchronize()
    ek2, ev2 = oracle.kv_block_swap(ek, ev, before_k, before_v, in_np)
    assert np.array_equal(storage(dk), ek2) and np.array_equal(storage(dv), ev2)
    assert ops.get_device_error() == 0
