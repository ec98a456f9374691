"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Integer and copy work must be bit-exact; bf16 attention within
|d| <= 2e-3 + 1e-2 |ref| and fp32 attention within 1e-5 of the fp64 oracle.
Pools are filled with NaN wherever no history token lives and block-table
rows carry garbage past their last used entry, so any stray read shows up.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_115_gb300 import workloads as wl
from tests._helpers import as_f64, check_attention, dtype_name, storage

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def ops():
    from paged_kv_cache_115_gb300 import build
    build.build()
    from paged_kv_cache_115_gb300 import ops as o
    o.get_device_error()   # start clean
    return o


def to_dev(t):
    return {k: v.to(DEV) for k, v in t.items()}


def gpu_step(ops, w, d, **attn_kw):
    if len(w.copy_pairs):
        ops.kv_block_copy(d["k_cache"], d["v_cache"], d["copy_pairs"])
    slots = ops.slot_mapping(d["block_tables"], d["positions"], w.block_size, w.num_blocks)
    ops.paged_kv_write(d["k_new"], d["v_new"], slots, d["k_cache"], d["v_cache"])
    out = ops.paged_attention_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                     d["context_lens"], w.scale,
                                     max_context_len=w.max_context_len, **attn_kw)
    return slots, out


def oracle_step_pool(w, c):
    """The oracle's own pools after the step's copy and write."""
    kc, vc = storage(c["k_cache"]), storage(c["v_cache"])
    if len(w.copy_pairs):
        kc, vc = oracle.kv_block_copy(kc, vc, w.copy_pairs)
    slots = oracle.slot_mapping(w.block_tables, w.positions, w.block_size)
    kc, vc = oracle.kv_write(kc, vc, storage(c["k_new"]), storage(c["v_new"]), slots)
    return slots, kc, vc


def full_check(ops, w, seed=0, **attn_kw):
    c = wl.materialize(w, seed=seed)
    d = to_dev(c)
    slots, out = gpu_step(ops, w, d, **attn_kw)
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    oslots, okc, ovc = oracle_step_pool(w, c)
    assert np.array_equal(slots.cpu().numpy(), oslots)
    assert np.array_equal(storage(d["k_cache"]), okc)
    assert np.array_equal(storage(d["v_cache"]), ovc)
    dt = dtype_name(c["q"])
    ref = oracle.paged_attention_decode(storage(c["q"]), okc, ovc, w.block_tables,
                                        w.context_lens, w.scale, dt)
    return check_attention(as_f64(out), ref, dt, w.name)


# ---------------------------------------------------------------------------
# slot mapping, KV write, block copy: bit exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", wl.CONFIG_NAMES)
def test_slot_mapping_configs(ops, name):
    w = wl.build(name)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    pos = torch.from_numpy(w.positions).to(DEV)
    got = ops.slot_mapping(bt, pos, w.block_size, w.num_blocks).cpu().numpy()
    assert np.array_equal(got, oracle.slot_mapping(w.block_tables, w.positions, w.block_size))
    assert ops.get_device_error() == 0


@pytest.mark.parametrize("K", [1, 3, 4, 16, 32, 48])
def test_slot_mapping_every_position(ops, K):
    rng = np.random.default_rng(K)
    S, maxB, nb = 9, 7, 80
    bt = rng.permutation(nb)[: S * maxB].reshape(S, maxB).astype(np.int32)
    pos = rng.integers(-2, maxB * K, size=S).astype(np.int32)
    pos[0] = maxB * K - 1
    got = ops.slot_mapping(torch.from_numpy(bt).to(DEV), torch.from_numpy(pos).to(DEV), K, nb)
    assert np.array_equal(got.cpu().numpy(), oracle.slot_mapping(bt, pos, K))
    assert ops.get_device_error() == 0


def test_slot_mapping_device_checks(ops):
    bt = torch.tensor([[3, 99], [1, 2]], dtype=torch.int32, device=DEV)
    got = ops.slot_mapping(bt, torch.tensor([5, 1], dtype=torch.int32, device=DEV), 4, 10)
    assert got.cpu().tolist() == [-1, 5]
    assert ops.get_device_error() == 1          # block id 99 out of range
    got = ops.slot_mapping(bt, torch.tensor([8, 0], dtype=torch.int32, device=DEV), 4, 10)
    assert got.cpu().tolist() == [-1, 4]
    assert ops.get_device_error() == 5          # position beyond the row
    assert ops.get_device_error() == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("H,D", [(8, 128), (2, 64), (3, 5)])
def test_kv_write_bit_exact(ops, dtype, H, D):
    g = torch.Generator().manual_seed(H * 100 + D)
    nb, K, T = 13, 4, 21
    kc = torch.full((nb, K, H, D), float("nan"), dtype=dtype)
    vc = torch.randn((nb, K, H, D), generator=g).to(dtype)
    k = torch.randn((T, H, D), generator=g).to(dtype)
    v = torch.randn((T, H, D), generator=g).to(dtype)
    slots = torch.randperm(nb * K, generator=g)[:T].to(torch.int64)
    slots[[2, 9]] = -1
    dkc, dvc = kc.to(DEV), vc.to(DEV)
    ops.paged_kv_write(k.to(DEV), v.to(DEV), slots.to(DEV), dkc, dvc)
    ek, ev = oracle.kv_write(storage(kc), storage(vc), storage(k), storage(v), slots.numpy())
    assert np.array_equal(storage(dkc), ek) and np.array_equal(storage(dvc), ev)
    assert ops.get_device_error() == 0


def test_kv_write_bad_slot_is_skipped(ops):
    kc = torch.zeros((4, 2, 1, 8), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    k = torch.ones((2, 1, 8), dtype=torch.bfloat16, device=DEV)
    ops.paged_kv_write(k, k, torch.tensor([8, 3], device=DEV), kc, vc)
    assert ops.get_device_error() == 2
    assert kc.view(-1, 1, 8)[3].eq(1).all() and kc.sum().item() == 8


def test_block_copy_prefix_cow(ops):
    w = wl.build("prefix_cow")
    c = wl.materialize(w)
    d = to_dev(c)
    ops.kv_block_copy(d["k_cache"], d["v_cache"], d["copy_pairs"])
    ek, ev = oracle.kv_block_copy(storage(c["k_cache"]), storage(c["v_cache"]), w.copy_pairs)
    assert np.array_equal(storage(d["k_cache"]), ek)
    assert np.array_equal(storage(d["v_cache"]), ev)
    assert ops.get_device_error() == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_block_copy_small_and_bad_pair(ops, dtype):
    g = torch.Generator().manual_seed(3)
    kc = torch.randn((9, 3, 2, 5), generator=g).to(dtype)
    vc = torch.randn((9, 3, 2, 5), generator=g).to(dtype)
    pairs = torch.tensor([[0, 4], [1, 5], [8, 2]], dtype=torch.int64)
    dk, dv = kc.to(DEV), vc.to(DEV)
    ops.kv_block_copy(dk, dv, pairs.to(DEV))
    ek, ev = oracle.kv_block_copy(storage(kc), storage(vc), pairs.numpy())
    assert np.array_equal(storage(dk), ek) and np.array_equal(storage(dv), ev)
    assert ops.get_device_error() == 0
    ops.kv_block_copy(dk, dv, torch.tensor([[0, 9]], dtype=torch.int64, device=DEV))
    assert ops.get_device_error() == 3
    assert np.array_equal(storage(dk), ek)


# ---------------------------------------------------------------------------
# attention: whole step at oracle-sized shapes
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("num_splits", [0, 1, 2, 3, 512])
def test_tiny_step(ops, num_splits):
    w = wl.build("tiny")
    full_check(ops, w, num_splits=num_splits)


LENS_RAGGED = [1, 15, 16, 17, 31, 33, 100, 257, 600]


@pytest.mark.parametrize("K", [8, 16, 32, 64])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_tc_kernel_shapes(ops, K, G, D):
    H_kv = 2 if D == 64 else 8 // max(1, G // 2)
    w = wl.build_decode("tc", LENS_RAGGED, G * H_kv, H_kv, D, K, "bf16", seed=K + G + D)
    full_check(ops, w, kernel=1)


@pytest.mark.parametrize("num_splits", [1, 2, 5, 13, 40, 400])
def test_tc_kernel_split_counts(ops, num_splits):
    w = wl.build_decode("tc_split", [1, 700, 0, 33, 1500, 16, 2, 300], 32, 8, 128, 16, "bf16",
                        seed=num_splits)
    full_check(ops, w, kernel=1, num_splits=num_splits)


@pytest.mark.parametrize("K", [16, 8])
@pytest.mark.parametrize("H_kv", [1, 2, 4, 8, 16])
def test_tc_kernel_head_groups(ops, H_kv, K):
    w = wl.build_decode("tc_heads", [70, 300, 5], 2 * H_kv, H_kv, 128, K, "bf16", seed=H_kv + K)
    full_check(ops, w, kernel=1)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("K", [1, 3, 4, 16])
@pytest.mark.parametrize("G", [1, 3, 8, 16])
@pytest.mark.parametrize("D", [32, 128, 256])
def test_simt_kernel_shapes(ops, dtype, K, G, D):
    w = wl.build_decode("simt", [1, 5, 17, 64, 130], 2 * G, 2, D, K, dtype, seed=K * G + D)
    full_check(ops, w, kernel=2, num_splits=48)


@pytest.mark.parametrize("num_splits", [0, 1, 7, 1024])
def test_simt_kernel_split_counts(ops, num_splits):
    w = wl.build_decode("simt_split", [0, 3, 1100, 64, 2049], 8, 2, 64, 8, "f32", seed=5)
    full_check(ops, w, kernel=2, num_splits=num_splits)


def test_empty_and_single_token_sequences(ops):
    w = wl.build_decode("edge", [0, 1, 0, 2, 1], 8, 2, 128, 16, "bf16", seed=1)
    for kernel in (1, 2):
        full_check(ops, w, kernel=kernel)


def test_many_sequences_batched(ops):
    rng = np.random.default_rng(9)
    lens = rng.integers(0, 40, size=2500)
    w = wl.build_decode("many", lens, 16, 8, 64, 16, "bf16", seed=2)
    full_check(ops, w, kernel=1)


def test_bad_block_id_reported(ops):
    w = wl.build_decode("bad", [40, 40], 8, 8, 128, 16, "bf16", seed=4)
    c = wl.materialize(w, canary=False)
    d = to_dev(c)
    d["block_tables"][1, 1] = w.num_blocks + 7
    out = ops.paged_attention_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                     d["context_lens"], w.scale, max_context_len=40, kernel=1)
    assert ops.get_device_error() == 1
    assert torch.isfinite(out.float()).all()


def test_length_beyond_bound_clamped_and_reported(ops):
    w = wl.build_decode("clamp", [48, 20], 8, 8, 128, 16, "bf16", seed=6)
    c = wl.materialize(w, canary=False)
    d = to_dev(c)
    for kernel in (1, 2):
        out = ops.paged_attention_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                         d["context_lens"], w.scale, max_context_len=32,
                                         kernel=kernel)
        assert ops.get_device_error() == 4
        lens32 = np.minimum(w.context_lens, 32)
        ref = oracle.paged_attention_decode(storage(c["q"]), storage(c["k_cache"]),
                                            storage(c["v_cache"]), w.block_tables, lens32,
                                            w.scale, "bf16")
        check_attention(as_f64(out), ref, "bf16", "clamped")


# ---------------------------------------------------------------------------
# full-size configurations, default launch plan (the one bench.py times)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["qwen3_0_6b", "mistral_7b", "llama31_70b", "prefix_cow"])
def test_full_size_step_all_rows(ops, name):
    """The step at full size in bench.py's launch plan: slots, written rows
    and copied blocks bit-exact over the whole pool, and every output element
    of every (sequence, query head) against the oracle (which gathers each
    (sequence, KV head) once and shares it by the group's query heads)."""
    w = wl.build(name)
    c = wl.materialize(w)
    d = to_dev(c)
    slots, out = gpu_step(ops, w, d)
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    oslots, okc, ovc = oracle_step_pool(w, c)
    assert np.array_equal(slots.cpu().numpy(), oslots)
    # written slots and copied blocks bit-exact, and nothing else changed
    assert np.array_equal(storage(d["k_cache"]), okc)
    assert np.array_equal(storage(d["v_cache"]), ovc)
    del c["k_cache"], c["v_cache"], d
    outf = as_f64(out)
    assert np.all(np.isfinite(outf))
    ref = oracle.paged_attention_decode(storage(c["q"]), okc, ovc, w.block_tables,
                                        w.context_lens, w.scale, "bf16")
    check_attention(outf, ref, "bf16", name)


# ---------------------------------------------------------------------------
# fused slot mapping + KV write
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "qwen3_0_6b", "prefix_cow"])
def test_kv_append_matches_oracle(ops, name):
    w = wl.build(name)
    c = wl.materialize(w)
    d = to_dev(c)
    if len(w.copy_pairs):
        ops.kv_block_copy(d["k_cache"], d["v_cache"], d["copy_pairs"])
    slots = torch.full((w.num_seqs,), 7, dtype=torch.int64, device=DEV)
    ops.paged_kv_append(d["k_new"], d["v_new"], d["block_tables"], d["positions"], d["k_cache"],
                        d["v_cache"], slots)
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    oslots, okc, ovc = oracle_step_pool(w, c)
    assert np.array_equal(slots.cpu().numpy(), oslots)
    assert np.array_equal(storage(d["k_cache"]), okc)
    assert np.array_equal(storage(d["v_cache"]), ovc)


def test_kv_append_padding_and_device_checks(ops):
    w = wl.build_decode("append_edge", [5, 0, 9, 3], 4, 2, 64, 4, "bf16", seed=3)
    c = wl.materialize(w)
    d = to_dev(c)
    ops.paged_kv_append(d["k_new"], d["v_new"], d["block_tables"], d["positions"], d["k_cache"],
                        d["v_cache"])                 # no slot output
    assert ops.get_device_error() == 0
    _, okc, ovc = oracle_step_pool(w, c)
    assert np.array_equal(storage(d["k_cache"]), okc)
    bad = d["block_tables"].clone()
    bad[2, 2] = -5                                    # the block of position 8
    slots = torch.empty(4, dtype=torch.int64, device=DEV)
    before = d["k_cache"].clone()
    ops.paged_kv_append(d["k_new"], d["v_new"], bad, d["positions"], d["k_cache"], d["v_cache"],
                        slots)
    assert ops.get_device_error() == 1
    assert slots.cpu().tolist()[1] == -1 and slots.cpu().tolist()[2] == -1
    assert torch.equal(before.view(torch.int16), d["k_cache"].view(torch.int16))


# ---------------------------------------------------------------------------
# failure path: a pipeline wait that can never complete gives up and reports
# ---------------------------------------------------------------------------

def test_bounded_wait_gives_up_and_context_survives(ops):
    assert ops.get_device_error() == 0
    ops.selftest_wait_timeout(20_000_000)             # ~10 ms of SM cycles
    assert ops.get_device_error() == 6
    assert ops.get_device_error() == 0                # the word was cleared
    full_check(ops, wl.build("tiny"))                 # the context still works


# ---------------------------------------------------------------------------
# one very long sequence among short ones: its partials come from most of
# the grid (more than the reduce's all-at-once fast path holds)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("share", [False, True])
def test_many_partials(ops, share):
    lens = [16, 3, 65536, 40] + [16 + 7 * i for i in range(36)]
    w = wl.build_decode("skew", lens, 32, 8, 128, 16, "bf16", seed=9)
    c = wl.materialize(w)
    d = to_dev(c)
    slots = ops.slot_mapping(d["block_tables"], d["positions"], w.block_size, w.num_blocks)
    ops.paged_kv_write(d["k_new"], d["v_new"], slots, d["k_cache"], d["v_cache"])
    out = ops.paged_attention_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                     d["context_lens"], w.scale,
                                     max_context_len=w.max_context_len, share_prefix=share)
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    _, okc, ovc = oracle_step_pool(w, c)
    ref = oracle.paged_attention_decode(storage(c["q"]), okc, ovc, w.block_tables,
                                        w.context_lens, w.scale, "bf16")
    check_attention(as_f64(out), ref, "bf16", "many partials")
