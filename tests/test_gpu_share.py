"""GPU parity of the shared-prefix mode of decode attention.

With ``share_prefix`` the tensor-core kernel takes aligned groups of
m = 16 / G consecutive sequences, stages once per group the leading tokens
whose block-table entries are the same physical blocks in every member's row
("推理与 KV Cache 02", 前缀索引与 Block Table: requests that share a prefix
point their tables at the same whole blocks), and reads each member's
remaining tokens on their own; the partial states merge in the split-K
reduce.  The result is the same attention, so every case is checked element
by element against the fp64 oracle (NaN in every slot without history,
garbage past each table row), next to the plain launch on the same inputs.
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


def _oracle_step(w, c):
    kc, vc = storage(c["k_cache"]), storage(c["v_cache"])
    if len(w.copy_pairs):
        kc, vc = oracle.kv_block_copy(kc, vc, w.copy_pairs)
    slots = oracle.slot_mapping(w.block_tables, w.positions, w.block_size)
    kc, vc = oracle.kv_write(kc, vc, storage(c["k_new"]), storage(c["v_new"]), slots)
    return kc, vc


def _step_both(ops, w, seed=0, num_splits=0):
    """The decode step (copies, append) once, then attention plain and with
    shared-prefix groups over the same pool; returns both outputs and the
    oracle's."""
    c = wl.materialize(w, seed=seed)
    d = {k: v.to(DEV) for k, v in c.items()}
    if len(w.copy_pairs):
        ops.kv_block_copy(d["k_cache"], d["v_cache"], d["copy_pairs"])
    ops.paged_kv_append(d["k_new"], d["v_new"], d["block_tables"], d["positions"], d["k_cache"],
                        d["v_cache"])
    outs = {}
    for share in (False, True):
        outs[share] = ops.paged_attention_decode(
            d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"], w.scale,
            max_context_len=w.max_context_len, kernel=1, num_splits=num_splits,
            share_prefix=share)
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    kc, vc = _oracle_step(w, c)
    assert np.array_equal(storage(d["k_cache"]), kc)
    ref = oracle.paged_attention_decode(storage(c["q"]), kc, vc, w.block_tables, w.context_lens,
                                        w.scale, w.dtype)
    return as_f64(outs[False]), as_f64(outs[True]), ref


@pytest.mark.parametrize("G,K,fork,D", [
    (4, 16, 4, 128),    # groups of 4 = the forks of one request
    (4, 16, 3, 128),    # groups straddle requests: only the common prefix is shared
    (1, 16, 4, 128),    # groups of 16 sequences
    (2, 32, 4, 128),    # 32-token blocks: shared runs end mid-block
    (8, 16, 2, 128),    # groups of 2
    (4, 8, 4, 128),     # 8-token blocks (two blocks per tile)
    (2, 16, 5, 64),     # head_dim 64, groups of 8 over forks of 5
])
def test_forked_requests(ops, G, K, fork, D):
    H_kv = 4
    w = wl.build_prefix_cow(num_parents=7, prefix_len=96 if K != 32 else 128,
                            suffix_range=(1, 70), fork=fork, num_q_heads=G * H_kv,
                            num_kv_heads=H_kv, head_dim=D, block_size=K, seed=G + K + fork)
    plain, shared, ref = _step_both(ops, w)
    check_attention(plain, ref, "bf16", "plain")
    check_attention(shared, ref, "bf16", "shared")


def test_full_size_prefix_cow(ops):
    """The prefix-sharing configuration at full size (1024 forked samples of
    256 requests over a 2048-token prefix), every output element."""
    w = wl.build("prefix_cow")
    plain, shared, ref = _step_both(ops, w)
    check_attention(shared, ref, "bf16", "prefix_cow shared")
    check_attention(plain, ref, "bf16", "prefix_cow plain")


def _duplicate_rows(w, reps):
    """Workload whose consecutive rows repeat each sequence `reps` times
    (identical tables and lengths: the whole context shared, members with no
    private tokens); the first copy of each sequence writes its new token,
    the others write nothing."""
    idx = np.repeat(np.arange(w.num_seqs), reps)
    first = np.zeros(len(idx), bool)
    first[::reps] = True
    w.block_tables = w.block_tables[idx].copy()
    w.context_lens = w.context_lens[idx].copy()
    w.positions = np.where(first, w.positions[idx], -1).astype(np.int32)
    w.num_seqs = len(idx)
    return w


@pytest.mark.parametrize("lens,G", [
    ([17, 40, 64, 1, 0, 300, 33], 4),   # an empty sequence, 1-token and ragged
    ([512, 48, 16, 15], 8),
    ([100] * 5, 1),                      # 5 x 16 = 80 rows: groups of 16
])
def test_identical_rows(ops, lens, G):
    H_kv = 2
    base = wl.build_decode("dup", lens, G * H_kv, H_kv, 128, 16, "bf16", seed=len(lens) + G)
    w = _duplicate_rows(base, 16 // G)
    plain, shared, ref = _step_both(ops, w, seed=3)
    check_attention(shared, ref, "bf16", "identical rows")
    check_attention(plain, ref, "bf16", "identical rows, plain")
    assert np.array_equal(shared[w.context_lens == 0], np.zeros_like(ref[w.context_lens == 0]))


def test_no_sharing_and_split_counts(ops):
    """A batch with no shared blocks takes the shared-prefix path unchanged;
    several split counts of the stream-K grid."""
    w = wl.build_decode("noshare", [1, 700, 2048, 16, 0, 1333, 90, 5, 4096], 32, 8, 128, 16,
                        "bf16", seed=21)
    for ns in (0, 1, 3, 40):
        plain, shared, ref = _step_both(ops, w, num_splits=ns)
        check_attention(shared, ref, "bf16", f"no sharing, {ns} splits")


def test_shared_block_id_out_of_range_reported(ops):
    w = _duplicate_rows(wl.build_decode("bad", [64, 64], 8, 2, 128, 16, "bf16", seed=5), 4)
    c = wl.materialize(w, canary=False)
    d = {k: v.to(DEV) for k, v in c.items()}
    d["block_tables"][0:4, 1] = w.num_blocks + 3        # inside the shared run of group 0
    out = ops.paged_attention_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                     d["context_lens"], w.scale, max_context_len=64,
                                     share_prefix=True)
    assert ops.get_device_error() == 1
    assert torch.isfinite(out.float()).all()


def test_workspace_and_launch_count(ops):
    S, H_q, H_kv, D, K, L = 1024, 32, 8, 128, 16, 3072
    # the tensor-core plans (the automatic query also covers the CUDA-core
    # plan a misaligned pool would take): shared units keep one region of
    # partial slots per member, and the groups' shared lengths
    plain = ops.attention_workspace_bytes(S, H_q, H_kv, D, K, L, torch.bfloat16, kernel=1)
    shared = ops.attention_workspace_bytes(S, H_q, H_kv, D, K, L, torch.bfloat16, kernel=1,
                                           share_prefix=True)
    assert shared > plain
    assert ops.attention_workspace_bytes(S, H_q, H_kv, D, K, L, torch.bfloat16,
                                         share_prefix=True) >= shared
    assert ops.attention_launch_count(S, H_q, H_kv, D, K, L, torch.bfloat16,
                                      share_prefix=True) == 3
