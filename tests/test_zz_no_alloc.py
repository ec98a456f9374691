"""The no-allocation attention entry point against the regular one.

pkv_attention_decode_noalloc serves callers that cannot allocate device
memory when they run decode attention — an engine whose KV pool already took
the free HBM, or a decode path that must not enter the CUDA allocator.  Its
split-K scratch is a fixed array inside the library instead of a caller
workspace.  This test calls it through the C ABI twice in a row (different
queries, so leftovers of the first call would show) and checks each result
against pkv_attention_decode with a torch-allocated workspace, within the
tolerance the parity tests use; it also checks that sizes needing more
scratch than the array holds are refused.  It lives in its own file so that
pytest collects it last.
"""

import pytest
import torch

from paged_kv_cache_115_gb300 import workloads as wl
from tests._helpers import as_f64, check_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from paged_kv_cache_115_gb300 import build
    build.build()
    from paged_kv_cache_115_gb300 import ops as o
    o.get_device_error()
    return o


@pytest.mark.parametrize("case", ["tc_bf16", "cuda_core_f32"])
def test_noalloc_matches_regular_entry_point(ops, case):
    if case == "tc_bf16":
        w = wl.build_decode("noalloc", [1, 37, 700, 2048, 16, 0, 1333, 90], 32, 8, 128, 16,
                            "bf16", seed=11)
    else:
        w = wl.build("tiny")
    dev = torch.device("cuda", 0)
    t = {k: v.to(dev) for k, v in wl.materialize(w, seed=1, canary=False).items()}
    need = ops.attention_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                         w.block_size, w.max_context_len, t["q"].dtype)
    assert need <= ops.NOALLOC_SCRATCH_BYTES
    out_fixed = torch.empty_like(t["q"])
    # CUDA-core kernel: 4 tokens per partition, so that the tiny sequences
    # (up to 16 tokens) split and the partials and the reduce go through the
    # fixed scratch too
    kw = {} if case == "tc_bf16" else {"kernel": 2, "num_splits": 4}
    g = torch.Generator(device="cpu").manual_seed(5)
    for call in range(2):
        if call == 1:   # new queries: the second call must not depend on the first's scratch
            t["q"].copy_(torch.randn(t["q"].shape, generator=g).to(t["q"].dtype))
        ref = ops.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                                         t["context_lens"], w.scale,
                                         max_context_len=w.max_context_len, **kw)
        ops.paged_attention_decode_noalloc(t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                                           t["context_lens"], w.scale, out_fixed,
                                           w.max_context_len, **kw)
        torch.cuda.synchronize(dev)
        assert ops.get_device_error(dev) == 0
        check_attention(as_f64(out_fixed), as_f64(ref), w.dtype, f"{case} call {call}")


def test_noalloc_refuses_sizes_beyond_its_scratch(ops):
    # the CUDA-core kernel keeps one slot per 512-token partition of every
    # sequence: 128 sequences of 131072 tokens need far more than the array
    S, H_q, H_kv, D, K, L = 128, 32, 8, 128, 16, 131072
    need = ops.attention_workspace_bytes(S, H_q, H_kv, D, K, L, torch.bfloat16, kernel=2)
    assert need > ops.NOALLOC_SCRATCH_BYTES
    dev = torch.device("cuda", 0)
    q = torch.zeros((S, H_q, D), dtype=torch.bfloat16, device=dev)
    kc = torch.zeros((8, K, H_kv, D), dtype=torch.bfloat16, device=dev)
    bt = torch.zeros((S, L // K), dtype=torch.int32, device=dev)
    lens = torch.full((S,), L, dtype=torch.int32, device=dev)
    with pytest.raises(ops.PagedKVError, match="scratch"):
        ops.paged_attention_decode_noalloc(q, kc, kc, bt, lens, 0.1, torch.empty_like(q), L,
                                           kernel=2)
