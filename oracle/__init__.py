"""CPU fp64 oracle for the paged KV-cache decode path.

TEST INFRASTRUCTURE ONLY.  The oracle exists to check the CUDA library; it is
not part of the product.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import or call anything in
this package.  It shares no code with the CUDA path (no kernels, headers,
helpers, tables or generators) and never imports the package
``paged_kv_cache_115_gb300``.

Every function follows the pages' own definitions, cited by page title and
section:

* "19.2 KV Cache 系统化管理" (book chapter 19.2), §19.2.2 (block table,
  copy-on-write) and §19.2.3 "PagedAttention 的简化实现" (physical block pool,
  block table ``append_token``, block-wise online-softmax attention, and the
  paged-vs-dense self-check).
* "KV Cache：长上下文为什么吃显存，PagedAttention 怎么救", §01 (new-token
  attention ``q_t K_{1:t}^T -> softmax(.) V_{1:t}``) and §02 (GQA ratio).
* "推理与 KV Cache 02:分页、共享与回收如何协作", section "从一个位置找到缓存块"
  (logical block, offset and token-slot formulas and the worked K=4 example).

Submodules: ``oracle.quant`` (FP8 e4m3 / INT8 per-token KV formats, pinned in
``tests/test_oracle_quant_pins.py``) and ``oracle.prefill`` (multi-query
attention of several new tokens per sequence, pinned in
``tests/test_oracle_prefill_pins.py``).

Pins (checks against things other than the oracle itself) live in
``tests/test_oracle_pins.py``.  No function here is "parity unpinned".
"""

from .paged_attention import (  # noqa: F401
    decode,
    slot_mapping,
    kv_write,
    kv_block_copy,
    kv_block_swap,
    gather_kv,
    dense_attention,
    attention_rows,
    paged_attention_decode,
    paged_attention_decode_one,
    paged_attention_streaming,
    partial_state,
    merge_partials,
)
