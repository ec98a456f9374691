"""Host-side pieces of bench.py (no GPU): the staged input buffer of the
end-to-end leg, the DRAM-traffic records and their source hashes, and the
kernel name reported for the multi-query workloads."""

import json
import os

import numpy as np
import pytest
import torch

import bench
from paged_kv_cache_115_gb300 import workloads as wl


def test_staged_inputs_views_hold_the_values():
    g = torch.Generator().manual_seed(0)
    t = {"q": torch.randn((5, 3, 8), generator=g).to(torch.bfloat16),
         "tables": torch.arange(21, dtype=torch.int32).view(3, 7),
         "pos": torch.arange(5, dtype=torch.int64),
         "odd": torch.arange(3, dtype=torch.uint8)}
    ref = {k: v.clone() for k, v in t.items()}
    dev_buf, host_buf = bench.staged_inputs(t, list(t), torch.device("cpu"), pin=False)
    assert dev_buf.numel() == host_buf.numel() and dev_buf.numel() % 256 == 0
    for k in ref:
        assert t[k].dtype == ref[k].dtype and t[k].shape == ref[k].shape
        assert torch.equal(t[k], ref[k])
        # every view starts on a 256-byte boundary of the device buffer
        off = t[k].untyped_storage().data_ptr() - dev_buf.untyped_storage().data_ptr()
        assert t[k].storage_offset() * t[k].element_size() % 256 == 0 and off == 0
    # one copy of the host twin refills every view
    dev_buf.zero_()
    assert not torch.equal(t["tables"], ref["tables"])
    dev_buf.copy_(host_buf)
    for k in ref:
        assert torch.equal(t[k], ref[k])


def _write(root, rel, text):
    p = os.path.join(root, rel)
    os.makedirs(os.path.dirname(p), exist_ok=True)
    with open(p, "w") as f:
        f.write(text)


def test_traffic_record_follows_its_sources(tmp_path, monkeypatch):
    root = str(tmp_path)
    _write(root, "src/a.cuh", "kernel a")
    _write(root, "src/b.cuh", "kernel b")
    monkeypatch.setattr(bench, "ROOT", root)
    sha = bench.src_sha(["src/a.cuh", "src/b.cuh"])
    rec = {"w1": {"sources": ["src/a.cuh", "src/b.cuh"], "kernel_src_sha": sha,
                  "bytes_per_launch": 123.0}}
    _write(root, "profiles/t.json", json.dumps(rec))
    assert bench.read_traffic("t.json", "w1")["bytes_per_launch"] == 123.0
    assert bench.read_traffic("t.json", "w2") is None          # another workload
    assert bench.read_traffic("missing.json", "w1") is None
    assert "unchanged" in bench.traffic_record("t.json", "w1")[1]
    _write(root, "src/b.cuh", "kernel b, changed")
    assert bench.read_traffic("t.json", "w1") is None          # stale after a change
    rec, note = bench.traffic_record("t.json", "w1")
    assert rec is None and "earlier kernel sources" in note
    assert "no ncu record for w2" in bench.traffic_record("t.json", "w2")[1]


def test_committed_traffic_records_name_their_workload():
    t = bench.read_traffic()
    if t is not None:
        assert t["workload"] in wl.CONFIG_NAMES and t["kv_format"] == "bf16"
    with open(os.path.join(bench.ROOT, "profiles", "prefill_traffic.json")) as f:
        recs = json.load(f)
    for name, r in recs.items():
        assert name in wl.PREFILL_NAMES and r["workload"] == name
        assert r["bytes_per_launch"] >= r["algorithmic_bytes_per_launch"] * 0.9


@pytest.mark.parametrize("name,kernel", [("suffix_prefill", "attn_prefill_tc05x2_kernel"),
                                         ("chunked_prefill", "attn_prefill_tc05x2_kernel (one"),
                                         ("speculative_decode", "attn_tc_kernel")])
def test_prefill_kernel_name(name, kernel):
    assert bench.prefill_kernel(wl.build_prefill(name)).startswith(kernel)


def test_prefill_flops_closed_form():
    # one sequence of P cached + n new tokens: sum over i < n of (P + i + 1) keys
    class W:
        prefix = np.array([10]); news = np.array([4]); head_dim = 2; num_q_heads = 3
    assert bench.prefill_flops(W) == 4 * 2 * 3 * (11 + 12 + 13 + 14)


def _reference_line(argv, capsys):
    bench.main(argv)
    out = capsys.readouterr().out.strip().splitlines()[-1]
    return json.loads(out)


def test_reference_arm_decode(capsys):
    d = _reference_line(["--impl", "reference", "--workload", "tiny", "--steps", "1",
                         "--warmup", "1", "--cpu-budget", "1"], capsys)
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert 1 <= d["cpu_baseline"]["cores"] <= bench._host_cores()
    assert d["e2e"]["value"] == d["value"] and d["gpu_launches"] == 0


@pytest.mark.parametrize("name,unit", [("chunked_prefill", "GB/s"),
                                       ("speculative_decode", "GB/s")])
def test_reference_arm_prefill_units(capsys, name, unit):
    # bandwidth-bound multi-query workloads report K/V GB/s, like the GPU arm
    d = _reference_line(["--impl", "reference", "--op", "prefill", "--workload", name,
                         "--steps", "1", "--warmup", "1", "--cpu-budget", "1"], capsys)
    assert d["unit"] == unit and d["cpu_baseline"]["unit"] == unit and d["value"] > 0


def test_deal_whole_sequences_or_items():
    items = [(s, j) for s in range(8) for j in range(2)]
    shares = bench._deal(items, 4, 8)              # 2 sequences per process: whole sequences
    assert sorted(it for sh in shares for it in sh) == items
    assert all(len({s for s, _ in sh}) == 2 and len(sh) == 4 for sh in shares)
    shares = bench._deal(items, 6, 8)              # fewer: items round robin
    assert sorted(it for sh in shares for it in sh) == items


@pytest.mark.parametrize("name", ["tiny", "prefix_cow"])
def test_accuracy_check_plumbing(name):
    """The bench's accuracy check on the CPU: the snapshot of the sampled
    sequences, the oracle's own step on it, and the comparison.  The stand-in
    "GPU output" is the oracle's result on the full workload, so the error is
    0; a perturbed copy is reported out of tolerance."""
    import numpy as np
    import torch
    import oracle
    from paged_kv_cache_115_gb300 import workloads as wl
    from tests._helpers import storage
    w = wl.build(name)
    if name == "prefix_cow":                        # keep the CPU work small
        w = wl.build_prefix_cow(num_parents=4, prefix_len=64, suffix_range=(3, 40))
    t = wl.materialize(w, canary=False)
    snap = bench._accuracy_snapshot(w, t, "bf16", None)
    kc, vc = storage(t["k_cache"]), storage(t["v_cache"])
    if len(w.copy_pairs):
        kc, vc = oracle.kv_block_copy(kc, vc, w.copy_pairs)
    slots = oracle.slot_mapping(w.block_tables, w.positions, w.block_size)
    kc, vc = oracle.kv_write(kc, vc, storage(t["k_new"]), storage(t["v_new"]), slots)
    ref = oracle.paged_attention_decode(storage(t["q"]), kc, vc, w.block_tables, w.context_lens,
                                        w.scale, w.dtype)
    td = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    out = torch.from_numpy(ref).to(td)
    path = bench._save_snapshot(snap, out)
    try:
        a = bench._accuracy(path)
    finally:
        os.remove(path)
    # the stand-in output is the reference rounded to the storage type
    assert a["within_tolerance"] and a["elements"] > 0
    bad = out.clone()
    bad[snap["_samples"][0], 0, 0] += 1.0
    path = bench._save_snapshot(snap, bad)
    try:
        assert not bench._accuracy(path)["within_tolerance"]
    finally:
        os.remove(path)
