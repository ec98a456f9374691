#!/usr/bin/env python
"""Benchmark of one decode step of the paged KV-cache path on GB300.

A step is the whole hot path for one attention layer of a decode batch:
copy-on-write block copies (when the workload has any), slot mapping of the
new tokens, the slot-mapped KV write, and paged decode attention (partition
kernel + split-K reduce).  The step is captured once as a CUDA graph and
replayed (`--eager`: plain launches).  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores

Under torchrun every rank runs its own replica of the workload on its own GPU
(weak scaling, no collective on the data path); the value is the sum of all
ranks' bytes over the slowest rank's time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention KV GB/s (% of GB300 HBM peak); decode tokens/s per layer"
DEFAULT_WORKLOAD = "qwen3_0_6b"
# sources of the dominant kernel (attn_tc_kernel); a recorded DRAM-traffic
# figure is used only while these files are unchanged
KERNEL_SRC = ["paged_kv_cache_115_gb300/csrc/pkv_attention_tc.cuh",
              "paged_kv_cache_115_gb300/csrc/pkv_attention_common.cuh",
              "paged_kv_cache_115_gb300/csrc/pkv_device.cuh"]
# sources of the two-tile tcgen05 prefill kernel
PREFILL_SRC = ["paged_kv_cache_115_gb300/csrc/pkv_prefill_tc05x2.cuh",
               "paged_kv_cache_115_gb300/csrc/pkv_prefill_tc05.cuh",
               "paged_kv_cache_115_gb300/csrc/pkv_umma.cuh",
               "paged_kv_cache_115_gb300/csrc/pkv_device.cuh"]


def src_sha(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def kernel_src_sha() -> str:
    return src_sha(KERNEL_SRC)


def read_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def traffic_record(name="attention_traffic.json", workload=None):
    """(record, note): DRAM bytes per launch of a kernel from a committed ncu
    summary, valid only while the kernel's sources are unchanged since the
    capture, and a note saying where the figure comes from or why there is
    none.  Files with several records are keyed by workload name."""
    try:
        with open(os.path.join(ROOT, "profiles", name)) as f:
            t = json.load(f)
    except OSError:
        return None, f"no ncu record (profiles/{name} missing)"
    if workload is not None:
        t = t.get(workload)
        if t is None:
            return None, f"no ncu record for {workload} in profiles/{name}"
    if t.get("kernel_src_sha") != src_sha(t.get("sources", KERNEL_SRC)):
        return None, (f"profiles/{name} was captured on earlier kernel sources; no ncu "
                      f"capture of the current ones")
    return t, (f"ncu dram__bytes_read.sum + dram__bytes_write.sum per launch, "
               f"profiles/{name} (kernel sources unchanged since the capture)")


def read_traffic(name="attention_traffic.json", workload=None):
    """The record of traffic_record, or None."""
    return traffic_record(name, workload)[0]


def workload_desc(w) -> dict:
    import numpy as np
    return {
        "workload": w.name,
        "num_seqs": w.num_seqs,
        "num_q_heads": w.num_q_heads,
        "num_kv_heads": w.num_kv_heads,
        "head_dim": w.head_dim,
        "block_size": w.block_size,
        "num_blocks": w.num_blocks,
        "context_lens": {"min": int(w.context_lens.min()), "max": int(w.context_lens.max()),
                         "mean": float(np.mean(w.context_lens)), "sum": int(w.context_lens.sum())},
        "copy_pairs": int(len(w.copy_pairs)),
        "new_tokens": int((w.positions >= 0).sum()),
        "step": ("kv_block_copy + " if len(w.copy_pairs) else "")
        + "paged_kv_append (slot mapping + KV write, fused) + paged_attention_decode "
          "(partition + split-K reduce)",
    }


def staged_inputs(t: dict, names, dev, pin: bool = True):
    """One device buffer and one pinned host buffer holding the tensors
    t[name] back to back (256-byte aligned), so that a step's host-to-device
    transfer is a single copy; t[name] is rebound to its view of the device
    buffer (same values, dtype and shape)."""
    import torch
    offs, total = {}, 0
    for k in names:
        offs[k] = total
        total += -(-(t[k].numel() * t[k].element_size()) // 256) * 256
    dev_buf = torch.empty(total, dtype=torch.uint8, device=dev)
    host_buf = torch.empty(total, dtype=torch.uint8, pin_memory=pin)
    for k in names:
        src = t[k].contiguous()
        n = src.numel() * src.element_size()
        host_buf[offs[k]:offs[k] + n].view(src.dtype).view(src.shape).copy_(src.cpu())
        view = dev_buf[offs[k]:offs[k] + n].view(src.dtype).view(src.shape)
        view.copy_(src)
        t[k] = view
    return dev_buf, host_buf


def run_pipelined(n, sets, compute, stream, cs, start_ev=None):
    """n end-to-end steps over two buffer sets (dev_in, host_in, dev_out,
    host_out): step i copies host_in -> dev_in of set i % 2 on the copy stream
    cs, computes on `stream` (compute(b) launches the step over set b), and
    copies dev_out -> host_out on cs.  Step i+1's input copy is queued before
    step i's output copy; a set is refilled only after the step two back has
    read it, and its output is overwritten only after it has been copied."""
    import torch
    h2d_ev = [torch.cuda.Event() for _ in range(2)]
    comp_ev = [torch.cuda.Event() for _ in range(2)]
    d2h_ev = [torch.cuda.Event() for _ in range(2)]

    def h2d_copy(i):
        b = i & 1
        with torch.cuda.stream(cs):
            if i >= 2:
                cs.wait_event(comp_ev[b])
            sets[b][0].copy_(sets[b][1], non_blocking=True)
            h2d_ev[b].record(cs)

    if start_ev is not None:
        cs.wait_event(start_ev)
    h2d_copy(0)
    for i in range(n):
        b = i & 1
        if i + 1 < n:
            h2d_copy(i + 1)
        stream.wait_event(h2d_ev[b])
        if i >= 2:
            stream.wait_event(d2h_ev[b])
        compute(b)
        comp_ev[b].record(stream)
        with torch.cuda.stream(cs):
            cs.wait_event(comp_ev[b])
            sets[b][3].copy_(sets[b][2], non_blocking=True)
            d2h_ev[b].record(cs)
    stream.wait_stream(cs)


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle baseline (the only place bench.py runs the oracle)
# ---------------------------------------------------------------------------
def _cpu_sample(name: str, seed: int, budget_s: float) -> dict:
    import numpy as np
    import torch
    import oracle
    from paged_kv_cache_115_gb300 import accounting, workloads as wl

    full = wl.build(name, seed=seed)
    order = list(range(full.num_seqs))
    done_bytes, done_tokens, done_seqs, elapsed = 0, 0, 0, 0.0
    H_kv, D = full.num_kv_heads, full.head_dim
    eb = full.elem_bytes
    for s in order:
        L = int(full.context_lens[s])
        sub = wl.build_decode("sample", [L], full.num_q_heads, H_kv, D, full.block_size,
                              full.dtype, seed=seed + s)
        t = wl.materialize(sub, seed=seed + s, canary=False)

        def st(x):
            x = x.contiguous()
            return x.view(torch.int16).numpy().view(np.uint16) if x.dtype == torch.bfloat16 \
                else x.numpy()
        q, kc, vc = st(t["q"]), st(t["k_cache"]), st(t["v_cache"])
        t0 = time.perf_counter()
        slots = oracle.slot_mapping(sub.block_tables, sub.positions, sub.block_size)
        kc, vc = oracle.kv_write(kc, vc, st(t["k_new"]), st(t["v_new"]), slots)
        oracle.paged_attention_decode(q, kc, vc, sub.block_tables, sub.context_lens, sub.scale,
                                      sub.dtype)
        elapsed += time.perf_counter() - t0
        done_bytes += accounting.attention_kv_bytes([L], H_kv, D, eb)
        done_tokens += 1
        done_seqs += 1
        if elapsed >= budget_s:
            break
    return {"bytes": done_bytes, "seconds": elapsed, "seqs": done_seqs,
            "of_seqs": full.num_seqs, "tokens": int(sum(full.context_lens[:done_seqs]))}


def run_cpu_baseline(name: str, seed: int, budget_s: float) -> dict:
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    code = ("import json,sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench._cpu_sample(%r, %d, %f)))" % (ROOT, name, seed, budget_s))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       cwd=ROOT, timeout=max(600, budget_s * 20))
    if r.returncode != 0:
        raise RuntimeError("cpu baseline failed: " + r.stderr[-2000:])
    res = json.loads(r.stdout.strip().splitlines()[-1])
    gbs = res["bytes"] / res["seconds"] / 1e9
    return {
        "value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
        "seconds": res["seconds"],
        "decode_tokens_per_s_per_layer": res["seqs"] / res["seconds"],
        "sample": (f"fp64 numpy oracle (slot mapping + KV write + attention), single-threaded, "
                   f"on the first {res['seqs']} of {res['of_seqs']} sequences of {name} "
                   f"({res['tokens']} cached tokens, {res['bytes'] / 1e6:.1f} MB of KV)"),
    }


# ---------------------------------------------------------------------------
# multi-rank helpers (one process per GPU; no collective on the data path)
# ---------------------------------------------------------------------------
def max_over_ranks(values, device):
    """Element-wise maximum of per-rank timings (the slowest rank sets the
    job's time).  A no-op without an initialised process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank draws its own replica of the workload (weak scaling)."""
    return base_seed + rank


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_gpu(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)

    from paged_kv_cache_115_gb300 import accounting, build, workloads as wl
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        dist.barrier()
    from paged_kv_cache_115_gb300 import ops

    w = wl.build(args.workload, seed=rank_seed(args.seed, rank),
                 block_size=args.block_size or None)
    t = wl.materialize(w, device=dev, seed=rank_seed(args.seed, rank), canary=False,
                       values_device="cuda")
    fmt = args.kv_format
    stream = torch.cuda.current_stream(dev)
    out = torch.empty_like(t["q"])
    slots = torch.empty(w.num_seqs, dtype=torch.int64, device=dev)
    has_copy = len(w.copy_pairs) > 0
    max_len = w.max_context_len
    if fmt == "bf16":
        kv_bytes = accounting.attention_kv_bytes(w.context_lens, w.num_kv_heads, w.head_dim,
                                                 w.elem_bytes)
        ws_bytes = ops.attention_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                                 w.head_dim, w.block_size, max_len, t["q"].dtype)
    else:
        # one-byte pools of seeded random codes (finite e4m3 codes; int8 codes
        # with per-slot scales); the bf16 pools are dropped
        g = torch.Generator(device=dev)
        g.manual_seed(rank_seed(args.seed, rank) + 7)
        shape = t["k_cache"].shape
        del t["k_cache"], t["v_cache"]
        for name in ("k_cache", "v_cache"):
            c = torch.randint(0, 256, shape, generator=g, device=dev, dtype=torch.int32)
            c = torch.where((c & 0x7F) == 0x7F, c - 1, c).to(torch.uint8)
            t[name] = c if fmt == "fp8" else c.view(torch.int8)
        if fmt == "int8":
            n = shape[0] * shape[1]
            t["k_ts"] = torch.rand(n, generator=g, device=dev) * 0.02 + 0.001
            t["v_ts"] = torch.rand(n, generator=g, device=dev) * 0.02 + 0.001
            qd = ops.kv_quant("int8", k_token_scales=t["k_ts"], v_token_scales=t["v_ts"])
        else:
            qd = ops.kv_quant("fp8", 0.05, 0.05)
        kv_bytes = accounting.attention_kv_bytes(w.context_lens, w.num_kv_heads, w.head_dim, 1)
        if fmt == "int8":
            kv_bytes += int(w.context_lens.sum()) * 2 * 4      # one K and one V scale per token
        ws_bytes = ops.attention_quant_workspace_bytes(w.num_seqs, w.num_q_heads,
                                                       w.num_kv_heads, w.head_dim, w.block_size,
                                                       max_len, t["q"].dtype, qd)
    workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    use_graph = not args.eager
    # the step's inputs live back to back in one device buffer with a pinned
    # host twin, so that the end-to-end leg moves them in one copy
    names = ["q", "k_new", "v_new", "block_tables", "context_lens", "positions"]
    if has_copy:
        names.append("copy_pairs")
    dev_stage, host_stage = staged_inputs(t, names, dev)

    def attention():
        if fmt == "bf16":
            ops.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                                       t["context_lens"], w.scale, out=out,
                                       max_context_len=max_len, workspace=workspace)
        else:
            ops.paged_attention_decode_quant(t["q"], t["k_cache"], t["v_cache"],
                                             t["block_tables"], t["context_lens"], w.scale, qd,
                                             out=out, max_context_len=max_len,
                                             workspace=workspace)

    def copy_fn():
        if fmt == "bf16":
            ops.kv_block_copy(t["k_cache"], t["v_cache"], t["copy_pairs"])
        else:
            ops.kv_block_copy_quant(t["k_cache"], t["v_cache"], t["copy_pairs"], qd)

    def append_fn():
        # slot mapping + KV write of the new tokens in one fused launch
        if fmt == "bf16":
            ops.paged_kv_append(t["k_new"], t["v_new"], t["block_tables"], t["positions"],
                                t["k_cache"], t["v_cache"], slots)
        else:
            ops.paged_kv_append_quant(t["k_new"], t["v_new"], t["block_tables"], t["positions"],
                                      t["k_cache"], t["v_cache"], qd, slots)

    def prologue():
        if has_copy:
            copy_fn()
        append_fn()

    # kernels launched per step (ours only)
    attn_launches = ops.attention_launch_count(w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                               w.head_dim, w.block_size, max_len, t["q"].dtype)
    copy_launches = (1 if fmt != "int8" else 2) if has_copy else 0
    launches_per_step = copy_launches + 1 + attn_launches

    for _ in range(max(args.warmup, 3)):
        prologue()
        attention()
    torch.cuda.synchronize(dev)
    assert ops.get_device_error(dev) == 0

    K = args.steps
    if use_graph:
        # the whole step as one graph; the attention call alone as another
        # (for the per-launch roofline timing)
        # (capture needs a side stream; replays run on the timing stream)
        g_step, g_attn = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.graph(g_step, stream=cap):
            prologue()
            attention()
        with torch.cuda.graph(g_attn, stream=cap):
            attention()
        stream.wait_stream(cap)
        torch.cuda.synchronize(dev)
        for _ in range(3):
            g_step.replay()
        torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index) if rank == 0 else None
    time.sleep(0.2 if clocks else 0)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    start.record(stream)
    for i in range(K):
        if use_graph:
            g_step.replay()
        else:
            prologue()
            ev[i][0].record(stream)
            attention()
            ev[i][1].record(stream)
    stop.record(stream)
    torch.cuda.synchronize(dev)
    if use_graph:
        for i in range(K):
            ev[i][0].record(stream)
            g_attn.replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
    clock_info = clocks.stop() if clocks else None
    if world > 1:
        dist.barrier()
    total_ms = start.elapsed_time(stop)
    attn_ms = [a.elapsed_time(b) for a, b in ev]
    attn_avg_ms = sum(attn_ms) / K
    assert ops.get_device_error(dev) == 0

    # ---- each row of the step alone: events around the row only, L2 flushed
    # (a 256 MB write) before every timed launch
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    row_fns = []
    pool_eb = w.elem_bytes if fmt == "bf16" else 1
    n_new = int((w.positions >= 0).sum())
    if has_copy:
        row_fns.append(("kv_block_copy", copy_fn,
                        accounting.block_copy_bytes(len(w.copy_pairs), w.block_size,
                                                    w.num_kv_heads, w.head_dim, pool_eb)))
    row_fns.append(("paged_kv_append", append_fn,
                    n_new * w.num_kv_heads * w.head_dim * 2 * (w.elem_bytes + pool_eb)))
    row_fns.append(("paged_attention_decode", attention, kv_bytes))
    rows = {}
    R = max(5, min(50, K))
    for name, fn, nbytes in row_fns:
        times = []
        for _ in range(R):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize(dev)
            times.append(a.elapsed_time(b))
        med = statistics.median(times)
        rows[name] = {"median_us": med * 1e3, "min_us": min(times) * 1e3,
                      "algorithmic_bytes": nbytes, "GBps": nbytes / (med * 1e-3) / 1e9,
                      "frac": None}
    del flush
    assert ops.get_device_error(dev) == 0

    # ---- end to end through the public API with host buffers.  Every step
    # copies its inputs from a pinned host buffer (one copy) and reads its
    # output back (one copy).  The copies run on a second stream against two
    # sets of staged inputs and outputs, so that step i+1's input copy and
    # step i's output copy overlap the neighbouring steps' compute.
    out0, views0 = out, {k: t[k] for k in names}
    t1 = dict(views0)
    dev_stage1, host_stage1 = staged_inputs(t1, names, dev)
    out1 = torch.empty_like(out0)
    sets = [(dev_stage, host_stage, views0, out0), (dev_stage1, host_stage1, t1, out1)]
    host_outs = [torch.empty(out0.shape, dtype=out0.dtype, pin_memory=True) for _ in range(2)]
    h2d = host_stage.numel()
    d2h = host_outs[0].numel() * host_outs[0].element_size()
    graphs = [g_step] if use_graph else []
    if use_graph:
        # the same step over the second set (closures read t and out when called)
        for k in names:
            t[k] = t1[k]
        out = out1
        g1 = torch.cuda.CUDAGraph()
        cap.wait_stream(stream)
        with torch.cuda.graph(g1, stream=cap):
            prologue()
            attention()
        stream.wait_stream(cap)
        graphs.append(g1)
        for k in names:
            t[k] = views0[k]
        out = out0
        torch.cuda.synchronize(dev)
    cs = torch.cuda.Stream(dev)
    pipe_sets = [(sets[i][0], sets[i][1], sets[i][3], host_outs[i]) for i in range(2)]

    def e2e_compute(b):
        nonlocal out
        if use_graph:
            graphs[b].replay()
            return
        for k in names:
            t[k] = sets[b][2][k]
        out = sets[b][3]
        prologue()
        attention()
        for k in names:
            t[k] = views0[k]
        out = out0

    def e2e_run(n, start_ev=None):
        run_pipelined(n, pipe_sets, e2e_compute, stream, cs, start_ev)

    e2e_steps = max(4, min(K, 200))
    e2e_run(4)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    e0.record(stream)
    e2e_run(e2e_steps, start_ev=e0)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    # the same inputs in both sets: the outputs read back equal the timed step's
    ref_out = out0.cpu()
    for h in host_outs:
        assert torch.equal(h.view(torch.int16), ref_out.view(torch.int16)), "e2e output differs"

    # ---- max over ranks
    total_ms, e2e_ms, attn_avg_ms = max_over_ranks([total_ms, e2e_ms, attn_avg_ms], dev)
    ms_step = total_ms / K
    value = world * kv_bytes / (ms_step * 1e-3) / 1e9
    e2e_value = world * kv_bytes / (e2e_ms * 1e-3) / 1e9

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None

    peaks, peak_src = read_peaks()
    hbm = float(peaks["hbm_gbs"])
    achieved = kv_bytes / (attn_avg_ms * 1e-3) / 1e9
    for r in rows.values():
        r["frac"] = r["GBps"] / hbm
    traffic, traffic_src = traffic_record()
    if traffic and (traffic.get("workload") != w.name or traffic.get("kv_format") != fmt
                    or traffic.get("block_size") != w.block_size):
        traffic = None                  # the record is for another workload
        traffic_src = "the ncu record is for another workload, pool format or block size"
    cfg = workload_desc(w)
    cfg["l2"] = (f"inputs larger than L2: {kv_bytes / 1e6:.0f} MB of KV read per step "
                 f"vs 129 MB L2; no flush between steps")
    cfg["parallelism"] = f"replicas x{world}" if world > 1 else "single GPU"
    cfg["launch"] = "CUDA graph replay (one graph per step)" if use_graph else "eager launches"
    blocks_used = int(sum(-(-int(L) // w.block_size) for L in w.context_lens))
    cfg["kv_reserved_bytes"] = blocks_used * w.block_size * w.num_kv_heads * w.head_dim * 2 * \
        (w.elem_bytes if fmt == "bf16" else 1)
    cfg["tail_waste_tokens"] = blocks_used * w.block_size - int(w.context_lens.sum())
    cfg["block_table_bytes"] = int(w.block_tables.nbytes)
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype if fmt == "bf16" else f"{w.dtype} q / {fmt} KV",
        "data": "synthetic: seeded N(0,1) q/k/v rounded to bf16; block tables from a seeded "
                "shuffled free list; lengths drawn per the workload recipe",
        "config": cfg,
        "hbm_frac": value / world / hbm,
        "decode_tokens_per_s_per_layer": world * w.num_seqs / (ms_step * 1e-3),
        "roofline": {
            "bound": "hbm",
            "kernel": "pkv_attention_decode (partition + split-K reduce)",
            "achieved": achieved,
            "peak": hbm,
            "peak_source": f"{peak_src} hbm_gbs (copy, read+write)",
            "unit": "GB/s",
            "frac": achieved / hbm,
            "algorithmic_bytes_per_launch": kv_bytes,
            "avg_launch_ms": attn_avg_ms,
            "traffic": traffic["bytes_per_launch"] if traffic else None,
            "traffic_source": traffic_src,
        },
        "e2e": {"value": e2e_value, "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "decode_tokens_per_s_per_layer": world * w.num_seqs / (e2e_ms * 1e-3),
                "copies": "per step one pinned-host-to-device copy of the inputs and one "
                          "device-to-pinned-host copy of the output, on a second stream with "
                          "two staged buffer sets, overlapping the neighbouring steps"},
        "rows": rows,
        "gpu_launches": launches_per_step * K,
        "clocks": clock_info,
    }
    if not args.no_cpu_baseline:
        try:
            line["cpu_baseline"] = run_cpu_baseline(args.workload, args.seed, args.cpu_budget)
        except Exception as e:  # report, do not hide the GPU number
            line["cpu_baseline"] = {"value": None, "error": str(e)[:300], "kind": "oracle"}
    if world > 1:
        dist.destroy_process_group()
    return line


# ---------------------------------------------------------------------------
# block swap (GPU <-> pinned host): preempt half the batch and bring it back
# ---------------------------------------------------------------------------
SWAP_METRIC = "KV block swap GB/s (GPU pool <-> pinned host pool, out + in)"


def swap_plan(w, seed: int):
    """Every other sequence of the workload is preempted by swap: its blocks
    (K and V) go to a host pool in a seeded shuffled order, and come back into
    a seeded permutation of the same GPU blocks (scattered placement)."""
    import numpy as np
    rng = np.random.default_rng(seed + 101)
    blocks = []
    for s in range(1, w.num_seqs, 2):
        n = -(-int(w.context_lens[s]) // w.block_size)
        blocks.extend(int(b) for b in w.block_tables[s, :n])
    blocks = np.array(blocks, np.int64)
    host = rng.permutation(len(blocks)).astype(np.int64)
    out_pairs = np.stack([blocks, host], 1)
    in_pairs = np.stack([host, rng.permutation(blocks)], 1)
    return out_pairs, in_pairs


def _swap_cpu_sample(budget_s: float) -> dict:
    """The oracle's swap on 512 pairs between two 512-block pools of the
    Qwen-shaped geometry, repeated for about budget_s seconds."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(0)
    shape = (512, 16, 8, 128)
    a = rng.integers(0, 2**16, size=shape, dtype=np.uint16)
    b = rng.integers(0, 2**16, size=shape, dtype=np.uint16)
    pairs = np.stack([rng.permutation(512), rng.permutation(512)], 1)
    moved, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        oracle.kv_block_swap(a, a, b, b, pairs)
        moved += 2 * a.nbytes
    sec = time.perf_counter() - t0
    return {"bytes": moved, "seconds": sec}


def run_swap(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    from paged_kv_cache_115_gb300 import build, workloads as wl
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        dist.barrier()
    from paged_kv_cache_115_gb300 import ops

    w = wl.build(args.workload, seed=rank_seed(args.seed, rank))
    out_np, in_np = swap_plan(w, rank_seed(args.seed, rank))
    n = len(out_np)
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    td = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    g = torch.Generator(device=dev)
    g.manual_seed(rank_seed(args.seed, rank))
    kc = torch.empty(shape, dtype=td, device=dev).normal_(generator=g)
    vc = torch.empty(shape, dtype=td, device=dev).normal_(generator=g)
    hk = torch.empty((n,) + shape[1:], dtype=td).pin_memory()
    hv = torch.empty((n,) + shape[1:], dtype=td).pin_memory()
    out_pairs = torch.from_numpy(out_np).to(dev)
    in_pairs = torch.from_numpy(in_np).to(dev)
    blk = w.block_size * w.num_kv_heads * w.head_dim * kc.element_size()
    dir_bytes = 2 * n * blk                       # K and V, one direction
    step_bytes = 2 * dir_bytes
    stream = torch.cuda.current_stream(dev)

    def swap_out():
        ops.kv_block_swap(kc, vc, hk, hv, out_pairs)

    def swap_in():
        ops.kv_block_swap(hk, hv, kc, vc, in_pairs)

    for _ in range(max(args.warmup, 3)):
        swap_out()
        swap_in()
    torch.cuda.synchronize(dev)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    for a, b, c in ev:
        a.record(stream)
        swap_out()
        b.record(stream)
        swap_in()
        c.record(stream)
    torch.cuda.synchronize(dev)
    clock_info = clocks.stop()
    out_ms = statistics.median(a.elapsed_time(b) for a, b, _ in ev)
    in_ms = statistics.median(b.elapsed_time(c) for _, b, c in ev)
    total_ms = ev[0][0].elapsed_time(ev[-1][2])

    # the link's own rate for the same bytes: one contiguous copy each way
    dflat = torch.empty(dir_bytes, dtype=torch.uint8, device=dev)
    hflat = torch.empty(dir_bytes, dtype=torch.uint8).pin_memory()

    def best(fn, reps=5):
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ts.append(e0.elapsed_time(e1))
        return min(ts)

    d2h_ms = best(lambda: hflat.copy_(dflat, non_blocking=True))
    h2d_ms = best(lambda: dflat.copy_(hflat, non_blocking=True))
    # one copy call per block and tensor, the way a loop of memcpys would do it
    blocks_np = out_np[: min(n, 1024)]
    pb_bytes = 2 * len(blocks_np) * blk

    def per_block():
        for s_, d_ in blocks_np:
            hk[int(d_)].copy_(kc[int(s_)], non_blocking=True)
            hv[int(d_)].copy_(vc[int(s_)], non_blocking=True)
    per_block()
    pb_ms = best(per_block, reps=2)
    del dflat, hflat

    # e2e: the public call with the pairs read straight from pinned host memory
    out_pin, in_pin = torch.from_numpy(out_np).pin_memory(), torch.from_numpy(in_np).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(3, min(K, 20))
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(e2e_steps):
        ops.kv_block_swap(kc, vc, hk, hv, out_pin)
        ops.kv_block_swap(hk, hv, kc, vc, in_pin)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps

    total_ms, e2e_ms = max_over_ranks([total_ms, e2e_ms], dev)
    ms_step = total_ms / K
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None
    link_ms = d2h_ms + h2d_ms
    achieved = step_bytes / ((out_ms + in_ms) * 1e-3) / 1e9
    peak = step_bytes / (link_ms * 1e-3) / 1e9
    cfg = {"workload": f"{w.name}: swap out and back in every other sequence",
           "sequences_swapped": len(range(1, w.num_seqs, 2)), "blocks_swapped": n,
           "block_bytes_per_tensor": blk, "num_kv_heads": w.num_kv_heads,
           "head_dim": w.head_dim, "block_size": w.block_size,
           "step": "kv_block_swap GPU->pinned host (K+V), then pinned host->GPU into a "
                   "permutation of the same blocks",
           "l2": f"{dir_bytes / 1e6:.0f} MB per direction vs 129 MB L2; no flush",
           "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}
    line = {
        "metric": SWAP_METRIC, "value": world * step_bytes / (ms_step * 1e-3) / 1e9,
        "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic: seeded N(0,1) pool values",
        "config": cfg,
        "roofline": {"bound": "link", "kernel": "block_move_kernel (swap out + swap in)",
                     "achieved": achieved, "peak": peak,
                     "peak_source": "measured in this run: one contiguous pinned-host copy of "
                                    "the same bytes each way (cudaMemcpyAsync via torch)",
                     "unit": "GB/s", "frac": achieved / peak,
                     "algorithmic_bytes_per_launch": dir_bytes,
                     "avg_launch_ms": (out_ms + in_ms) / 2, "traffic": None,
                     "traffic_source": "none: the swap is bound by the host link, not DRAM"},
        "rows": {"swap_out": {"median_us": out_ms * 1e3,
                              "GBps": dir_bytes / (out_ms * 1e-3) / 1e9,
                              "contiguous_copy_GBps": dir_bytes / (d2h_ms * 1e-3) / 1e9},
                 "swap_in": {"median_us": in_ms * 1e3,
                             "GBps": dir_bytes / (in_ms * 1e-3) / 1e9,
                             "contiguous_copy_GBps": dir_bytes / (h2d_ms * 1e-3) / 1e9},
                 "per_block_copy_calls": {"blocks": len(blocks_np), "ms": pb_ms,
                                          "GBps": pb_bytes / (pb_ms * 1e-3) / 1e9}},
        "e2e": {"value": world * step_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": dir_bytes + 2 * out_pin.nbytes,
                "d2h_bytes_per_step": dir_bytes},
        "gpu_launches": 2 * K,
        "clocks": clock_info,
    }
    if not args.no_cpu_baseline:
        r = _swap_cpu_sample(min(args.cpu_budget, 10.0))
        line["cpu_baseline"] = {"value": r["bytes"] / r["seconds"] / 1e9, "unit": "GB/s",
                                "cores": 1, "kind": "oracle",
                                "sample": "oracle kv_block_swap, 512 pairs between two "
                                          "512-block bf16 pools, single-threaded, repeated "
                                          f"for {r['seconds']:.1f} s"}
    if world > 1:
        dist.destroy_process_group()
    return line


# ---------------------------------------------------------------------------
# multi-query (prefill) attention: packed new tokens per sequence
# ---------------------------------------------------------------------------
PREFILL_METRIC = "paged multi-query attention (prefill) TFLOP/s and KV GB/s"


def prefill_kernel(w) -> str:
    """The kernel the automatic prefill plan picks for workload w (mirrors
    the library's plan on a 152-SM GB300: up to 8 query rows per KV head ->
    the stream-K decode kernel; more -> tcgen05 (two query tiles per CTA
    above 128 rows, one below), unless 9 .. 64 rows come with fewer
    (sequence, KV head) pairs than SMs -> mma.sync)."""
    rows = int(w.news.max()) * (w.num_q_heads // w.num_kv_heads)
    if rows <= 8 and w.num_seqs <= 2048:
        return "attn_tc_kernel (stream-K decode kernel, query rows as score columns)"
    if w.scale > 0 and (rows > 64 or w.num_seqs * w.num_kv_heads >= 152):
        return ("attn_prefill_tc05x2_kernel" if rows > 128
                else "attn_prefill_tc05x2_kernel (one query tile per CTA)")
    return "attn_prefill_kernel (mma.sync)"


def prefill_flops(w) -> int:
    """Dense causal attention FLOPs: 4 * D per (query head, key) pair, each new
    token at position p seeing p + 1 keys."""
    tot = 0
    for P_, n in zip(w.prefix, w.news):
        # sum over i < n of (P_ + i + 1)
        tot += int(n) * int(P_) + int(n) * (int(n) + 1) // 2
    return 4 * w.head_dim * w.num_q_heads * tot


def _prefill_cpu_sample(name: str, seed: int, budget_s: float) -> dict:
    """The oracle on the first new tokens of the workload until budget_s."""
    import numpy as np
    import oracle
    from oracle import prefill as OP
    from paged_kv_cache_115_gb300 import workloads as wl
    w = wl.build_prefill(name, seed=seed)
    rng = np.random.default_rng(seed)
    D, H_q, H_kv, K = w.head_dim, w.num_q_heads, w.num_kv_heads, w.block_size
    flops, t0, done = 0, time.perf_counter(), 0
    s = 0
    L = int(w.context_lens[s])
    nb = -(-L // K)
    # a private pool with just this sequence's blocks, renumbered 0 .. nb-1
    kc = rng.standard_normal((nb, K, H_kv, D)).astype(np.float32)
    vc = rng.standard_normal((nb, K, H_kv, D)).astype(np.float32)
    bt = np.arange(nb, dtype=np.int64)[None, :]
    n_all = int(w.news[s])
    while time.perf_counter() - t0 < budget_s and done < n_all:
        # one new token at a time (its own causal row), the last ones first
        i = n_all - 1 - done
        q = rng.standard_normal((1, H_q, D)).astype(np.float32)
        pos = L - n_all + i
        OP.paged_attention_prefill(q, kc, vc, bt, [0, 1], [pos + 1], w.scale, "f32")
        flops += 4 * D * H_q * (pos + 1)
        done += 1
    sec = time.perf_counter() - t0
    return {"flops": flops, "seconds": sec, "tokens": done}


def run_prefill(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    from paged_kv_cache_115_gb300 import build, workloads as wl
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        dist.barrier()
    from paged_kv_cache_115_gb300 import ops

    w = wl.build_prefill(args.workload, seed=rank_seed(args.seed, rank))
    g = torch.Generator(device=dev)
    g.manual_seed(rank_seed(args.seed, rank))
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    T = w.num_tokens
    kc = torch.empty(shape, dtype=torch.bfloat16, device=dev).normal_(generator=g)
    vc = torch.empty(shape, dtype=torch.bfloat16, device=dev).normal_(generator=g)
    q = torch.empty((T, w.num_q_heads, w.head_dim), dtype=torch.bfloat16,
                    device=dev).normal_(generator=g)
    k_new = torch.empty((T, w.num_kv_heads, w.head_dim), dtype=torch.bfloat16,
                        device=dev).normal_(generator=g)
    v_new = torch.empty_like(k_new).normal_(generator=g)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cu = torch.from_numpy(w.cu_seqlens).to(dev)
    lens = torch.from_numpy(w.context_lens).to(dev)
    out = torch.empty_like(q)
    max_q, max_len = int(w.news.max()), int(w.context_lens.max())
    stream = torch.cuda.current_stream(dev)

    def append():
        ops.paged_kv_append_varlen(k_new, v_new, cu, lens, bt, kc, vc)

    ws_bytes = ops.prefill_workspace_bytes(w.num_seqs, T, max_q, max_len, w.num_q_heads,
                                           w.num_kv_heads, w.head_dim, w.block_size, w.scale,
                                           torch.bfloat16)
    workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    # append + attention (+ the merge of key-range partials when the kernel splits keys)
    launches_per_step = 2 + (1 if ws_bytes > 0 else 0)

    def attention():
        ops.paged_attention_prefill(q, kc, vc, bt, cu, lens, w.scale, max_q, max_len, out=out,
                                    workspace=workspace)

    for _ in range(max(args.warmup, 3)):
        append()
        attention()
    torch.cuda.synchronize(dev)
    assert ops.get_device_error(dev) == 0
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index) if rank == 0 else None
    time.sleep(0.2 if clocks else 0)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    start.record(stream)
    for i in range(K):
        append()
        ev[i][0].record(stream)
        attention()
        ev[i][1].record(stream)
    stop.record(stream)
    torch.cuda.synchronize(dev)
    clock_info = clocks.stop() if clocks else None
    total_ms = start.elapsed_time(stop)
    attn_ms = sum(a.elapsed_time(b) for a, b in ev) / K
    assert ops.get_device_error(dev) == 0

    # end to end through the public calls: every step copies its inputs (q,
    # the new K/V rows, tables, cu_seqlens, lengths) from one pinned host
    # buffer and reads its output back, on a second stream with two staged
    # buffer sets that overlap the neighbouring steps' compute
    base = {"q": q, "k": k_new, "v": v_new, "bt": bt, "cu": cu, "lens": lens}
    names = list(base)
    sets = []
    for _ in range(2):
        views = dict(base)
        dev_in, host_in = staged_inputs(views, names, dev)
        o = torch.empty_like(out)
        sets.append((dev_in, host_in, o, torch.empty(o.shape, dtype=o.dtype, pin_memory=True),
                     views))
    h2d = sets[0][1].numel()
    d2h = sets[0][3].numel() * sets[0][3].element_size()
    cs = torch.cuda.Stream(dev)

    def e2e_compute(b_):
        x = sets[b_][4]
        ops.paged_kv_append_varlen(x["k"], x["v"], x["cu"], x["lens"], x["bt"], kc, vc)
        ops.paged_attention_prefill(x["q"], kc, vc, x["bt"], x["cu"], x["lens"], w.scale, max_q,
                                    max_len, out=sets[b_][2], workspace=workspace)

    pipe_sets = [st[:4] for st in sets]
    run_pipelined(3, pipe_sets, e2e_compute, stream, cs)
    e2e_steps = max(4, min(K, 50))
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run_pipelined(e2e_steps, pipe_sets, e2e_compute, stream, cs, e0)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    # the same inputs in both sets: the outputs read back equal the timed step's
    ref_out = out.cpu()
    for st in sets:
        assert torch.equal(st[3].view(torch.int16), ref_out.view(torch.int16)), \
            "e2e output differs"

    total_ms, attn_ms, e2e_ms = max_over_ranks([total_ms, attn_ms, e2e_ms], dev)
    ms_step = total_ms / K
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None
    flops = prefill_flops(w)
    kv_bytes = int(w.context_lens.sum()) * w.num_kv_heads * w.head_dim * 2 * 2
    peaks, peak_src = read_peaks()
    tflops = flops / (attn_ms * 1e-3) / 1e12
    gbs = kv_bytes / (attn_ms * 1e-3) / 1e9
    tensor_bound = flops / kv_bytes > 400            # FLOP per byte vs ridge of ~280
    if tensor_bound:
        peak = float(peaks.get("bf16_tflops", 1900.0))
        roof = {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                "frac": tflops / peak,
                "peak_source": f"{peak_src} bf16_tflops (cuBLAS dense bf16, burst)"}
    else:
        peak = float(peaks["hbm_gbs"])
        roof = {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                "frac": gbs / peak, "peak_source": f"{peak_src} hbm_gbs (copy, read+write)"}
    traffic, traffic_src = traffic_record("prefill_traffic.json", w.name)
    roof.update({"kernel": prefill_kernel(w),
                 "algorithmic_flops_per_launch": flops,
                 "algorithmic_bytes_per_launch": kv_bytes, "avg_launch_ms": attn_ms,
                 "traffic": traffic["bytes_per_launch"] if traffic else None,
                 "traffic_source": traffic_src})
    value = world * (tflops if tensor_bound else gbs)
    cfg = {"workload": w.name, "num_seqs": w.num_seqs, "new_tokens": T,
           "new_tokens_per_seq": {"min": int(w.news.min()), "max": max_q},
           "cached_prefix": {"min": int(w.prefix.min()), "max": int(w.prefix.max()),
                             "mean": float(w.prefix.mean())},
           "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
           "head_dim": w.head_dim, "block_size": w.block_size, "num_blocks": w.num_blocks,
           "step": "paged_kv_append_varlen (slot mapping + KV write of the new tokens) + "
                   "paged_attention_prefill",
           "l2": f"{kv_bytes / 1e6:.0f} MB of KV per step vs 129 MB L2; no flush",
           "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}
    line = {
        "metric": PREFILL_METRIC, "value": value,
        "unit": "TFLOP/s" if tensor_bound else "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) q / new K,V / pool values; block tables from a "
                "seeded shuffled free list",
        "config": cfg, "attention_tflops": tflops, "attention_kv_GBps": gbs,
        "new_tokens_per_s": world * T / (ms_step * 1e-3),
        "roofline": roof,
        "e2e": {"value": world * (flops if tensor_bound else kv_bytes) / (e2e_ms * 1e-3) /
                (1e12 if tensor_bound else 1e9),
                "unit": "TFLOP/s" if tensor_bound else "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": "per step one pinned-host-to-device copy of the inputs and one "
                          "device-to-pinned-host copy of the output, on a second stream with "
                          "two staged buffer sets, overlapping the neighbouring steps"},
        "gpu_launches": launches_per_step * K,
        "clocks": clock_info,
    }
    if not args.no_cpu_baseline:
        env = dict(os.environ)
        for k_ in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            env[k_] = "1"
        env["CUDA_VISIBLE_DEVICES"] = ""
        code = ("import json,sys; sys.path.insert(0, %r); import bench; "
                "print(json.dumps(bench._prefill_cpu_sample(%r, %d, %f)))"
                % (ROOT, args.workload, args.seed, min(args.cpu_budget, 10.0)))
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                           cwd=ROOT, timeout=600)
        if r.returncode == 0:
            res = json.loads(r.stdout.strip().splitlines()[-1])
            # in the line's own unit (K/V bytes taken as the sample's share of FLOPs)
            cpu_v = (res["flops"] / res["seconds"] / 1e12 if tensor_bound else
                     res["flops"] / flops * kv_bytes / res["seconds"] / 1e9)
            line["cpu_baseline"] = {
                "value": cpu_v, "unit": "TFLOP/s" if tensor_bound else "GB/s", "cores": 1,
                "kind": "oracle",
                "sample": f"fp64 numpy oracle, single-threaded, {res['tokens']} of the first "
                          f"sequence's new tokens ({res['seconds']:.1f} s)"}
        else:
            line["cpu_baseline"] = {"value": None, "kind": "oracle", "error": r.stderr[-300:]}
    if world > 1:
        dist.destroy_process_group()
    return line


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle as it stands
# ---------------------------------------------------------------------------
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    from paged_kv_cache_115_gb300 import workloads as wl
    per_step = max(1.0, args.cpu_budget / max(1, args.steps))
    w = wl.build(args.workload, seed=args.seed) if args.op == "decode" else None
    if args.op == "prefill":
        fl, sec = 0, 0.0
        for _ in range(args.steps):
            r = _prefill_cpu_sample(args.workload, args.seed, per_step)
            fl += r["flops"]
            sec += r["seconds"]
        # the GPU arm's unit: TFLOP/s when the workload is tensor-bound, else
        # K/V GB/s, the sample's bytes taken as its share of the workload's FLOPs
        pw = wl.build_prefill(args.workload, seed=args.seed)
        total_flops = prefill_flops(pw)
        total_bytes = int(pw.context_lens.sum()) * pw.num_kv_heads * pw.head_dim * 2 * 2
        if total_flops / total_bytes > 400:
            value, unit = fl / sec / 1e12, "TFLOP/s"
        else:
            value, unit = fl / total_flops * total_bytes / sec / 1e9, "GB/s"
        return {
            "impl": "reference", "metric": PREFILL_METRIC, "value": value, "unit": unit,
            "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": args.workload},
            "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle",
                             "sample": "fp64 numpy oracle on the first sequence's last new "
                                       "tokens"},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0,
        }
    if args.op == "swap":
        _swap_cpu_sample(min(per_step, 1.0))
        moved, sec = 0, 0.0
        for _ in range(args.steps):
            r = _swap_cpu_sample(per_step)
            moved += r["bytes"]
            sec += r["seconds"]
        value = moved / sec / 1e9
        return {
            "impl": "reference", "metric": SWAP_METRIC, "value": value, "unit": "GB/s",
            "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bytes",
            "data": "synthetic", "config": {"workload": f"{args.workload} geometry, 512-pair "
                                                        "sample"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": "oracle kv_block_swap, 512 pairs between two 512-block "
                                       "bf16 pools"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0,
        }
    for _ in range(args.warmup):
        _cpu_sample(args.workload, args.seed, min(per_step, 1.0))
    tot_bytes, tot_s, seqs = 0, 0.0, 0
    for _ in range(args.steps):
        r = _cpu_sample(args.workload, args.seed, per_step)
        tot_bytes += r["bytes"]
        tot_s += r["seconds"]
        seqs += r["seqs"]
    value = tot_bytes / tot_s / 1e9
    cfg = workload_desc(w)
    sample = (f"fp64 numpy oracle on the first sequences of {args.workload}, about "
              f"{per_step:.0f} s of CPU work per step, {seqs} sequences in all")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_s / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same recipe as the GPU arm)", "config": cfg,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--kv-format", choices=["bf16", "fp8", "int8"], default="bf16",
                    help="KV pool storage: bf16, FP8 e4m3 (per-tensor scale) or INT8 "
                         "(per-token scale)")
    ap.add_argument("--block-size", type=int, default=0,
                    help="override the workload's block size (block-size sweep); 0 keeps it")
    ap.add_argument("--eager", action="store_true",
                    help="decode: time eager launches instead of CUDA-graph replays of the step")
    ap.add_argument("--graph", action="store_true",
                    help="decode: time CUDA-graph replays of the step (the default)")
    ap.add_argument("--op", choices=["decode", "swap", "prefill"], default="decode",
                    help="decode: the decode step (default); swap: block swap GPU <-> host; "
                         "prefill: multi-query attention (workloads suffix_prefill, "
                         "chunked_prefill, speculative_decode)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of CPU work for the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        # the oracle runs single-threaded: set before numpy / torch load
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[k] = "1"
    if args.warmup < 3 and args.impl == "gpu":
        args.warmup = 3
    if args.impl == "reference":
        line = run_reference(args)
    else:
        line = {"swap": run_swap, "prefill": run_prefill}.get(args.op, run_gpu)(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
