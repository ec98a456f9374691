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
DEFAULT_WORKLOAD = "mistral_7b"
# further decode workloads timed by the default run (same protocol, no e2e leg)
DEFAULT_ALSO = "llama31_70b"
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
def _host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:          # not Linux
        return os.cpu_count() or 1


def _cpu_items(name: str, seed: int):
    """The workload and its (sequence, KV head) work items, sequence-major."""
    from paged_kv_cache_115_gb300 import workloads as wl
    w = wl.build(name, seed=seed)
    items = [(s, j) for s in range(w.num_seqs) if int(w.context_lens[s]) > 0
             for j in range(w.num_kv_heads)]
    return w, items


def _cpu_worker(name: str, seed: int, items, budget_s: float, rounds: int, barrier,
                queue) -> None:
    """One process of the CPU baseline: prepares the inputs of its work items
    (untimed), then for each round waits for every other process and runs the
    oracle (slot mapping + KV write + attention) over its items until they
    are done or the budget has passed, reporting (round, bytes, start, end,
    items, tokens)."""
    import numpy as np
    import torch
    import oracle
    from paged_kv_cache_115_gb300 import accounting, workloads as wl

    torch.set_num_threads(1)
    full = wl.build(name, seed=seed)
    G = full.num_q_heads // full.num_kv_heads

    def st(x):
        x = x.contiguous()
        return x.view(torch.int16).numpy().view(np.uint16) if x.dtype == torch.bfloat16 \
            else x.numpy()

    prepared, cur = [], None
    for s, j in items:
        L = int(full.context_lens[s])
        if cur is None or cur[0] != s:
            sub = wl.build_decode("sample", [L], full.num_q_heads, full.num_kv_heads,
                                  full.head_dim, full.block_size, full.dtype, seed=seed + s)
            t = wl.materialize(sub, seed=seed + s, canary=False)
            cur = (s, sub, {k: st(t[k]) for k in ("q", "k_cache", "v_cache", "k_new", "v_new")})
            del t
        _, sub, a = cur
        # the head-j slice of the sequence's inputs (query heads j*G .. j*G+G-1)
        prepared.append((sub, L, np.ascontiguousarray(a["q"][:, j * G:(j + 1) * G]),
                         np.ascontiguousarray(a["k_cache"][:, :, j:j + 1]),
                         np.ascontiguousarray(a["v_cache"][:, :, j:j + 1]),
                         np.ascontiguousarray(a["k_new"][:, j:j + 1]),
                         np.ascontiguousarray(a["v_new"][:, j:j + 1])))
    cur = None
    for r in range(rounds):
        barrier.wait(timeout=900)
        t0 = time.monotonic()
        nbytes = ntok = n = 0
        for sub, L, q, kc, vc, kn, vn in prepared:
            slots = oracle.slot_mapping(sub.block_tables, sub.positions, sub.block_size)
            kc2, vc2 = oracle.kv_write(kc, vc, kn, vn, slots)
            oracle.paged_attention_decode(q, kc2, vc2, sub.block_tables, sub.context_lens,
                                          sub.scale, sub.dtype)
            nbytes += accounting.attention_kv_bytes([L], 1, full.head_dim, full.elem_bytes)
            ntok += L
            n += 1
            if time.monotonic() - t0 >= budget_s:
                break
        queue.put((r, nbytes, t0, time.monotonic(), n, ntok))


def _deal(items, procs: int, num_seqs: int):
    """Items per process: whole sequences (all their KV heads) dealt round
    robin when there are at least two sequences per process, else the
    (sequence, KV head) items themselves dealt round robin."""
    if num_seqs >= 2 * procs:
        by_seq = {}
        for it in items:
            by_seq.setdefault(it[0], []).append(it)
        seqs = sorted(by_seq)
        return [[it for s in seqs[i::procs] for it in by_seq[s]] for i in range(procs)]
    return [items[i::procs] for i in range(procs)]


def _cpu_parallel(name: str, seed: int, budget_s: float, procs: int, rounds: int = 1):
    """The oracle on `procs` spawned host processes, each on its share of the
    workload's (sequence, KV head) items; per round, throughput = all bytes /
    wall time from the common start to the last finish.  Returns the last
    round's result (with the list of all rounds under "rounds")."""
    import multiprocessing as mp
    import queue as _queue
    w, items = _cpu_items(name, seed)
    ctx = mp.get_context("spawn")
    procs = max(1, min(procs, len(items)))
    shares = _deal(items, procs, w.num_seqs)
    barrier, queue = ctx.Barrier(procs), ctx.Queue()
    ps = [ctx.Process(target=_cpu_worker,
                      args=(name, seed, shares[i], budget_s, rounds, barrier, queue))
          for i in range(procs)]
    for p_ in ps:
        p_.start()
    res, deadline = [], time.monotonic() + 900 + rounds * 20 * budget_s
    while len(res) < procs * rounds:
        try:
            res.append(queue.get(timeout=2))
        except _queue.Empty:
            dead = [p_.exitcode for p_ in ps if p_.exitcode not in (None, 0)]
            if dead or time.monotonic() > deadline:
                for p_ in ps:
                    if p_.is_alive():
                        p_.kill()
                raise RuntimeError(f"cpu baseline worker failed (exit codes {dead})")
    for p_ in ps:
        p_.join(timeout=60)
    out = []
    for r in range(rounds):
        rr = [x for x in res if x[0] == r]
        wall = max(x[3] for x in rr) - min(x[2] for x in rr)
        done = sum(x[4] for x in rr)
        out.append({"bytes": sum(x[1] for x in rr), "seconds": wall, "items": done,
                    "of_items": len(items), "tokens": sum(x[5] for x in rr), "procs": procs,
                    "seqs_per_s": done / w.num_kv_heads / wall})
    last = dict(out[-1])
    last["rounds"] = out
    return last


def _accuracy(check_path: str) -> dict:
    """Max-abs / max-rel error of the GPU outputs saved in `check_path`
    against the oracle run on the same inputs (taken before any library
    kernel ran): block copies, slot mapping, KV write, then attention, on the
    sampled sequences and KV heads."""
    import numpy as np
    import oracle
    z = np.load(check_path)
    fmt, dt = str(z["fmt"]), str(z["dtype"])
    bt, lens, pos, pairs = z["block_tables"], z["context_lens"], z["positions"], z["copy_pairs"]
    kc, vc, K = z["k_blocks"], z["v_blocks"], int(z["block_size"])
    if fmt == "bf16":          # plain pools (bf16 or f32)
        if len(pairs):
            kc, vc = oracle.kv_block_copy(kc, vc, pairs)
        slots = oracle.slot_mapping(bt, pos, K)
        kc, vc = oracle.kv_write(kc, vc, z["k_new"], z["v_new"], slots)
        ref = oracle.paged_attention_decode(z["q"], kc, vc, bt, lens, float(z["scale"]), dt)
    else:
        from oracle import quant as Q
        slots = oracle.slot_mapping(bt, pos, K)
        kf = oracle.decode(z["k_new"], "bf16").astype(np.float32)
        vf = oracle.decode(z["v_new"], "bf16").astype(np.float32)
        if fmt == "fp8":
            ks, vs = float(z["k_scale"]), float(z["v_scale"])
            kc, vc = Q.kv_write_fp8(kc, vc, kf, vf, slots, ks, vs)
            ref = Q.paged_attention_decode_quant(z["q"], kc, vc, bt, lens, float(z["scale"]),
                                                 "bf16", "fp8", k_scale=ks, v_scale=vs)
        elif fmt == "k16v8":
            vs = float(z["v_scale"])
            kc, vc = Q.kv_write_k16v8(kc, vc, kf, vf, slots, vs)
            ref = Q.paged_attention_decode_quant(z["q"], kc, vc, bt, lens, float(z["scale"]),
                                                 "bf16", "k16v8", v_scale=vs)
        else:
            kc, vc, kts, vts = Q.kv_write_int8(kc, vc, z["k_ts"], z["v_ts"], kf, vf, slots)
            ref = Q.paged_attention_decode_quant(z["q"], kc, vc, bt, lens, float(z["scale"]),
                                                 "bf16", "int8", k_tok_scales=kts,
                                                 v_tok_scales=vts)
    got = oracle.decode(z["out"], dt)
    err = np.abs(got - ref)
    tol = 2e-3 + 1e-2 * np.abs(ref) if dt == "bf16" else np.full_like(ref, 1e-5)
    return {"max_abs": float(err.max()), "max_rel": float((err / np.maximum(np.abs(ref), 1e-30)).max()),
            "elements": int(err.size), "within_tolerance": bool((err <= tol).all()),
            "tolerance": ("|gpu - oracle| <= 2e-3 + 1e-2 |oracle| element-wise" if dt == "bf16"
                          else "|gpu - oracle| <= 1e-5 element-wise"),
            "sample": str(z["sample"])}


def _cpu_job(name: str, seed: int, budget_s: float, check_paths: str = "") -> dict:
    """The CPU leg (CUDA hidden): the accuracy checks of the saved GPU outputs
    (`check_paths`: JSON object, workload name -> .npz path), then the oracle
    timed on one core and on every host core."""
    out = {}
    if check_paths:
        out["accuracy"] = {nm: _accuracy(pth) for nm, pth in json.loads(check_paths).items()}
    cores = _host_cores()
    out["one_core"] = _cpu_parallel(name, seed, min(budget_s / 3, 5.0), 1)
    out["all_cores"] = _cpu_parallel(name, seed, budget_s, cores)
    return out


def run_cpu_job(name: str, seed: int, budget_s: float, check_paths: str = "") -> dict:
    """Runs _cpu_job in a fresh interpreter with CUDA hidden (the oracle never
    shares a process with the GPU arm) and returns its result."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    code = ("import json,sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench._cpu_job(%r, %d, %f, %r)))"
            % (ROOT, name, seed, budget_s, check_paths))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       cwd=ROOT, timeout=max(900, budget_s * 30))
    if r.returncode != 0:
        raise RuntimeError("cpu leg failed: " + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline_line(name: str, res: dict) -> dict:
    """The bench line's cpu_baseline object from a _cpu_job result."""
    a, o = res["all_cores"], res["one_core"]
    gbs = a["bytes"] / a["seconds"] / 1e9
    return {
        "value": gbs, "unit": "GB/s", "cores": a["procs"], "kind": "oracle",
        "seconds": a["seconds"],
        "decode_tokens_per_s_per_layer": a["seqs_per_s"],
        "one_core": {"value": o["bytes"] / o["seconds"] / 1e9, "unit": "GB/s",
                     "seconds": o["seconds"], "items": o["items"]},
        "sample": (f"fp64 numpy oracle (slot mapping + KV write + attention) over {a['items']} "
                   f"of the {a['of_items']} (sequence, KV head) items of {name} "
                   f"({a['tokens']} cached tokens, {a['bytes'] / 1e6:.1f} MB of KV), "
                   f"{a['procs']} spawned processes, one thread each, items dealt round robin; "
                   f"time = wall clock from the common start to the last finish"),
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
def shares_blocks(w) -> bool:
    """Whether two sequences of the step read the same physical block."""
    seen = set()
    for s in range(w.num_seqs):
        n = -(-int(w.context_lens[s]) // w.block_size)
        row = set(int(b) for b in w.block_tables[s, :n])
        if seen & row:
            return True
        seen |= row
    return False


def _pick_samples(w, max_tokens: int = 40000):
    """Sequences for the accuracy check: the longest, the first, the last and
    the middle one, as many as fit in `max_tokens` cached tokens (at least
    one)."""
    import numpy as np
    S = w.num_seqs
    cand = [int(np.argmax(w.context_lens)), 0, S - 1, S // 2]
    picks, tok = [], 0
    for s in cand:
        L = int(w.context_lens[s])
        if s in picks or L <= 0:
            continue
        if picks and tok + L > max_tokens:
            continue
        picks.append(s)
        tok += L
    return picks


def _accuracy_snapshot(w, t, fmt: str, quant_scales) -> dict:
    """Inputs of the accuracy check, taken before any library kernel touches
    the pool: the blocks the sampled sequences read (and the sources of the
    copy-on-write pairs that write them), renumbered into a small pool, two of
    the KV heads, and the sampled rows of q and of the new tokens."""
    import numpy as np
    import torch
    samples = _pick_samples(w)
    K = w.block_size
    heads = sorted({0, w.num_kv_heads - 1})
    G = w.num_q_heads // w.num_kv_heads
    need = set()
    for s in samples:
        need.update(int(b) for b in w.block_tables[s, :-(-int(w.context_lens[s]) // K)])
    pairs = [tuple(int(x) for x in p) for p in w.copy_pairs]
    while True:
        more = {src for src, dst in pairs if dst in need and src not in need}
        if not more:
            break
        need |= more
    blocks = np.array(sorted(need), np.int64)
    remap = {int(b): i for i, b in enumerate(blocks)}
    maxb = max(-(-int(w.context_lens[s]) // K) for s in samples)
    bt = np.zeros((len(samples), maxb), np.int32)
    for i, s in enumerate(samples):
        n = -(-int(w.context_lens[s]) // K)
        bt[i, :n] = [remap[int(b)] for b in w.block_tables[s, :n]]
    sel = [(remap[src], remap[dst]) for src, dst in pairs if dst in need]
    idx = torch.from_numpy(blocks).to(t["k_cache"].device)
    hsel = torch.tensor(heads, device=idx.device)
    qh = torch.tensor([j * G + g for j in heads for g in range(G)], device=idx.device)
    sidx = torch.tensor(samples, device=idx.device)

    def host(x):
        x = x.contiguous().cpu()
        if x.dtype == torch.bfloat16:
            return x.view(torch.int16).numpy().view(np.uint16)
        return x.numpy()

    snap = {
        "fmt": np.array(fmt), "dtype": np.array(w.dtype), "block_size": np.array(K),
        "scale": np.array(w.scale),
        "k_blocks": host(t["k_cache"].index_select(0, idx).index_select(2, hsel)),
        "v_blocks": host(t["v_cache"].index_select(0, idx).index_select(2, hsel)),
        "block_tables": bt,
        "context_lens": w.context_lens[samples].astype(np.int32),
        "positions": w.positions[samples].astype(np.int32),
        "copy_pairs": np.array(sel, np.int64).reshape(-1, 2),
        "q": host(t["q"].index_select(0, sidx).index_select(1, qh)),
        "k_new": host(t["k_new"].index_select(0, sidx).index_select(1, hsel)),
        "v_new": host(t["v_new"].index_select(0, sidx).index_select(1, hsel)),
        "sample": np.array(f"sequences {samples} (of {w.num_seqs}), KV heads {heads} with their "
                           f"{G} query heads each, {len(blocks)} blocks"),
        "_samples": samples, "_qh": qh,
    }
    if fmt in ("fp8", "k16v8"):
        snap["k_scale"], snap["v_scale"] = np.array(quant_scales[0]), np.array(quant_scales[1])
    elif fmt == "int8":
        slot_idx = (idx[:, None] * K + torch.arange(K, device=idx.device)[None, :]).reshape(-1)
        snap["k_ts"] = host(t["k_ts"].index_select(0, slot_idx))
        snap["v_ts"] = host(t["v_ts"].index_select(0, slot_idx))
    return snap


def _save_snapshot(snap: dict, out) -> str:
    """Adds the GPU output rows to a snapshot and writes it to a temporary
    .npz file; returns its path."""
    import tempfile
    import numpy as np
    import torch
    sidx = torch.tensor(snap["_samples"], device=out.device)
    rows = out.index_select(0, sidx).index_select(1, snap["_qh"]).contiguous().cpu()
    data = {k: v for k, v in snap.items() if not k.startswith("_")}
    data["out"] = rows.view(torch.int16).numpy().view(np.uint16) \
        if rows.dtype == torch.bfloat16 else rows.numpy()
    fd, path = tempfile.mkstemp(suffix=".npz", prefix="pkv_check_")
    os.close(fd)
    np.savez(path, **data)
    return path


class DecodeCase:
    """One decode workload set up on the GPU: pools, step inputs staged in
    one device buffer with a pinned host twin, workspace, and the step's
    calls (block copy, fused slot mapping + KV write, attention)."""

    def __init__(self, args, name, dev, rank, snapshot: bool):
        import torch
        from paged_kv_cache_115_gb300 import accounting, ops, workloads as wl
        self.ops = ops
        self.fmt = fmt = args.kv_format
        self.dev = dev
        w = self.w = wl.build(name, seed=rank_seed(args.seed, rank),
                              block_size=args.block_size or None)
        t = self.t = wl.materialize(w, device=dev, seed=rank_seed(args.seed, rank),
                                    canary=False, values_device="cuda")
        self.out = torch.empty_like(t["q"])
        self.slots = torch.empty(w.num_seqs, dtype=torch.int64, device=dev)
        self.has_copy = len(w.copy_pairs) > 0
        self.max_len = max_len = w.max_context_len
        # shared-prefix groups: on when the tables share blocks (auto) or asked
        self.share = fmt == "bf16" and (args.share_prefix == "on" or
                                        (args.share_prefix == "auto" and shares_blocks(w)))
        scales = None
        if fmt == "bf16":
            self.qd = None
            self.kv_bytes = accounting.attention_kv_bytes(w.context_lens, w.num_kv_heads,
                                                          w.head_dim, w.elem_bytes)
            ws_bytes = ops.attention_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                                     w.head_dim, w.block_size, max_len,
                                                     t["q"].dtype, share_prefix=self.share)
        else:
            # one-byte pools of seeded random codes (finite e4m3 codes; int8
            # codes with per-slot scales); the bf16 pools are dropped
            g = torch.Generator(device=dev)
            g.manual_seed(rank_seed(args.seed, rank) + 7)
            shape = t["k_cache"].shape
            # k16v8: the bf16 K pool stays, only V becomes one-byte codes
            one_byte = ("v_cache",) if fmt == "k16v8" else ("k_cache", "v_cache")
            for nm in one_byte:
                del t[nm]
                c = torch.randint(0, 256, shape, generator=g, device=dev, dtype=torch.int32)
                c = torch.where((c & 0x7F) == 0x7F, c - 1, c).to(torch.uint8)
                t[nm] = c.view(torch.int8) if fmt == "int8" else c
            if fmt == "int8":
                n = shape[0] * shape[1]
                t["k_ts"] = torch.rand(n, generator=g, device=dev) * 0.02 + 0.001
                t["v_ts"] = torch.rand(n, generator=g, device=dev) * 0.02 + 0.001
                self.qd = ops.kv_quant("int8", k_token_scales=t["k_ts"],
                                       v_token_scales=t["v_ts"])
            elif fmt == "k16v8":
                scales = (1.0, 0.05)
                self.qd = ops.kv_quant("k16v8", v_scale=scales[1])
            else:
                scales = (0.05, 0.05)
                self.qd = ops.kv_quant("fp8", *scales)
            # K and V bytes per token row: 1 + 1, or 2 + 1 with the bf16 K pool
            self.kv_bytes = accounting.attention_kv_bytes(w.context_lens, w.num_kv_heads,
                                                          w.head_dim, 1)
            if fmt == "k16v8":
                self.kv_bytes = self.kv_bytes * 3 // 2
            if fmt == "int8":
                self.kv_bytes += int(w.context_lens.sum()) * 2 * 4   # a K and a V scale per token
            ws_bytes = ops.attention_quant_workspace_bytes(w.num_seqs, w.num_q_heads,
                                                           w.num_kv_heads, w.head_dim,
                                                           w.block_size, max_len, t["q"].dtype,
                                                           self.qd)
        # the accuracy check's inputs, before any library kernel runs
        self.snap = None
        if snapshot and not (fmt != "bf16" and self.has_copy):
            self.snap = _accuracy_snapshot(w, t, fmt, scales)
        self.workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
        self.names = ["q", "k_new", "v_new", "block_tables", "context_lens", "positions"]
        if self.has_copy:
            self.names.append("copy_pairs")
        # the step's inputs back to back in one device buffer with a pinned
        # host twin, so that the end-to-end leg moves them in one copy
        self.dev_stage, self.host_stage = staged_inputs(t, self.names, dev)
        attn_launches = ops.attention_launch_count(w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                                   w.head_dim, w.block_size, max_len,
                                                   t["q"].dtype, share_prefix=self.share)
        copy_launches = (2 if fmt in ("int8", "k16v8") else 1) if self.has_copy else 0
        self.launches_per_step = copy_launches + 1 + attn_launches
        pool_eb = pool_elem_bytes(fmt, w)
        n_new = int((w.positions >= 0).sum())
        self.row_fns = []
        if self.has_copy:
            self.row_fns.append(("kv_block_copy", self.copy_fn,
                                 int(accounting.block_copy_bytes(len(w.copy_pairs),
                                                                 w.block_size, w.num_kv_heads,
                                                                 w.head_dim, pool_eb))))
        self.row_fns.append(("paged_kv_append", self.append_fn,
                             int(n_new * w.num_kv_heads * w.head_dim * 2 *
                                 (w.elem_bytes + pool_eb))))
        self.row_fns.append(("paged_attention_decode", self.attention, self.kv_bytes))

    # ---- the step's calls (they read self.t / self.out when called) ----
    def attention(self):
        t, w, ops = self.t, self.w, self.ops
        if self.fmt == "bf16":
            ops.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                                       t["context_lens"], w.scale, out=self.out,
                                       max_context_len=self.max_len, workspace=self.workspace,
                                       share_prefix=self.share)
        else:
            ops.paged_attention_decode_quant(t["q"], t["k_cache"], t["v_cache"],
                                             t["block_tables"], t["context_lens"], w.scale,
                                             self.qd, out=self.out, max_context_len=self.max_len,
                                             workspace=self.workspace)

    def copy_fn(self):
        t, ops = self.t, self.ops
        if self.fmt == "bf16":
            ops.kv_block_copy(t["k_cache"], t["v_cache"], t["copy_pairs"])
        else:
            ops.kv_block_copy_quant(t["k_cache"], t["v_cache"], t["copy_pairs"], self.qd)

    def append_fn(self):
        # slot mapping + KV write of the new tokens in one fused launch
        t, ops = self.t, self.ops
        if self.fmt == "bf16":
            ops.paged_kv_append(t["k_new"], t["v_new"], t["block_tables"], t["positions"],
                                t["k_cache"], t["v_cache"], self.slots)
        else:
            ops.paged_kv_append_quant(t["k_new"], t["v_new"], t["block_tables"], t["positions"],
                                      t["k_cache"], t["v_cache"], self.qd, self.slots)

    def step(self):
        if self.has_copy:
            self.copy_fn()
        self.append_fn()
        self.attention()

    def release(self):
        self.t = self.out = self.workspace = self.dev_stage = self.host_stage = None


def _time_case(case, K: int, warmup: int, use_graph: bool, stream, world: int) -> dict:
    """Warm-up, then K timed steps (graph replays of the whole step, or eager
    launches) bracketed by events on the launching stream; then K replays of
    the attention call alone, each between events, for the per-launch
    roofline; then each row of the step alone with L2 flushed before it."""
    import torch
    import torch.distributed as dist
    dev, ops = case.dev, case.ops
    for _ in range(max(warmup, 3)):
        case.step()
    torch.cuda.synchronize(dev)
    assert ops.get_device_error(dev) == 0
    g_step = g_attn = cap = None
    if use_graph:
        # the whole step as one graph; the attention call alone as another
        # (capture needs a side stream; replays run on the timing stream)
        g_step, g_attn = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.graph(g_step, stream=cap):
            case.step()
        with torch.cuda.graph(g_attn, stream=cap):
            case.attention()
        stream.wait_stream(cap)
        torch.cuda.synchronize(dev)
        for _ in range(3):
            g_step.replay()
        torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    start.record(stream)
    for i in range(K):
        if use_graph:
            g_step.replay()
        else:
            if case.has_copy:
                case.copy_fn()
            case.append_fn()
            ev[i][0].record(stream)
            case.attention()
            ev[i][1].record(stream)
    stop.record(stream)
    torch.cuda.synchronize(dev)
    if use_graph:
        for i in range(K):
            ev[i][0].record(stream)
            g_attn.replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    total_ms = start.elapsed_time(stop)
    attn_avg_ms = sum(a.elapsed_time(b) for a, b in ev) / K
    assert ops.get_device_error(dev) == 0

    # each row of the step alone: events around the row only, L2 flushed (a
    # 256 MB write) before every timed launch.  The attention row is also
    # timed after the write plus a 256 MB read of another buffer, which
    # leaves L2 holding only clean lines: the write alone leaves up to the
    # whole L2 dirty, and writing those lines back shares DRAM with the
    # launch's first microseconds.
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    clean = torch.ones(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    rows = {}
    R = max(5, min(50, K))
    variants = [(nm, fn, nbytes, False) for nm, fn, nbytes in case.row_fns]
    variants += [(nm + "_clean_l2", fn, nbytes, True) for nm, fn, nbytes in case.row_fns
                 if nm == "paged_attention_decode"]
    for nm, fn, nbytes, read_after in variants:
        times = []
        for _ in range(R):
            flush.fill_(1)
            if read_after:
                clean.sum()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize(dev)
            times.append(a.elapsed_time(b))
        med = statistics.median(times)
        rows[nm] = {"median_us": med * 1e3, "min_us": min(times) * 1e3,
                    "algorithmic_bytes": nbytes, "GBps": nbytes / (med * 1e-3) / 1e9,
                    "frac": None,
                    "l2": ("flushed by a 256 MB write, then a 256 MB read of another buffer "
                           "before each launch (no dirty line left; eager, one launch each)"
                           if read_after else
                           "flushed before each launch (eager, one launch each)")}
    del flush, clean
    assert ops.get_device_error(dev) == 0
    return {"total_ms": total_ms, "attn_avg_ms": attn_avg_ms, "rows": rows,
            "g_step": g_step, "cap": cap}


def _e2e_case(case, timing: dict, K: int, use_graph: bool, stream, world: int) -> dict:
    """End to end through the public API with host buffers.  Every step
    copies its inputs from a pinned host buffer (one copy) and reads its
    output back (one copy).  The copies run on a second stream against two
    sets of staged inputs and outputs, so that step i+1's input copy and step
    i's output copy overlap the neighbouring steps' compute."""
    import torch
    import torch.distributed as dist
    dev, t, names = case.dev, case.t, case.names
    out0, views0 = case.out, {k: t[k] for k in names}
    t1 = dict(views0)
    dev_stage1, host_stage1 = staged_inputs(t1, names, dev)
    out1 = torch.empty_like(out0)
    sets = [(case.dev_stage, case.host_stage, views0, out0), (dev_stage1, host_stage1, t1, out1)]
    host_outs = [torch.empty(out0.shape, dtype=out0.dtype, pin_memory=True) for _ in range(2)]
    h2d = case.host_stage.numel()
    d2h = host_outs[0].numel() * host_outs[0].element_size()
    graphs = [timing["g_step"]] if use_graph else []
    if use_graph:
        # the same step over the second set (the calls read t and out when called)
        for k in names:
            t[k] = t1[k]
        case.out = out1
        g1 = torch.cuda.CUDAGraph()
        cap = timing["cap"]
        cap.wait_stream(stream)
        with torch.cuda.graph(g1, stream=cap):
            case.step()
        stream.wait_stream(cap)
        graphs.append(g1)
        for k in names:
            t[k] = views0[k]
        case.out = out0
        torch.cuda.synchronize(dev)
    cs = torch.cuda.Stream(dev)
    pipe_sets = [(sets[i][0], sets[i][1], sets[i][3], host_outs[i]) for i in range(2)]

    def e2e_compute(b):
        if use_graph:
            graphs[b].replay()
            return
        for k in names:
            t[k] = sets[b][2][k]
        case.out = sets[b][3]
        case.step()
        for k in names:
            t[k] = views0[k]
        case.out = out0

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
    return {"ms": e2e_ms, "h2d": h2d, "d2h": d2h}


def pool_elem_bytes(fmt: str, w) -> float:
    """Mean bytes per K / V element of the pools: the workload's dtype, one
    byte for FP8 / INT8, 1.5 for the bf16-K / FP8-V pair."""
    return {"bf16": w.elem_bytes, "k16v8": 1.5}.get(fmt, 1)


def unique_kv_bytes(w, pool_eb: float) -> int:
    """K and V bytes of the distinct token slots the step's sequences read
    (each physical slot once, however many tables point at its block)."""
    import numpy as np
    slots = []
    for s in range(w.num_seqs):
        L = int(w.context_lens[s])
        t = np.arange(L, dtype=np.int64)
        slots.append(w.block_tables[s][t // w.block_size].astype(np.int64) * w.block_size
                     + t % w.block_size)
    n = len(np.unique(np.concatenate(slots))) if slots else 0
    return int(n * w.num_kv_heads * w.head_dim * 2 * pool_eb)


def _roofline(case, attn_avg_ms: float, hbm: float, peak_src: str) -> dict:
    w = case.w
    achieved = case.kv_bytes / (attn_avg_ms * 1e-3) / 1e9
    traffic, traffic_src = traffic_record()
    if traffic and (traffic.get("workload") != w.name or traffic.get("kv_format") != case.fmt
                    or traffic.get("block_size") != w.block_size):
        traffic = None                  # the record is for another workload
        traffic_src = "the ncu record is for another workload, pool format or block size"
    extra = {}
    if shares_blocks(w):
        # the logical bytes count a shared block once per table that reads it;
        # DRAM need deliver each physical slot only once
        ub = unique_kv_bytes(w, pool_elem_bytes(case.fmt, w))
        extra = {"unique_bytes_per_launch": ub,
                 "unique_GBps": ub / (attn_avg_ms * 1e-3) / 1e9,
                 "unique_frac": ub / (attn_avg_ms * 1e-3) / 1e9 / hbm,
                 "note": "achieved counts logical bytes (each table's reads); shared blocks can "
                         "come from L2 or be staged once per group, so achieved may exceed the "
                         "DRAM peak; unique_* count each physical slot once"}
    return {
        **extra,
        "bound": "hbm",
        "kernel": ("pkv_attention_decode (share_prefix_kernel + attn_tc_kernel shared-prefix "
                   "groups + attn_reduce_kernel)" if case.share else
                   "pkv_attention_decode (attn_tc_kernel + attn_reduce_kernel)"),
        "achieved": achieved,
        "peak": hbm,
        "peak_source": f"{peak_src} hbm_gbs (copy, read+write)",
        "unit": "GB/s",
        "frac": achieved / hbm,
        "algorithmic_bytes_per_launch": case.kv_bytes,
        "avg_launch_ms": attn_avg_ms,
        "timing": "CUDA events around back-to-back graph replays of the attention call "
                  "on the launching stream (L2 warm from the previous replay only where the "
                  "KV fits in it)",
        "traffic": traffic["bytes_per_launch"] if traffic else None,
        "traffic_source": traffic_src,
    }


def run_gpu(args):
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

    from paged_kv_cache_115_gb300 import build
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        dist.barrier()
    from paged_kv_cache_115_gb300 import ops  # noqa: F401  (loads the library)

    check = rank == 0 and not args.no_cpu_baseline
    use_graph = not args.eager
    stream = torch.cuda.current_stream(dev)
    K = args.steps
    also = [n for n in (args.also.split(",") if args.also else []) if n and n != args.workload]

    case = DecodeCase(args, args.workload, dev, rank, snapshot=check)
    clocks = ClockSampler(dev.index) if rank == 0 else None
    time.sleep(0.2 if clocks else 0)
    tm = _time_case(case, K, args.warmup, use_graph, stream, world)
    e2e = _e2e_case(case, tm, K, use_graph, stream, world)
    checks = {}
    if case.snap is not None:
        checks[case.w.name] = _save_snapshot(case.snap, case.out)
    head = {"w": case.w, "kv_bytes": case.kv_bytes, "launches": case.launches_per_step,
            "fmt": case.fmt, "case": case}
    # further workloads, same protocol (no end-to-end leg)
    extra = []
    tm["g_step"] = tm["cap"] = None
    for nm in also:
        case.release()
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
        c2 = DecodeCase(args, nm, dev, rank, snapshot=check)
        tm2 = _time_case(c2, K, args.warmup, use_graph, stream, world)
        if c2.snap is not None:
            checks[c2.w.name] = _save_snapshot(c2.snap, c2.out)
        extra.append((c2, tm2))
        case = c2
    clock_info = clocks.stop() if clocks else None

    # ---- max over ranks
    vals = [tm["total_ms"], e2e["ms"], tm["attn_avg_ms"]]
    for _, t2 in extra:
        vals += [t2["total_ms"], t2["attn_avg_ms"]]
    vals = max_over_ranks(vals, dev)
    total_ms, e2e_ms, attn_avg_ms = vals[:3]
    w, kv_bytes = head["w"], head["kv_bytes"]
    ms_step = total_ms / K
    value = world * kv_bytes / (ms_step * 1e-3) / 1e9
    e2e_value = world * kv_bytes / (e2e_ms * 1e-3) / 1e9

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None

    peaks, peak_src = read_peaks()
    hbm = float(peaks["hbm_gbs"])
    for r in tm["rows"].values():
        r["frac"] = r["GBps"] / hbm
    cfg = workload_desc(w)
    cfg["share_prefix"] = head["case"].share
    cfg["l2"] = (f"inputs larger than L2: {kv_bytes / 1e6:.0f} MB of KV read per step "
                 f"vs 129 MB L2; no flush between steps")
    cfg["parallelism"] = f"replicas x{world}" if world > 1 else "single GPU"
    cfg["launch"] = "CUDA graph replay (one graph per step)" if use_graph else "eager launches"
    blocks_used = int(sum(-(-int(L) // w.block_size) for L in w.context_lens))
    pool_eb = pool_elem_bytes(head["fmt"], w)
    cfg["kv_reserved_bytes"] = int(blocks_used * w.block_size * w.num_kv_heads * w.head_dim * 2 *
                                   pool_eb)
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
        "dtype": w.dtype if head["fmt"] == "bf16" else f"{w.dtype} q / {head['fmt']} KV",
        "data": "synthetic: seeded N(0,1) q/k/v rounded to bf16; block tables from a seeded "
                "shuffled free list; lengths drawn per the workload recipe",
        "config": cfg,
        "hbm_frac": value / world / hbm,
        "decode_tokens_per_s_per_layer": world * w.num_seqs / (ms_step * 1e-3),
        "roofline": _roofline(head["case"], attn_avg_ms, hbm, peak_src),
        "e2e": {"value": e2e_value, "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "decode_tokens_per_s_per_layer": world * w.num_seqs / (e2e_ms * 1e-3),
                "copies": "per step one pinned-host-to-device copy of the inputs and one "
                          "device-to-pinned-host copy of the output, on a second stream with "
                          "two staged buffer sets, overlapping the neighbouring steps"},
        "rows": tm["rows"],
        "gpu_launches": head["launches"] * K,
        "clocks": clock_info,
    }
    workloads = {}
    for i, (c2, t2) in enumerate(extra):
        tot2, att2 = vals[3 + 2 * i], vals[4 + 2 * i]
        ms2 = tot2 / K
        for r in t2["rows"].values():
            r["frac"] = r["GBps"] / hbm
        workloads[c2.w.name] = {
            "value": world * c2.kv_bytes / (ms2 * 1e-3) / 1e9, "unit": "GB/s",
            "ms_per_step": ms2, "steps": K,
            "hbm_frac": c2.kv_bytes / (ms2 * 1e-3) / 1e9 / hbm,
            "decode_tokens_per_s_per_layer": world * c2.w.num_seqs / (ms2 * 1e-3),
            "config": dict(workload_desc(c2.w), share_prefix=c2.share),
            "roofline": _roofline(c2, att2, hbm, peak_src),
            "rows": t2["rows"],
            "gpu_launches": c2.launches_per_step * K,
        }
        line["gpu_launches"] += c2.launches_per_step * K
    if workloads:
        line["workloads"] = workloads
    if check:
        try:
            res = run_cpu_job(args.workload, args.seed, args.cpu_budget,
                              json.dumps(checks))
            line["cpu_baseline"] = cpu_baseline_line(args.workload, res)
            acc = res.get("accuracy", {})
            if w.name in acc:
                line["accuracy"] = acc[w.name]
            for nm, a in acc.items():
                if nm in workloads:
                    workloads[nm]["accuracy"] = a
        except Exception as e:  # report, do not hide the GPU number
            line["cpu_baseline"] = {"value": None, "error": str(e)[:300], "kind": "oracle"}
        finally:
            for pth in checks.values():
                try:
                    os.remove(pth)
                except OSError:
                    pass
    if world > 1:
        dist.destroy_process_group()
    return line


# ---------------------------------------------------------------------------
# block swap (GPU <-> pinned host): preempt half the batch and bring it back
# ---------------------------------------------------------------------------
SWAP_METRIC = "KV block swap GB/s (GPU pool <-> pinned host pool, out + in)"


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
    out_np, in_np = wl.swap_plan(w, rank_seed(args.seed, rank))
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
    # each step: the oracle on every host core over the workload's (sequence,
    # KV head) items, for about per_step seconds (the whole workload when it
    # finishes sooner); warm-up steps are short
    cores = _host_cores()
    r = _cpu_parallel(args.workload, args.seed, per_step, cores, rounds=args.warmup + args.steps)
    timed = r["rounds"][args.warmup:]
    tot_bytes = sum(x["bytes"] for x in timed)
    tot_s = sum(x["seconds"] for x in timed)
    items = sum(x["items"] for x in timed)
    procs = r["procs"]
    value = tot_bytes / tot_s / 1e9
    cfg = workload_desc(w)
    sample = (f"fp64 numpy oracle (slot mapping + KV write + attention) on {procs} spawned "
              f"processes over the (sequence, KV head) items of {args.workload}, up to about "
              f"{per_step:.0f} s per step, {items} items in all")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_s / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same recipe as the GPU arm)", "config": cfg,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": procs, "kind": "oracle",
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
    ap.add_argument("--also", default=DEFAULT_ALSO,
                    help="decode: comma-separated further workloads timed after the headline "
                         "one (same protocol, reported under \"workloads\"); '' for none")
    ap.add_argument("--kv-format", choices=["bf16", "fp8", "int8", "k16v8"], default="bf16",
                    help="KV pool storage: bf16, FP8 e4m3 (per-tensor scale), INT8 "
                         "(per-token scale), or k16v8 (bf16 K pool, FP8 V pool)")
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
    ap.add_argument("--share-prefix", choices=["auto", "on", "off"], default="auto",
                    help="decode: shared-prefix groups in the attention call (auto: on when "
                         "the step's block tables share blocks)")
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
