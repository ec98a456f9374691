"""Thin torch-facing binding of libpagedkv (include/pagedkv.h).

Argument marshalling only: every function checks devices / dtypes / shapes,
passes raw device pointers and the current CUDA stream to the C ABI, and
raises if the library reports an error.  All compute runs in the library's
CUDA kernels; there is no CPU path.  Importing this module loads the shared
library and raises ImportError when it has not been built.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

_LIB_PATH = _build.LIB_PATH

if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"libpagedkv is not built ({_LIB_PATH} missing); run "
        "`python -c 'import __graft_entry__ as g; g.build()'` on a machine with nvcc")

_lib = ctypes.CDLL(_LIB_PATH)

PKV_OK = 0
PKV_ERR_INVALID_ARGUMENT = 1
PKV_ERR_DEVICE_CHECK = 5
PKV_F32, PKV_BF16 = 0, 1

DEVICE_ERRORS = {
    0: "none", 1: "block id out of range", 2: "slot out of range", 3: "copy pair out of range",
    4: "context length out of range", 5: "position beyond block-table row", 6: "pipeline timeout",
}

c_i32, c_i64, c_vp, c_sz, c_f = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_float


class AttentionConfig(ctypes.Structure):
    _fields_ = [("kernel", c_i32), ("num_splits", c_i32), ("share_prefix", c_i32),
                ("reserved", c_i32 * 5)]


class KvQuant(ctypes.Structure):
    """pkv_kv_quant: format 1 = FP8 e4m3 (per-tensor scales), 2 = INT8 per token."""
    _fields_ = [("format", c_i32), ("k_scale", c_f), ("v_scale", c_f),
                ("k_token_scales", c_vp), ("v_token_scales", c_vp)]


KV_FP8_E4M3, KV_INT8_TOKEN, KV_BF16K_FP8V = 1, 2, 3


def _sig(name, restype, *argtypes):
    f = getattr(_lib, name)
    f.restype = restype
    f.argtypes = list(argtypes)
    return f


_status_string = _sig("pkv_status_string", ctypes.c_char_p, c_i32)
_last_msg = _sig("pkv_last_error_message", ctypes.c_char_p)
_version = _sig("pkv_version", c_i32)
_slot_mapping = _sig("pkv_slot_mapping", c_i32, c_vp, c_i32, c_vp, c_i32, c_i32, c_i64, c_vp, c_vp)
_kv_write = _sig("pkv_kv_write", c_i32, c_vp, c_vp, c_vp, c_i64, c_vp, c_vp, c_i64, c_i32, c_i32,
                 c_i32, c_i32, c_vp)
_kv_append = _sig("pkv_kv_append", c_i32, c_vp, c_vp, c_vp, c_i32, c_vp, c_i32, c_vp, c_vp, c_i64,
                  c_i32, c_i32, c_i32, c_i32, c_vp, c_vp)
_selftest_timeout = _sig("pkv_selftest_wait_timeout", c_i32, c_i64, c_vp)
_block_copy = _sig("pkv_kv_block_copy", c_i32, c_vp, c_vp, c_vp, c_i64, c_i64, c_i32, c_i32, c_i32,
                   c_i32, c_vp)
_block_swap = _sig("pkv_kv_block_swap", c_i32, c_vp, c_vp, c_i64, c_vp, c_vp, c_i64, c_i64, c_vp,
                   c_i64, c_vp)
_prefill = _sig("pkv_attention_prefill", c_i32, c_vp, c_vp, c_vp, c_vp, c_i32, c_vp, c_vp, c_i32,
                c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_i64, c_f, c_vp, c_vp, c_sz,
                c_i32, ctypes.POINTER(AttentionConfig), c_vp)
_prefill_ws = _sig("pkv_attention_prefill_workspace_bytes", c_i32, c_i32, c_i32, c_i32, c_i32,
                   c_i32, c_i32, c_i32, c_i32, c_f, c_i32, ctypes.POINTER(AttentionConfig),
                   ctypes.POINTER(c_sz))
_append_varlen = _sig("pkv_kv_append_varlen", c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, c_i32,
                      c_i32, c_vp, c_vp, c_i64, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp)
_ws_bytes = _sig("pkv_attention_workspace_bytes", c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_i32,
                 c_i32, ctypes.POINTER(AttentionConfig), ctypes.POINTER(c_sz))
_launch_count = _sig("pkv_attention_launch_count", c_i32, c_i32, c_i32, c_i32, c_i32, c_i32,
                     c_i32, c_i32, ctypes.POINTER(AttentionConfig), ctypes.POINTER(c_i32))
_attention = _sig("pkv_attention_decode", c_i32, c_vp, c_vp, c_vp, c_vp, c_i32, c_vp, c_i32, c_i32,
                  c_i32, c_i32, c_i32, c_i32, c_i64, c_f, c_vp, c_vp, c_sz, c_i32,
                  ctypes.POINTER(AttentionConfig), c_vp)
_attention_noalloc = _sig("pkv_attention_decode_noalloc", c_i32, c_vp, c_vp, c_vp, c_vp, c_i32,
                          c_vp, c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_i64, c_f, c_vp, c_i32,
                          ctypes.POINTER(AttentionConfig), c_vp)
_append_quant = _sig("pkv_kv_append_quant", c_i32, c_vp, c_vp, c_vp, c_i32, c_vp, c_i32, c_vp,
                     c_vp, c_i64, c_i32, c_i32, c_i32, c_i32, ctypes.POINTER(KvQuant), c_vp,
                     c_vp)
_copy_quant = _sig("pkv_kv_block_copy_quant", c_i32, c_vp, c_vp, c_vp, c_i64, c_i64, c_i32, c_i32,
                   c_i32, ctypes.POINTER(KvQuant), c_vp)
_ws_quant = _sig("pkv_attention_quant_workspace_bytes", c_i32, c_i32, c_i32, c_i32, c_i32, c_i32,
                 c_i32, c_i32, ctypes.POINTER(KvQuant), ctypes.POINTER(AttentionConfig),
                 ctypes.POINTER(c_sz))
_attention_quant = _sig("pkv_attention_decode_quant", c_i32, c_vp, c_vp, c_vp, c_vp, c_i32, c_vp,
                        c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_i64, c_f, c_vp, c_vp, c_sz,
                        c_i32, ctypes.POINTER(KvQuant), ctypes.POINTER(AttentionConfig), c_vp)
_dev_error = _sig("pkv_get_device_error", c_i32, ctypes.POINTER(c_i32), c_vp)

# bytes of the library's fixed attention scratch (PKV_NOALLOC_SCRATCH_BYTES)
NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024

EXPORTED = ("pkv_status_string", "pkv_last_error_message", "pkv_version", "pkv_slot_mapping",
            "pkv_kv_write", "pkv_kv_append", "pkv_kv_block_copy", "pkv_kv_block_swap",
            "pkv_selftest_wait_timeout", "pkv_attention_workspace_bytes",
            "pkv_attention_launch_count", "pkv_attention_decode",
            "pkv_attention_decode_noalloc", "pkv_kv_append_quant", "pkv_kv_block_copy_quant",
            "pkv_attention_quant_workspace_bytes", "pkv_attention_decode_quant",
            "pkv_attention_prefill", "pkv_attention_prefill_workspace_bytes",
            "pkv_kv_append_varlen", "pkv_get_device_error")


class PagedKVError(RuntimeError):
    pass


def _check(status: int, what: str) -> None:
    if status != PKV_OK:
        raise PagedKVError(f"{what}: {_status_string(status).decode()} "
                           f"({_last_msg().decode()})")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return PKV_BF16
    if t.dtype == torch.float32:
        return PKV_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream(device: torch.device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t: torch.Tensor, name: str, dtype=None, dim=None) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dims, got {t.dim()}")


def _ptr(t: torch.Tensor) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr())


def _device_call(fn):
    """Runs a binding with the device of its CUDA tensor arguments current
    (the library launches on the current device and picks per-device state
    from it), after checking that all of them live on that one device."""
    import functools

    @functools.wraps(fn)
    def wrapper(*args, **kwargs):
        devs = {a.device for a in list(args) + list(kwargs.values())
                if isinstance(a, torch.Tensor) and a.is_cuda}
        if len(devs) > 1:
            raise ValueError(f"{fn.__name__}: CUDA tensors on several devices {sorted(map(str, devs))}")
        if not devs:
            return fn(*args, **kwargs)
        with torch.cuda.device(devs.pop()):
            return fn(*args, **kwargs)
    return wrapper


def version() -> int:
    return int(_version())


@_device_call
def slot_mapping(block_tables: torch.Tensor, positions: torch.Tensor, block_size: int,
                 num_blocks: int, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """int64 slot of each sequence's token at ``positions`` (-1 for padding)."""
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(positions, "positions", torch.int32, 1)
    S = positions.shape[0]
    if out is None:
        out = torch.empty(S, dtype=torch.int64, device=positions.device)
    _need(out, "out", torch.int64, 1)
    _check(_slot_mapping(_ptr(block_tables), block_tables.shape[1], _ptr(positions), S,
                         block_size, num_blocks, _ptr(out), _stream(positions.device)),
           "pkv_slot_mapping")
    return out


@_device_call
def paged_kv_write(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                   k_cache: torch.Tensor, v_cache: torch.Tensor) -> None:
    """k_cache.view(-1, H_kv, D)[slot_mapping[i]] = k[i] (same for v), in place."""
    _need(k_cache, "k_cache", None, 4)
    _need(v_cache, "v_cache", k_cache.dtype, 4)
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    nb, K, H, D = k_cache.shape
    _need(k, "k", k_cache.dtype, 3)
    _need(v, "v", k_cache.dtype, 3)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    T = k.shape[0]
    if tuple(k.shape) != (T, H, D) or tuple(v.shape) != (T, H, D) or slot_mapping.shape[0] != T:
        raise ValueError("k/v/slot_mapping shapes do not match the pool")
    _check(_kv_write(_ptr(k), _ptr(v), _ptr(slot_mapping), T, _ptr(k_cache), _ptr(v_cache), nb, K,
                     H, D, _dtype_code(k_cache), _stream(k_cache.device)), "pkv_kv_write")


@_device_call
def paged_kv_append(k: torch.Tensor, v: torch.Tensor, block_tables: torch.Tensor,
                    positions: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                    slot_mapping_out: Optional[torch.Tensor] = None) -> None:
    """Slot mapping and KV write in one launch: token i (block-table row i) goes
    to the slot of ``positions[i]``; optionally stores the slots."""
    _need(k_cache, "k_cache", None, 4)
    _need(v_cache, "v_cache", k_cache.dtype, 4)
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    nb, K, H, D = k_cache.shape
    _need(k, "k", k_cache.dtype, 3)
    _need(v, "v", k_cache.dtype, 3)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(positions, "positions", torch.int32, 1)
    T = k.shape[0]
    if tuple(k.shape) != (T, H, D) or tuple(v.shape) != (T, H, D) or positions.shape[0] != T \
            or block_tables.shape[0] != T:
        raise ValueError("k/v/positions/block_tables shapes do not match")
    sp = None
    if slot_mapping_out is not None:
        _need(slot_mapping_out, "slot_mapping_out", torch.int64, 1)
        sp = _ptr(slot_mapping_out)
    _check(_kv_append(_ptr(k), _ptr(v), _ptr(block_tables), block_tables.shape[1],
                      _ptr(positions), T, _ptr(k_cache), _ptr(v_cache), nb, K, H, D,
                      _dtype_code(k_cache), sp, _stream(k_cache.device)), "pkv_kv_append")


def selftest_wait_timeout(limit_cycles: int, device=None) -> None:
    """Run the bounded-wait self test (records device error 6 when it gives up)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    _check(_selftest_timeout(int(limit_cycles), _stream(dev)), "pkv_selftest_wait_timeout")


@_device_call
def kv_block_copy(k_cache: torch.Tensor, v_cache: torch.Tensor,
                  src_dst_pairs: torch.Tensor) -> None:
    """Copy-on-write block copy: block dst <- block src for each row of pairs."""
    _need(k_cache, "k_cache", None, 4)
    _need(v_cache, "v_cache", k_cache.dtype, 4)
    _need(src_dst_pairs, "src_dst_pairs", torch.int64, 2)
    nb, K, H, D = k_cache.shape
    _check(_block_copy(_ptr(k_cache), _ptr(v_cache), _ptr(src_dst_pairs), src_dst_pairs.shape[0],
                       nb, K, H, D, _dtype_code(k_cache), _stream(k_cache.device)),
           "pkv_kv_block_copy")


def _need_swap_side(t: torch.Tensor, name: str) -> None:
    if t.is_cuda:
        _need(t, name)
    elif t.device.type == "cpu" and t.is_pinned():
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    else:
        raise ValueError(f"{name} must be a CUDA tensor or a pinned CPU tensor")


def kv_block_swap(src_k: torch.Tensor, src_v: Optional[torch.Tensor], dst_k: torch.Tensor,
                  dst_v: Optional[torch.Tensor], src_dst_pairs: torch.Tensor) -> None:
    """Block swap between pools that may live in different memories:
    ``dst[pairs[i][1]] = src[pairs[i][0]]`` for K and V (V may be None on
    both sides).  Each pool is a CUDA tensor or a pinned CPU tensor whose
    first axis counts blocks (a KV pool ``[nb, K, H_kv, D]`` in any format, or
    an INT8 pool's slot scales viewed as ``[nb, K]``); the pairs are int64
    ``[n, 2]`` on the GPU or pinned.  One launch on the current stream; the
    caller keeps pinned buffers alive until the stream passes the copy."""
    if (src_v is None) != (dst_v is None):
        raise ValueError("src_v and dst_v must both be given or both be None")
    sides = [(src_k, "src_k"), (dst_k, "dst_k")]
    if src_v is not None:
        sides += [(src_v, "src_v"), (dst_v, "dst_v")]
    for t, name in sides:
        _need_swap_side(t, name)
        if t.dtype != src_k.dtype or tuple(t.shape[1:]) != tuple(src_k.shape[1:]):
            raise ValueError(f"{name}: every pool needs src_k's dtype and block shape")
    if src_v is not None and (src_v.shape[0] != src_k.shape[0] or dst_v.shape[0] != dst_k.shape[0]):
        raise ValueError("K and V pools of one side must have the same number of blocks")
    _need_swap_side(src_dst_pairs, "src_dst_pairs")
    if src_dst_pairs.dtype != torch.int64 or src_dst_pairs.dim() != 2 or \
            src_dst_pairs.shape[1] != 2:
        raise ValueError("src_dst_pairs must be int64 [n, 2]")
    block_bytes = src_k[0].numel() * src_k.element_size() if src_k.shape[0] else 0
    cuda = [t.device for t, _ in sides if t.is_cuda]
    dev = cuda[0] if cuda else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        _check(_block_swap(_ptr(src_k), _ptr(src_v) if src_v is not None else None,
                           src_k.shape[0], _ptr(dst_k),
                           _ptr(dst_v) if dst_v is not None else None, dst_k.shape[0],
                           block_bytes, _ptr(src_dst_pairs), src_dst_pairs.shape[0],
                           _stream(dev)), "pkv_kv_block_swap")


def _cfg(kernel: int, num_splits: int, share_prefix: bool = False) -> AttentionConfig:
    c = AttentionConfig()
    c.kernel = kernel
    c.num_splits = num_splits
    c.share_prefix = 1 if share_prefix else 0
    return c


def attention_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                              max_context_len, dtype: torch.dtype, kernel: int = 0,
                              num_splits: int = 0, share_prefix: bool = False) -> int:
    out = c_sz(0)
    cfg = _cfg(kernel, num_splits, share_prefix)
    code = PKV_BF16 if dtype == torch.bfloat16 else PKV_F32
    _check(_ws_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                     code, ctypes.byref(cfg), ctypes.byref(out)), "pkv_attention_workspace_bytes")
    return int(out.value)


def attention_launch_count(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                           max_context_len, dtype: torch.dtype, kernel: int = 0,
                           num_splits: int = 0, share_prefix: bool = False) -> int:
    """Kernel launches one paged_attention_decode call makes for these sizes."""
    out = c_i32(0)
    cfg = _cfg(kernel, num_splits, share_prefix)
    code = PKV_BF16 if dtype == torch.bfloat16 else PKV_F32
    _check(_launch_count(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                         max_context_len, code, ctypes.byref(cfg), ctypes.byref(out)),
           "pkv_attention_launch_count")
    return int(out.value)


@_device_call
def paged_attention_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                           out: Optional[torch.Tensor] = None,
                           max_context_len: Optional[int] = None,
                           workspace: Optional[torch.Tensor] = None,
                           kernel: int = 0, num_splits: int = 0,
                           share_prefix: bool = False) -> torch.Tensor:
    """Decode attention over the paged cache (GQA, split-K).

    ``max_context_len`` is a host-side bound on ``context_lens``; when omitted
    it is read from the device (one synchronising copy).  ``workspace`` is a
    uint8 CUDA tensor of at least :func:`attention_workspace_bytes` bytes
    (for the same ``kernel``, ``num_splits`` and ``share_prefix``); when
    omitted one is allocated with torch.  ``share_prefix``: stage blocks that
    consecutive sequences share once per group (see pkv_attention_config).
    """
    _need(q, "q", None, 3)
    _need(k_cache, "k_cache", q.dtype, 4)
    _need(v_cache, "v_cache", q.dtype, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    S, H_q, D = q.shape
    nb, K, H_kv, D2 = k_cache.shape
    if D2 != D or v_cache.shape != k_cache.shape or context_lens.shape[0] != S \
            or block_tables.shape[0] != S:
        raise ValueError("shape mismatch between q, caches, tables and lengths")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", q.dtype, 3)
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if S else 0
    need = attention_workspace_bytes(S, H_q, H_kv, D, K, max_context_len, q.dtype, kernel,
                                     num_splits, share_prefix)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", torch.uint8, 1)
    cfg = _cfg(kernel, num_splits, share_prefix)
    _check(_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                      block_tables.shape[1], _ptr(context_lens), max_context_len, S, H_q, H_kv, D,
                      K, nb, float(scale), _ptr(out), _ptr(workspace), workspace.numel(),
                      _dtype_code(q), ctypes.byref(cfg), _stream(q.device)),
           "pkv_attention_decode")
    return out


@_device_call
def paged_attention_decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor,
                                   v_cache: torch.Tensor, block_tables: torch.Tensor,
                                   context_lens: torch.Tensor, scale: float,
                                   out: torch.Tensor, max_context_len: int,
                                   kernel: int = 0, num_splits: int = 0) -> torch.Tensor:
    """Same result as :func:`paged_attention_decode`, for callers that cannot
    allocate device memory at this point (an engine whose KV pool took the free
    HBM, or a decode path that must stay out of the CUDA allocator).  The
    split-K scratch is the library's fixed in-module array, so ``out`` must be
    given, ``max_context_len`` must be a host value, and nothing here (torch
    included) allocates.  Sizes needing more than NOALLOC_SCRATCH_BYTES of
    scratch raise.  Calls that overlap on the GPU share that scratch and race.
    """
    _need(q, "q", None, 3)
    _need(k_cache, "k_cache", q.dtype, 4)
    _need(v_cache, "v_cache", q.dtype, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    _need(out, "out", q.dtype, 3)
    S, H_q, D = q.shape
    nb, K, H_kv, D2 = k_cache.shape
    if D2 != D or v_cache.shape != k_cache.shape or context_lens.shape[0] != S \
            or block_tables.shape[0] != S or out.shape != q.shape:
        raise ValueError("shape mismatch between q, caches, tables, lengths and out")
    cfg = _cfg(kernel, num_splits)
    _check(_attention_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                              block_tables.shape[1], _ptr(context_lens), int(max_context_len), S,
                              H_q, H_kv, D, K, nb, float(scale), _ptr(out), _dtype_code(q),
                              ctypes.byref(cfg), _stream(q.device)),
           "pkv_attention_decode_noalloc")
    return out


def get_device_error(device=None) -> int:
    """Synchronise, read and clear the library's device error word (0 = none)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    code = c_i32(0)
    st = _dev_error(ctypes.byref(code), _stream(dev))
    if st not in (PKV_OK, PKV_ERR_DEVICE_CHECK):
        _check(st, "pkv_get_device_error")
    return int(code.value)


# ---------------------------------------------------------------------------
# quantized KV cache (FP8 e4m3 per-tensor scale, INT8 per-token scale)
# ---------------------------------------------------------------------------

def kv_quant(fmt: str, k_scale: float = 1.0, v_scale: float = 1.0,
             k_token_scales: Optional[torch.Tensor] = None,
             v_token_scales: Optional[torch.Tensor] = None) -> KvQuant:
    """Describe a quantized pool: ``fmt`` "fp8" (scales per tensor), "int8"
    (float32 CUDA tensors of one scale per token slot) or "k16v8" (a bf16 K
    pool with an FP8 V pool of scale ``v_scale``).  The description holds
    references to the scale tensors, so that their memory lives as long as
    it does."""
    qd = KvQuant()
    qd.fmt = fmt
    if fmt == "fp8":
        qd.format, qd.k_scale, qd.v_scale = KV_FP8_E4M3, float(k_scale), float(v_scale)
    elif fmt == "k16v8":
        qd.format, qd.k_scale, qd.v_scale = KV_BF16K_FP8V, 1.0, float(v_scale)
    elif fmt == "int8":
        for name, t in (("k_token_scales", k_token_scales), ("v_token_scales", v_token_scales)):
            if t is None:
                raise ValueError(f"int8 pools need {name}")
            _need(t, name, torch.float32, 1)
        qd.format = KV_INT8_TOKEN
        qd.k_token_scales = k_token_scales.data_ptr()
        qd.v_token_scales = v_token_scales.data_ptr()
        qd._scale_tensors = (k_token_scales, v_token_scales)
    else:
        raise ValueError(f"unknown quantized format {fmt!r}")
    return qd


def _need_pool(t: torch.Tensor, name: str, quant: Optional[KvQuant] = None) -> None:
    _need(t, name, None, 4)
    if quant is not None and quant.format == KV_BF16K_FP8V and name == "k_cache":
        if t.dtype != torch.bfloat16:
            raise TypeError("k_cache of a k16v8 pool pair must be bfloat16")
        return
    if t.dtype not in (torch.uint8, torch.int8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        raise TypeError(f"{name} must hold one-byte codes (uint8 / int8 / float8_e4m3fn)")


@_device_call
def paged_kv_append_quant(k: torch.Tensor, v: torch.Tensor, block_tables: torch.Tensor,
                          positions: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                          quant: KvQuant,
                          slot_mapping_out: Optional[torch.Tensor] = None) -> None:
    """Slot mapping + quantized KV write in one launch (rows k, v in bf16/fp32)."""
    _need_pool(k_cache, "k_cache", quant)
    _need_pool(v_cache, "v_cache")
    nb, K, H, D = k_cache.shape
    _need(k, "k", None, 3)
    _need(v, "v", k.dtype, 3)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(positions, "positions", torch.int32, 1)
    T = k.shape[0]
    if tuple(k.shape) != (T, H, D) or tuple(v.shape) != (T, H, D) or positions.shape[0] != T \
            or block_tables.shape[0] != T or v_cache.shape != k_cache.shape:
        raise ValueError("k/v/positions/block_tables/pool shapes do not match")
    sp = None
    if slot_mapping_out is not None:
        _need(slot_mapping_out, "slot_mapping_out", torch.int64, 1)
        sp = _ptr(slot_mapping_out)
    _check(_append_quant(_ptr(k), _ptr(v), _ptr(block_tables), block_tables.shape[1],
                         _ptr(positions), T, _ptr(k_cache), _ptr(v_cache), nb, K, H, D,
                         _dtype_code(k), ctypes.byref(quant), sp, _stream(k_cache.device)),
           "pkv_kv_append_quant")


@_device_call
def kv_block_copy_quant(k_cache: torch.Tensor, v_cache: torch.Tensor,
                        src_dst_pairs: torch.Tensor, quant: KvQuant) -> None:
    """Copy-on-write block copy of a quantized pool (codes and, for INT8, scales)."""
    _need_pool(k_cache, "k_cache", quant)
    _need_pool(v_cache, "v_cache")
    _need(src_dst_pairs, "src_dst_pairs", torch.int64, 2)
    nb, K, H, D = k_cache.shape
    _check(_copy_quant(_ptr(k_cache), _ptr(v_cache), _ptr(src_dst_pairs), src_dst_pairs.shape[0],
                       nb, K, H, D, ctypes.byref(quant), _stream(k_cache.device)),
           "pkv_kv_block_copy_quant")


def attention_quant_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                    max_context_len, q_dtype: torch.dtype, quant: KvQuant,
                                    kernel: int = 0, num_splits: int = 0) -> int:
    out = c_sz(0)
    cfg = _cfg(kernel, num_splits)
    code = PKV_BF16 if q_dtype == torch.bfloat16 else PKV_F32
    _check(_ws_quant(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                     code, ctypes.byref(quant), ctypes.byref(cfg), ctypes.byref(out)),
           "pkv_attention_quant_workspace_bytes")
    return int(out.value)


@_device_call
def paged_attention_decode_quant(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                 block_tables: torch.Tensor, context_lens: torch.Tensor,
                                 scale: float, quant: KvQuant,
                                 out: Optional[torch.Tensor] = None,
                                 max_context_len: Optional[int] = None,
                                 workspace: Optional[torch.Tensor] = None,
                                 kernel: int = 0, num_splits: int = 0) -> torch.Tensor:
    """Decode attention over a quantized pool (values read back as code * scale)."""
    _need(q, "q", None, 3)
    _need_pool(k_cache, "k_cache", quant)
    _need_pool(v_cache, "v_cache")
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    S, H_q, D = q.shape
    nb, K, H_kv, D2 = k_cache.shape
    if D2 != D or v_cache.shape != k_cache.shape or context_lens.shape[0] != S \
            or block_tables.shape[0] != S:
        raise ValueError("shape mismatch between q, caches, tables and lengths")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", q.dtype, 3)
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if S else 0
    need = attention_quant_workspace_bytes(S, H_q, H_kv, D, K, max_context_len, q.dtype, quant,
                                           kernel, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", torch.uint8, 1)
    cfg = _cfg(kernel, num_splits)
    _check(_attention_quant(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                            block_tables.shape[1], _ptr(context_lens), max_context_len, S, H_q,
                            H_kv, D, K, nb, float(scale), _ptr(out), _ptr(workspace),
                            workspace.numel(), _dtype_code(q), ctypes.byref(quant),
                            ctypes.byref(cfg), _stream(q.device)),
           "pkv_attention_decode_quant")
    return out


# ---------------------------------------------------------------------------
# multi-query (prefill) attention over the paged cache
# ---------------------------------------------------------------------------

@_device_call
def paged_kv_append_varlen(k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor,
                           context_lens: torch.Tensor, block_tables: torch.Tensor,
                           k_cache: torch.Tensor, v_cache: torch.Tensor,
                           slot_mapping_out: Optional[torch.Tensor] = None) -> None:
    """Store the packed new tokens (k, v: [T, H_kv, D]) of every sequence at
    their positions context_lens[s] - n_s + i (slot mapping + write, one
    launch)."""
    _need(k_cache, "k_cache", None, 4)
    _need(v_cache, "v_cache", k_cache.dtype, 4)
    nb, K, H, D = k_cache.shape
    _need(k, "k", k_cache.dtype, 3)
    _need(v, "v", k_cache.dtype, 3)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    _need(context_lens, "context_lens", torch.int32, 1)
    _need(block_tables, "block_tables", torch.int32, 2)
    T, S = k.shape[0], context_lens.shape[0]
    if tuple(k.shape) != (T, H, D) or tuple(v.shape) != (T, H, D) or \
            cu_seqlens.shape[0] != S + 1 or block_tables.shape[0] != S or \
            v_cache.shape != k_cache.shape:
        raise ValueError("inconsistent shapes")
    sm = None
    if slot_mapping_out is not None:
        _need(slot_mapping_out, "slot_mapping_out", torch.int64, 1)
        sm = _ptr(slot_mapping_out)
    _check(_append_varlen(_ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(context_lens),
                          _ptr(block_tables), block_tables.shape[1], S, T, _ptr(k_cache),
                          _ptr(v_cache), nb, K, H, D, _dtype_code(k_cache), sm,
                          _stream(k.device)), "pkv_kv_append_varlen")


@_device_call
def paged_attention_prefill(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_tables: torch.Tensor, cu_seqlens: torch.Tensor,
                            context_lens: torch.Tensor, scale: float, max_query_len: int,
                            max_context_len: int, out: Optional[torch.Tensor] = None,
                            kernel: int = 0, num_splits: int = 0,
                            workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Multi-query paged attention: packed queries q [T, H_q, D] of several new
    tokens per sequence (cu_seqlens int32 [S+1]); token i of n at position
    context_lens[s] - n + i attends to positions 0 .. itself.  The host bounds
    max_query_len / max_context_len size the launch.  ``kernel``: 0 automatic,
    1 tcgen05 tiles of 128 query rows, 2 mma.sync tiles, 3 the stream-K decode
    kernel (at most 8 query rows per KV head); ``num_splits``: key
    ranges per row tile (mma.sync), 0 automatic.  ``workspace``: uint8 CUDA
    tensor of :func:`prefill_workspace_bytes` bytes (allocated when None)."""
    _need(q, "q", None, 3)
    _need(k_cache, "k_cache", q.dtype, 4)
    _need(v_cache, "v_cache", q.dtype, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    _need(context_lens, "context_lens", torch.int32, 1)
    T, H_q, D = q.shape
    nb, K, H_kv, D2 = k_cache.shape
    S = context_lens.shape[0]
    if D2 != D or v_cache.shape != k_cache.shape or cu_seqlens.shape[0] != S + 1 or \
            block_tables.shape[0] != S:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", q.dtype, 3)
    if tuple(out.shape) != tuple(q.shape):
        raise ValueError("out must have q's shape")
    cfg = _cfg(kernel, num_splits)
    need = prefill_workspace_bytes(S, T, max_query_len, max_context_len, H_q, H_kv, D, K,
                                   scale, q.dtype, kernel, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", torch.uint8, 1)
    _check(_prefill(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                    block_tables.shape[1], _ptr(cu_seqlens), _ptr(context_lens), S, T,
                    int(max_query_len), int(max_context_len), H_q, H_kv, D, K, nb, float(scale),
                    _ptr(out), _ptr(workspace), workspace.numel(), _dtype_code(q),
                    ctypes.byref(cfg), _stream(q.device)), "pkv_attention_prefill")
    return out


def prefill_workspace_bytes(num_seqs, num_tokens, max_query_len, max_context_len, num_q_heads,
                            num_kv_heads, head_dim, block_size, scale, dtype: torch.dtype,
                            kernel: int = 0, num_splits: int = 0) -> int:
    out = c_sz(0)
    code = PKV_BF16 if dtype == torch.bfloat16 else PKV_F32
    _check(_prefill_ws(num_seqs, num_tokens, int(max_query_len), int(max_context_len),
                       num_q_heads, num_kv_heads, head_dim, block_size, float(scale), code,
                       ctypes.byref(_cfg(kernel, num_splits)), ctypes.byref(out)),
           "pkv_attention_prefill_workspace_bytes")
    return int(out.value)
