"""Shared test utilities: storage views for the oracle and tolerances."""

import numpy as np
import torch

# bf16 outputs with fp32 accumulation: |gpu - ref| <= 2e-3 + 1e-2 * |ref|
BF16_ATOL, BF16_RTOL = 2e-3, 1e-2
# fp32 outputs: the pages' own paged-vs-dense bound
F32_ATOL = 1e-5


def storage(t: torch.Tensor) -> np.ndarray:
    """CPU numpy view of a tensor's raw storage: uint16 bits for bf16, uint32
    bits for fp32 (so that NaN canaries compare bit for bit)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32)
    return t.numpy()


def dtype_name(t: torch.Tensor) -> str:
    return {torch.bfloat16: "bf16", torch.float32: "f32"}[t.dtype]


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def check_attention(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    """Element-wise tolerance check; returns (max_abs, max_rel)."""
    err = np.abs(got - ref)
    max_abs = float(err.max()) if err.size else 0.0
    max_rel = float((err / np.maximum(np.abs(ref), 1e-30)).max()) if err.size else 0.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if dtype == "bf16":
        bad = err > BF16_ATOL + BF16_RTOL * np.abs(ref)
    else:
        bad = err > F32_ATOL
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance "
                             f"(max abs {max_abs:.3e}, max rel {max_rel:.3e}); first {idx.tolist()}")
    return max_abs, max_rel
