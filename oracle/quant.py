"""Quantized KV-cache formats for the oracle (fp64 / exact integer work).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``.

Two formats, from the pages:

* FP8 e4m3 with one scale per tensor ("学习大模型推理的显存优化", section
  KV Cache 量化: 1 sign, 4 exponent, 3 mantissa bits, largest value 448; the
  stored value is x / scale, read back as code * scale; the default scale is
  1.0).  Encoding rounds to the nearest representable value, ties to the
  even mantissa, and saturates to +-448 (no infinities in e4m3).
* INT8 with one scale per token ("19.2 KV Cache 系统化管理" §19.2.4:
  k_int8 = round(k / scale_k), scale_k = max(|k|) / 127; dequantize by
  multiplying the scale back).

Readings: the INT8 "token vector" is the token's whole row in this layer's
pool (all KV heads x head_dim); the scale and the division are float32
(IEEE, as the page's fp16 inputs are widened), rounding is half to even; an
all-zero row gets scale 0 and codes 0.

A third pool pair keeps K at higher precision than V ("19.2 KV Cache
系统化管理" §19.2.4: K is more sensitive to quantization than V, so it is
kept more precise): K in bfloat16, V in FP8 e4m3 with one scale per tensor.
Reading: "more precise" is the pool's 16-bit storage type (bf16), the V
format the FP8 one above; a K row given in float32 is rounded to bfloat16 to
nearest, ties to even.
"""

from __future__ import annotations

import numpy as np

__all__ = ["E4M3_MAX", "e4m3_values", "e4m3_decode", "e4m3_encode",
           "int8_token_quantize", "int8_decode", "bf16_encode", "kv_write_fp8",
           "kv_write_int8", "kv_write_k16v8", "dequantize_rows",
           "paged_attention_decode_quant"]

E4M3_MAX = 448.0


def e4m3_values() -> np.ndarray:
    """float64 value of every e4m3 code 0..255 (NaN for the two NaN codes).

    Exponent field e (bias 7) and mantissa field m: e = 0 gives subnormals
    (m / 8) * 2^-6; e >= 1 gives (1 + m / 8) * 2^(e - 7); e = 15, m = 7 is NaN.
    """
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        s = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            vals[code] = np.nan
        elif e == 0:
            vals[code] = s * (m / 8.0) * 2.0 ** -6
        else:
            vals[code] = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_VALS = e4m3_values()
_POS = _VALS[:0x7F]            # codes 0x00..0x7E, increasing, 0 .. 448


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    return _VALS[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Nearest e4m3 code (ties to even mantissa), saturating to +-448."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint8)
    flat = x.reshape(-1)
    o = out.reshape(-1)
    for i, v in enumerate(flat):
        if np.isnan(v):
            o[i] = 0x7F
            continue
        sign = 0x80 if np.signbit(v) else 0x00
        a = abs(v)
        if a >= E4M3_MAX:
            o[i] = sign | 0x7E
            continue
        j = int(np.searchsorted(_POS, a))          # _POS[j-1] < a <= _POS[j]
        if _POS[j] == a:
            o[i] = sign | j
            continue
        lo, hi = j - 1, j
        dlo, dhi = a - _POS[lo], _POS[hi] - a
        if dlo < dhi or (dlo == dhi and lo % 2 == 0):
            o[i] = sign | lo
        else:
            o[i] = sign | hi
    return out


def int8_token_quantize(row: np.ndarray):
    """One token's row (float32 values) -> (int8 codes, float32 scale)."""
    r = np.asarray(row, dtype=np.float32)
    amax = np.float32(np.max(np.abs(r))) if r.size else np.float32(0)
    if amax == 0:
        return np.zeros(r.shape, dtype=np.int8), np.float32(0)
    scale = np.float32(amax / np.float32(127))
    q = np.rint(r / scale)                          # float32 division, half to even
    q = np.clip(q, -127, 127)
    return q.astype(np.int8), scale


def int8_decode(codes: np.ndarray, scale) -> np.ndarray:
    return np.asarray(codes, dtype=np.int8).astype(np.float64) * float(scale)


def bf16_encode(x: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) of float32 values, rounded to nearest
    with ties to the even pattern.

    A bfloat16 number is the upper 16 bits of a binary32 one.  Rounding the
    32-bit pattern u to its upper half: add 0x7FFF plus the lowest kept bit
    (bit 16) and drop the low 16 bits; a carry out of the mantissa moves into
    the exponent, which is the next representable value (and the largest
    finite values round up to infinity).  NaNs keep their sign and upper
    payload with the quiet bit set.
    """
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    rounded = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) & 0xFFFF
    quiet = ((u >> 16) | 0x0040) & 0xFFFF
    return np.where(nan, quiet, rounded).astype(np.uint16)


# --------------------------------------------------------------------------
# quantized KV write and attention over a quantized pool
# --------------------------------------------------------------------------

def _flat(pool):
    nb, K = pool.shape[0], pool.shape[1]
    return pool.reshape(nb * K, *pool.shape[2:])


def kv_write_fp8(k_pool, v_pool, k_rows, v_rows, slots, k_scale, v_scale):
    """FP8 pools (uint8 codes [nb, K, H, D]) after storing token i's rows
    (float32 values [T, H, D]) at slots[i]: code = e4m3(float32(x / scale)).
    Slot -1 skips the token."""
    kp, vp = k_pool.copy(), v_pool.copy()
    kf, vf = _flat(kp), _flat(vp)
    ks, vs = np.float32(k_scale), np.float32(v_scale)
    for i, s in enumerate(np.asarray(slots)):
        if s < 0:
            continue
        kf[s] = e4m3_encode(np.asarray(k_rows[i], np.float32) / ks)
        vf[s] = e4m3_encode(np.asarray(v_rows[i], np.float32) / vs)
    return kp, vp


def kv_write_int8(k_pool, v_pool, k_tok_scales, v_tok_scales, k_rows, v_rows, slots):
    """INT8 pools (int8 codes [nb, K, H, D]) and per-slot scales (float32
    [nb * K]) after storing token i's rows at slots[i]."""
    kp, vp = k_pool.copy(), v_pool.copy()
    kts, vts = np.array(k_tok_scales, np.float32), np.array(v_tok_scales, np.float32)
    kf, vf = _flat(kp), _flat(vp)
    for i, s in enumerate(np.asarray(slots)):
        if s < 0:
            continue
        kf[s], kts[s] = int8_token_quantize(k_rows[i])
        vf[s], vts[s] = int8_token_quantize(v_rows[i])
    return kp, vp, kts, vts


def kv_write_k16v8(k_pool, v_pool, k_rows, v_rows, slots, v_scale):
    """K pool (bfloat16 bit patterns, uint16 [nb, K, H, D]) and V pool (e4m3
    codes, uint8) after storing token i's rows (float32 values [T, H, D]) at
    slots[i]: K = bfloat16(x) to nearest even, V = e4m3(float32(x / v_scale)).
    Slot -1 skips the token."""
    kp, vp = k_pool.copy(), v_pool.copy()
    kf, vf = _flat(kp), _flat(vp)
    vs = np.float32(v_scale)
    for i, s in enumerate(np.asarray(slots)):
        if s < 0:
            continue
        kf[s] = bf16_encode(np.asarray(k_rows[i], np.float32))
        vf[s] = e4m3_encode(np.asarray(v_rows[i], np.float32) / vs)
    return kp, vp


def dequantize_rows(pool, rows_slot, kv_head, fmt, tensor_scale=None, tok_scales=None):
    """float64 values of pool rows (flattened slots ``rows_slot``) for one KV
    head: ``fmt`` "fp8", "int8", or "bf16" (bit patterns, exact)."""
    flat = _flat(pool)
    codes = flat[np.asarray(rows_slot, np.int64), kv_head, :]
    if fmt == "bf16":
        bits = np.asarray(codes).view(np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    if fmt == "fp8":
        return e4m3_decode(codes) * float(np.float32(tensor_scale))
    if fmt == "int8":
        sc = np.asarray(tok_scales, np.float32)[np.asarray(rows_slot, np.int64)].astype(np.float64)
        return codes.astype(np.float64) * sc[:, None]
    raise ValueError(fmt)


def paged_attention_decode_quant(q, k_pool, v_pool, block_tables, context_lens, scale, q_dtype,
                                 fmt, k_scale=1.0, v_scale=1.0, k_tok_scales=None,
                                 v_tok_scales=None):
    """Decode attention over a quantized pool: gather through the block table,
    dequantize (code * scale, exactly in float64), then the dense definition
    of "KV Cache：长上下文为什么吃显存" §01 with GQA head h -> h // G.
    ``fmt`` "fp8", "int8", or "k16v8" (K pool bfloat16, V pool e4m3 with
    ``v_scale``)."""
    from .paged_attention import decode, dense_attention
    S, H_q, D = q.shape
    H_kv, K = k_pool.shape[2], k_pool.shape[1]
    G = H_q // H_kv
    q64 = decode(q, q_dtype)
    out = np.zeros((S, H_q, D))
    for s in range(S):
        L = int(context_lens[s])
        t = np.arange(L, dtype=np.int64)
        slots = np.asarray(block_tables[s], np.int64)[t // K] * K + t % K
        for j in range(H_kv):
            kf, vf = ("bf16", "fp8") if fmt == "k16v8" else (fmt, fmt)
            Kj = dequantize_rows(k_pool, slots, j, kf, k_scale, k_tok_scales)
            Vj = dequantize_rows(v_pool, slots, j, vf, v_scale, v_tok_scales)
            for h in range(j * G, (j + 1) * G):
                out[s, h] = dense_attention(q64[s, h], Kj, Vj, scale)
    return out
