"""Pins of the quantized-KV oracle (oracle/quant.py) against the format
definitions and the pages' formulas, not against itself."""

import math

import numpy as np
import pytest

import oracle
from oracle import quant as Q


# --------------------------------------------------------------------------
# FP8 e4m3 ("学习大模型推理的显存优化", KV Cache 量化: 1 sign, 4 exponent,
# 3 mantissa bits, largest value 448)
# --------------------------------------------------------------------------

def test_e4m3_table_structure():
    v = Q.e4m3_values()
    nan = np.isnan(v)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    fin = v[~nan]
    assert np.nanmax(v) == 448.0 == Q.E4M3_MAX          # the page's range
    assert np.nanmin(v) == -448.0
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)                     # codes 0..0x7E increase
    assert len(set(fin.tolist())) == 253                # +0 and -0 compare equal
    # known points of the format
    assert v[0x38] == 1.0 and v[0x40] == 2.0 and v[0xC0] == -2.0
    assert v[0x01] == 2.0 ** -9 and v[0x08] == 2.0 ** -6 and v[0x07] == 7 * 2.0 ** -9
    assert v[0x7E] == 448.0 and v[0x7D] == 416.0
    assert v[0x80] == 0.0 and math.copysign(1, v[0x80]) == -1
    # negative codes mirror positive ones
    assert np.array_equal(v[0x80:0xFF], -v[0x00:0x7F])


def test_e4m3_relative_step():
    # 3 mantissa bits: between 1 and 2 the spacing is 1/8 (page: "about 1/8")
    v = Q.e4m3_values()
    ones = v[0x38:0x40]
    assert np.allclose(np.diff(np.append(ones, 2.0)), 0.125)


def test_e4m3_encode_round_trip_and_rounding():
    v = Q.e4m3_values()
    codes = np.array([c for c in range(256) if not np.isnan(v[c])], dtype=np.uint8)
    assert np.array_equal(Q.e4m3_encode(v[codes]), codes)     # exact values keep their code
    # midpoints between neighbours go to the even code (ties to even mantissa)
    pos = v[:0x7F]
    mids = (pos[:-1] + pos[1:]) / 2
    got = Q.e4m3_encode(mids)
    want = np.array([i if i % 2 == 0 else i + 1 for i in range(len(mids))], dtype=np.uint8)
    assert np.array_equal(got, want)
    # saturation: no infinities in e4m3
    assert list(Q.e4m3_encode(np.array([448.0, 460.0, 1e6, np.inf, -np.inf]))) == \
        [0x7E, 0x7E, 0x7E, 0x7E, 0xFE]
    # signed zero and values below half the smallest subnormal
    assert list(Q.e4m3_encode(np.array([0.0, -0.0, 2.0 ** -11, -2.0 ** -11]))) == \
        [0x00, 0x80, 0x00, 0x80]
    assert Q.e4m3_encode(np.array([np.nan]))[0] == 0x7F


def test_e4m3_encode_is_nearest_brute_force():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.uniform(-4, 3, 3000),
                        rng.uniform(-448, 448, 1000)])
    v = Q.e4m3_values()
    fin = v[~np.isnan(v)]
    got = Q.e4m3_decode(Q.e4m3_encode(x))
    best = np.min(np.abs(x[:, None] - fin[None, :]), axis=1)
    assert np.all(np.abs(x - got) <= best + 0.0)


# --------------------------------------------------------------------------
# INT8 per token ("19.2 KV Cache 系统化管理" §19.2.4:
# k_int8 = round(k / scale), scale = max|k| / 127)
# --------------------------------------------------------------------------

def test_int8_formula_examples():
    codes, s = Q.int8_token_quantize(np.array([127.0, 2.5, -3.5, 0.5, -1.5], np.float32))
    assert s == np.float32(1.0)
    assert codes.tolist() == [127, 2, -4, 0, -2]          # half to even
    m = np.float32(3.0)
    codes, s = Q.int8_token_quantize(np.array([m, m / 2, -m / 3, -m], np.float32))
    assert s == np.float32(m / np.float32(127))
    assert codes[0] == 127 and codes[3] == -127
    assert codes[1] == int(np.rint(np.float32(m / 2) / s))
    codes, s = Q.int8_token_quantize(np.zeros(8, np.float32))
    assert s == 0 and not codes.any()


def test_int8_error_bound_random():
    rng = np.random.default_rng(1)
    for _ in range(200):
        row = (rng.standard_normal(64) * 10.0 ** rng.uniform(-3, 3)).astype(np.float32)
        codes, s = Q.int8_token_quantize(row)
        assert np.abs(codes).max() == 127
        deq = Q.int8_decode(codes, s)
        # rounding to the grid: at most half a step (+ float32 division rounding)
        assert np.all(np.abs(deq - row) <= 0.5 * float(s) * (1 + 1e-5))


# --------------------------------------------------------------------------
# quantized write and attention
# --------------------------------------------------------------------------

def test_kv_write_fp8_and_int8_brute_force():
    rng = np.random.default_rng(2)
    nb, K, H, D, T = 5, 4, 2, 3, 6
    slots = rng.choice(nb * K, size=T, replace=False).astype(np.int64)
    slots[1] = -1
    k = (rng.standard_normal((T, H, D)) * 3).astype(np.float32)
    v = (rng.standard_normal((T, H, D)) * 3).astype(np.float32)
    kp = np.full((nb, K, H, D), 0x55, np.uint8)
    vp = np.full((nb, K, H, D), 0x66, np.uint8)
    ok, ov = Q.kv_write_fp8(kp, vp, k, v, slots, 0.5, 2.0)
    for i, s in enumerate(slots):
        b, o = divmod(int(s), K) if s >= 0 else (None, None)
        if s < 0:
            continue
        for h in range(H):
            for d in range(D):
                assert ok[b, o, h, d] == Q.e4m3_encode(np.array([k[i, h, d] / np.float32(0.5)]))[0]
                assert ov[b, o, h, d] == Q.e4m3_encode(np.array([v[i, h, d] / np.float32(2.0)]))[0]
    written = {int(s) for s in slots if s >= 0}
    for flat in range(nb * K):
        if flat not in written:
            assert np.all(ok.reshape(nb * K, H, D)[flat] == 0x55)
    ki = np.zeros((nb, K, H, D), np.int8)
    vi = np.zeros((nb, K, H, D), np.int8)
    kts = np.full(nb * K, -1.0, np.float32)
    vts = np.full(nb * K, -1.0, np.float32)
    ok, ov, okts, ovts = Q.kv_write_int8(ki, vi, kts, vts, k, v, slots)
    for i, s in enumerate(slots):
        if s < 0:
            continue
        c, sc = Q.int8_token_quantize(k[i])
        assert okts[s] == sc and np.array_equal(ok.reshape(nb * K, H, D)[s], c)
        c, sc = Q.int8_token_quantize(v[i])
        assert ovts[s] == sc and np.array_equal(ov.reshape(nb * K, H, D)[s], c)
    assert np.all(okts[[f for f in range(nb * K) if f not in written]] == -1.0)


def test_quant_attention_equals_plain_attention_on_grid_values():
    """When every cached value is exactly a code times its scale, attention
    over the quantized pool equals the plain oracle on those values."""
    rng = np.random.default_rng(3)
    S, H_q, H_kv, D, K = 3, 4, 2, 8, 4
    lens = [5, 9, 1]
    nb = sum(-(-L // K) for L in lens) + 2
    order = rng.permutation(nb)
    bt = np.full((S, 4), 10**6, np.int64)
    p = 0
    for s, L in enumerate(lens):
        for i in range(-(-L // K)):
            bt[s, i] = order[p]
            p += 1
    q = rng.standard_normal((S, H_q, D)).astype(np.float32)
    # fp8: codes drawn from the finite e4m3 codes, power-of-two scales
    v = Q.e4m3_values()
    finite = np.array([c for c in range(256) if not np.isnan(v[c]) and abs(v[c]) <= 8],
                      np.uint8)
    kc = rng.choice(finite, size=(nb, K, H_kv, D)).astype(np.uint8)
    vc = rng.choice(finite, size=(nb, K, H_kv, D)).astype(np.uint8)
    got = Q.paged_attention_decode_quant(q, kc, vc, bt, lens, 0.3, "f32", "fp8",
                                         k_scale=0.25, v_scale=2.0)
    ref = oracle.paged_attention_decode(q, (Q.e4m3_decode(kc) * 0.25).astype(np.float32),
                                        (Q.e4m3_decode(vc) * 2.0).astype(np.float32), bt, lens,
                                        0.3, "f32")
    assert np.abs(got - ref).max() < 1e-12
    # int8: per-slot power-of-two scales
    ki = rng.integers(-127, 128, size=(nb, K, H_kv, D)).astype(np.int8)
    vi = rng.integers(-127, 128, size=(nb, K, H_kv, D)).astype(np.int8)
    kts = (2.0 ** rng.integers(-9, -3, size=nb * K)).astype(np.float32)
    vts = (2.0 ** rng.integers(-9, -3, size=nb * K)).astype(np.float32)
    got = Q.paged_attention_decode_quant(q, ki, vi, bt, lens, 0.3, "f32", "int8",
                                         k_tok_scales=kts, v_tok_scales=vts)
    kd = (ki.astype(np.float64) * kts.reshape(nb, K)[:, :, None, None]).astype(np.float32)
    vd = (vi.astype(np.float64) * vts.reshape(nb, K)[:, :, None, None]).astype(np.float32)
    ref = oracle.paged_attention_decode(q, kd, vd, bt, lens, 0.3, "f32")
    assert np.abs(got - ref).max() < 1e-12


# --------------------------------------------------------------------------
# K at higher precision than V ("19.2 KV Cache 系统化管理" §19.2.4): bf16 K,
# FP8 e4m3 V
# --------------------------------------------------------------------------

def test_bf16_encode_matches_torch_cast():
    """Round to nearest even from float32 to bfloat16 is a library routine
    (torch's cast): the oracle's encoder agrees on specials, exact ties with
    even and odd kept bits, mantissa carries into the exponent, overflow to
    infinity and random values over the whole exponent range."""
    torch = pytest.importorskip("torch")
    specials = np.array([0.0, -0.0, 1.0, -2.5, np.inf, -np.inf, 3.3895314e38,
                         np.finfo(np.float32).max, np.finfo(np.float32).tiny, 1e-45],
                        np.float32)
    ties = np.array([0x3F808000, 0x3F818000, 0x3F80FFFF, 0x3F807FFF, 0x3FFF8000, 0x7F7F8000,
                     0x80008000, 0x00018000], np.uint32).view(np.float32)
    rng = np.random.default_rng(40)
    rnd = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    rnd = rnd[~np.isnan(rnd)]
    x = np.concatenate([specials, ties, rnd])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(Q.bf16_encode(x), want)
    # a NaN stays a NaN (sign kept, quiet bit set)
    n = Q.bf16_encode(np.array([np.nan], np.float32))[0]
    assert (n & 0x7F80) == 0x7F80 and (n & 0x007F) != 0


def test_bf16_encode_planted_truncation_fails():
    """Truncation instead of rounding disagrees with the cast on ties and
    above-half cases (the pin above would catch such a mistake)."""
    torch = pytest.importorskip("torch")
    x = np.array([0x3F80C000, 0x3F818000], np.uint32).view(np.float32)
    trunc = (x.view(np.uint32) >> 16).astype(np.uint16)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert not np.array_equal(trunc, want)
    assert np.array_equal(Q.bf16_encode(x), want)


def test_kv_write_k16v8_brute_force():
    rng = np.random.default_rng(41)
    nb, K, H, D, T = 5, 4, 2, 3, 6
    slots = rng.choice(nb * K, size=T, replace=False).astype(np.int64)
    slots[2] = -1
    k = (rng.standard_normal((T, H, D)) * 3).astype(np.float32)
    v = (rng.standard_normal((T, H, D)) * 3).astype(np.float32)
    kp = np.full((nb, K, H, D), 0x7FC1, np.uint16)      # NaN canaries
    vp = np.full((nb, K, H, D), 0x7F, np.uint8)
    ok, ov = Q.kv_write_k16v8(kp, vp, k, v, slots, 0.75)
    for i, s in enumerate(slots):
        if s < 0:
            continue
        b, o = divmod(int(s), K)
        for h in range(H):
            for d in range(D):
                assert ok[b, o, h, d] == Q.bf16_encode(np.array([k[i, h, d]]))[0]
                assert ov[b, o, h, d] == Q.e4m3_encode(np.array([v[i, h, d] / np.float32(0.75)]))[0]
    written = {int(s) for s in slots if s >= 0}
    for flat in range(nb * K):
        if flat not in written:
            assert np.all(ok.reshape(nb * K, H, D)[flat] == 0x7FC1)
            assert np.all(ov.reshape(nb * K, H, D)[flat] == 0x7F)


def test_k16v8_attention_equals_plain_attention():
    """K values exact in bf16 and V values exactly e4m3 codes times a power-of-
    two scale: attention over the pool pair equals the plain oracle on those
    values; a K pool read as FP8 (a format mix-up) does not."""
    rng = np.random.default_rng(42)
    S, H_q, H_kv, D, K = 3, 8, 2, 8, 4
    lens = [6, 11, 1]
    nb = sum(-(-L // K) for L in lens) + 2
    order = rng.permutation(nb)
    bt = np.full((S, 4), 10**6, np.int64)
    p = 0
    for s, L in enumerate(lens):
        for i in range(-(-L // K)):
            bt[s, i] = order[p]
            p += 1
    q = rng.standard_normal((S, H_q, D)).astype(np.float32)
    kbits = Q.bf16_encode(rng.standard_normal((nb, K, H_kv, D)).astype(np.float32))
    v = Q.e4m3_values()
    finite = np.array([c for c in range(256) if not np.isnan(v[c]) and abs(v[c]) <= 8],
                      np.uint8)
    vc = rng.choice(finite, size=(nb, K, H_kv, D)).astype(np.uint8)
    got = Q.paged_attention_decode_quant(q, kbits, vc, bt, lens, 0.3, "f32", "k16v8",
                                         v_scale=0.5)
    kf = (kbits.astype(np.uint32) << 16).view(np.float32)
    ref = oracle.paged_attention_decode(q, kf, (Q.e4m3_decode(vc) * 0.5).astype(np.float32),
                                        bt, lens, 0.3, "f32")
    assert np.abs(got - ref).max() < 1e-12
    wrong = Q.paged_attention_decode_quant(q, (kbits & 0xFF).astype(np.uint8), vc, bt, lens, 0.3,
                                           "f32", "fp8", k_scale=1.0, v_scale=0.5)
    assert not np.all(np.abs(wrong - ref) < 1e-3)
