"""GPU parity of the quantized KV cache (FP8 e4m3 per-tensor scale, INT8 per
token, and the pair that keeps K in bf16 with V in FP8) against the oracle:
quantized writes and copies bit-exact (codes, bf16 patterns and scales),
attention within the tolerance of the plain path."""

import numpy as np
import pytest
import torch

from oracle import quant as Q
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


def f32_rows(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().float().numpy()


def identity_tables(T, K, nb, rng):
    """One token per row, each token in its own (shuffled) block at offset
    t % K: row i holds position i % K in block perm[i]."""
    perm = rng.permutation(nb)[:T]
    bt = perm.reshape(T, 1).astype(np.int32)
    pos = (np.arange(T) % K).astype(np.int32)
    return bt, pos


@pytest.mark.parametrize("scale", [1.0, 0.37, 3.0])
def test_fp8_append_every_bf16_value(ops, scale):
    # every finite bf16 bit pattern, as K rows; V rows the same values reversed
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    bits = bits[np.isfinite(vals)]
    n = (len(bits) // 256) * 256
    H, D = 2, 128
    T = n // (H * D)
    kb = torch.from_numpy(bits[:n].view(np.int16).reshape(T, H, D).copy()).view(torch.bfloat16)
    vb = torch.from_numpy(bits[:n][::-1].view(np.int16).reshape(T, H, D).copy()).view(torch.bfloat16)
    K, nb = 4, T + 3
    rng = np.random.default_rng(0)
    bt, pos = identity_tables(T, K, nb, rng)
    kc = torch.full((nb, K, H, D), 0x7F, dtype=torch.uint8)
    vc = torch.full((nb, K, H, D), 0x7F, dtype=torch.uint8)
    dkc, dvc = kc.to(DEV), vc.to(DEV)
    qd = ops.kv_quant("fp8", scale, scale * 2)
    slots = torch.empty(T, dtype=torch.int64, device=DEV)
    ops.paged_kv_append_quant(kb.to(DEV), vb.to(DEV), torch.from_numpy(bt).to(DEV),
                              torch.from_numpy(pos).to(DEV), dkc, dvc, qd, slots)
    assert ops.get_device_error() == 0
    oslots = oracle.slot_mapping(bt, pos, K)
    assert np.array_equal(slots.cpu().numpy(), oslots)
    ek, ev = Q.kv_write_fp8(kc.numpy(), vc.numpy(), f32_rows(kb), f32_rows(vb), oslots,
                            scale, scale * 2)
    assert np.array_equal(dkc.cpu().numpy(), ek)
    assert np.array_equal(dvc.cpu().numpy(), ev)


@pytest.mark.parametrize("in_dtype", [torch.bfloat16, torch.float32])
def test_int8_append_bit_exact(ops, in_dtype):
    rng = np.random.default_rng(1)
    T, H, D, K, nb = 200, 8, 128, 16, 230
    mags = 10.0 ** rng.uniform(-4, 4, size=(T, 1, 1))
    k = torch.from_numpy((rng.standard_normal((T, H, D)) * mags).astype(np.float32)).to(in_dtype)
    v = torch.from_numpy((rng.standard_normal((T, H, D)) * mags).astype(np.float32)).to(in_dtype)
    k[3] = 0.0                                   # all-zero row: scale 0, codes 0
    v[7, 2, 5] = 1e4                             # one outlier dominates its row
    bt, pos = identity_tables(T, K, nb, rng)
    pos[5] = -1                                  # padding token
    kc = torch.full((nb, K, H, D), 99, dtype=torch.int8)
    vc = torch.full((nb, K, H, D), 99, dtype=torch.int8)
    kts = torch.full((nb * K,), -5.0)
    vts = torch.full((nb * K,), -5.0)
    d = [x.to(DEV) for x in (kc, vc, kts, vts)]
    qd = ops.kv_quant("int8", k_token_scales=d[2], v_token_scales=d[3])
    ops.paged_kv_append_quant(k.to(DEV), v.to(DEV), torch.from_numpy(bt).to(DEV),
                              torch.from_numpy(pos).to(DEV), d[0], d[1], qd)
    assert ops.get_device_error() == 0
    oslots = oracle.slot_mapping(bt, pos, K)
    ek, ev, ekt, evt = Q.kv_write_int8(kc.numpy(), vc.numpy(), kts.numpy(), vts.numpy(),
                                       f32_rows(k), f32_rows(v), oslots)
    assert np.array_equal(d[0].cpu().numpy(), ek) and np.array_equal(d[1].cpu().numpy(), ev)
    assert np.array_equal(d[2].cpu().numpy().view(np.uint32), ekt.view(np.uint32))
    assert np.array_equal(d[3].cpu().numpy().view(np.uint32), evt.view(np.uint32))


@pytest.mark.parametrize("fmt", ["fp8", "int8", "k16v8"])
def test_quant_block_copy(ops, fmt):
    rng = np.random.default_rng(2)
    nb, K, H, D = 12, 16, 8, 128
    if fmt == "k16v8":        # bf16 K pool (2 bytes per element), one-byte V pool
        kc = torch.from_numpy(rng.integers(0, 2**16, size=(nb, K, H, D), dtype=np.uint16)
                              .view(np.int16)).view(torch.bfloat16)
        vc = torch.from_numpy(rng.integers(0, 256, size=(nb, K, H, D), dtype=np.uint8))
        pairs = np.array([[0, 5], [3, 9], [11, 2]], dtype=np.int64)
        dk, dv = kc.to(DEV), vc.to(DEV)
        ops.kv_block_copy_quant(dk, dv, torch.from_numpy(pairs).to(DEV), ops.kv_quant("k16v8"))
        assert ops.get_device_error() == 0
        ek, ev = oracle.kv_block_copy(storage(kc), vc.numpy(), pairs)
        assert np.array_equal(storage(dk), ek) and np.array_equal(dv.cpu().numpy(), ev)
        return
    kc = torch.from_numpy(rng.integers(0, 256, size=(nb, K, H, D), dtype=np.uint8))
    vc = torch.from_numpy(rng.integers(0, 256, size=(nb, K, H, D), dtype=np.uint8))
    kts = torch.from_numpy(rng.standard_normal(nb * K).astype(np.float32))
    vts = torch.from_numpy(rng.standard_normal(nb * K).astype(np.float32))
    pairs = np.array([[0, 5], [3, 9], [11, 2]], dtype=np.int64)
    d = [x.to(DEV) for x in (kc, vc, kts, vts)]
    qd = ops.kv_quant(fmt, 1.0, 1.0, d[2], d[3]) if fmt == "int8" else ops.kv_quant(fmt)
    ops.kv_block_copy_quant(d[0], d[1], torch.from_numpy(pairs).to(DEV), qd)
    assert ops.get_device_error() == 0
    ek, ev = oracle.kv_block_copy(kc.numpy(), vc.numpy(), pairs)
    assert np.array_equal(d[0].cpu().numpy(), ek) and np.array_equal(d[1].cpu().numpy(), ev)
    if fmt == "int8":
        ekt, evt = oracle.kv_block_copy(kts.numpy().reshape(nb, K), vts.numpy().reshape(nb, K),
                                        pairs)
        assert np.array_equal(d[2].cpu().numpy(), ekt.reshape(-1))
        assert np.array_equal(d[3].cpu().numpy(), evt.reshape(-1))
    else:
        assert np.array_equal(d[2].cpu().numpy(), kts.numpy())   # fp8: scales untouched


def quant_problem(fmt, lens, H_q, H_kv, D, K, q_dtype, seed):
    """A decode step whose pool already holds quantized history: codes drawn
    directly (fp8: finite codes with |value| <= 8; int8: any code with a
    random per-slot scale); slots without history hold NaN canaries (fp8 code
    0x7F, int8 scale NaN)."""
    w = wl.build_decode("quant", lens, H_q, H_kv, D, K, q_dtype, seed=seed)
    rng = np.random.default_rng(seed)
    nb, hist = w.num_blocks, w.history_mask
    shape = (nb, K, H_kv, D)
    c = wl.materialize(w, seed=seed, canary=False)
    if fmt in ("fp8", "k16v8"):
        vals = Q.e4m3_values()
        ok = np.array([i for i in range(256) if np.isfinite(vals[i]) and abs(vals[i]) <= 8],
                      np.uint8)
        kc = rng.choice(ok, size=shape).astype(np.uint8)
        vc = rng.choice(ok, size=shape).astype(np.uint8)
        kc[~hist] = 0x7F
        vc[~hist] = 0x7F
        if fmt == "k16v8":    # K: bf16 patterns of N(0, 1) draws, NaN without history
            kc = (rng.standard_normal(shape).astype(np.float32).view(np.uint32) >> 16).astype(
                np.uint16)
            kc[~hist] = 0x7FC1
        return w, c, kc, vc, None, None
    kc = rng.integers(-127, 128, size=shape).astype(np.int8)
    vc = rng.integers(-127, 128, size=shape).astype(np.int8)
    kts = rng.uniform(0.002, 0.03, size=nb * K).astype(np.float32)
    vts = rng.uniform(0.002, 0.03, size=nb * K).astype(np.float32)
    kts[~hist.reshape(-1)] = np.nan
    vts[~hist.reshape(-1)] = np.nan
    return w, c, kc, vc, kts, vts


SHAPES = [(128, 4, 16), (64, 2, 4), (128, 8, 32)]


@pytest.mark.parametrize("fmt", ["fp8", "int8", "k16v8"])
@pytest.mark.parametrize("q_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("D,G,K", SHAPES)
@pytest.mark.parametrize("num_splits", [0, 64])
def test_quant_step_matches_oracle(ops, fmt, q_dtype, D, G, K, num_splits):
    run_quant_step(ops, fmt, q_dtype, D, G, K, [1, 17, 0, 300, 64, 601], H_kv=2,
                   num_splits=num_splits)


@pytest.mark.parametrize("fmt", ["fp8", "int8", "k16v8"])
@pytest.mark.parametrize("kernel", [1, 2])
@pytest.mark.parametrize("num_splits", [0, 3, 40])
def test_quant_tensor_core_and_cuda_core(ops, fmt, kernel, num_splits):
    lens = [0, 1, 15, 16, 17, 700, 33, 2048]
    run_quant_step(ops, fmt, "bf16", 128, 4, 16, lens, H_kv=8, kernel=kernel,
                   num_splits=num_splits)


@pytest.mark.parametrize("fmt", ["fp8", "int8", "k16v8"])
@pytest.mark.parametrize("G,K,H_kv", [(8, 32, 8), (2, 64, 4), (1, 16, 1), (4, 8, 8), (2, 8, 2)])
def test_quant_tensor_core_shapes(ops, fmt, G, K, H_kv):
    # the bf16-K / FP8-V pair has no 8-token-block tiles: automatic plan there
    kern = 0 if fmt == "k16v8" and K == 8 else 1
    run_quant_step(ops, fmt, "bf16", 128, G, K, [5, 130, 1000, 64], H_kv=H_kv, kernel=kern)


@pytest.mark.parametrize("in_dtype", [torch.bfloat16, torch.float32])
def test_k16v8_append_bit_exact(ops, in_dtype):
    """K rows stored as bfloat16 (float32 input rounded to nearest even, bf16
    input copied), V rows as e4m3 codes of x / v_scale."""
    rng = np.random.default_rng(5)
    T, H, D, K, nb = 150, 8, 128, 16, 170
    mags = 10.0 ** rng.uniform(-3, 3, size=(T, 1, 1))
    k = torch.from_numpy((rng.standard_normal((T, H, D)) * mags).astype(np.float32)).to(in_dtype)
    v = torch.from_numpy((rng.standard_normal((T, H, D)) * mags).astype(np.float32)).to(in_dtype)
    bt, pos = identity_tables(T, K, nb, rng)
    pos[4] = -1
    kc = torch.full((nb, K, H, D), float("nan"), dtype=torch.bfloat16)
    vc = torch.full((nb, K, H, D), 0x7F, dtype=torch.uint8)
    dk, dv = kc.to(DEV), vc.to(DEV)
    qd = ops.kv_quant("k16v8", v_scale=0.3)
    ops.paged_kv_append_quant(k.to(DEV), v.to(DEV), torch.from_numpy(bt).to(DEV),
                              torch.from_numpy(pos).to(DEV), dk, dv, qd)
    assert ops.get_device_error() == 0
    slots = oracle.slot_mapping(bt, pos, K)
    ek, ev = Q.kv_write_k16v8(storage(kc), vc.numpy(), f32_rows(k), f32_rows(v), slots, 0.3)
    assert np.array_equal(storage(dk), ek) and np.array_equal(dv.cpu().numpy(), ev)


def run_quant_step(ops, fmt, q_dtype, D, G, K, lens, H_kv=2, **attn_kw):
    w, c, kc, vc, kts, vts = quant_problem(fmt, lens, G * H_kv, H_kv, D, K, q_dtype,
                                           seed=D + G + K + len(lens))
    dkc, dvc = torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV)
    if fmt == "fp8":
        qd = ops.kv_quant("fp8", 0.5, 1.5)
        scales = dict(k_scale=0.5, v_scale=1.5)
    elif fmt == "k16v8":
        dkc = torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16).to(DEV)
        qd = ops.kv_quant("k16v8", v_scale=1.5)
        scales = dict(v_scale=1.5)
    else:
        dkt, dvt = torch.from_numpy(kts.copy()).to(DEV), torch.from_numpy(vts.copy()).to(DEV)
        qd = ops.kv_quant("int8", k_token_scales=dkt, v_token_scales=dvt)
    d = {k: v.to(DEV) for k, v in c.items()}
    ops.paged_kv_append_quant(d["k_new"], d["v_new"], d["block_tables"], d["positions"], dkc,
                              dvc, qd)
    out = ops.paged_attention_decode_quant(d["q"], dkc, dvc, d["block_tables"],
                                           d["context_lens"], w.scale, qd,
                                           max_context_len=w.max_context_len, **attn_kw)
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    slots = oracle.slot_mapping(w.block_tables, w.positions, w.block_size)
    if fmt == "fp8":
        okc, ovc = Q.kv_write_fp8(kc, vc, f32_rows(c["k_new"]), f32_rows(c["v_new"]), slots,
                                  0.5, 1.5)
        tok = {}
    elif fmt == "k16v8":
        okc, ovc = Q.kv_write_k16v8(kc, vc, f32_rows(c["k_new"]), f32_rows(c["v_new"]), slots,
                                    1.5)
        tok = {}
    else:
        okc, ovc, okt, ovt = Q.kv_write_int8(kc, vc, kts, vts, f32_rows(c["k_new"]),
                                             f32_rows(c["v_new"]), slots)
        scales = {}
        tok = dict(k_tok_scales=okt, v_tok_scales=ovt)
        assert np.array_equal(dkt.cpu().numpy().view(np.uint32), okt.view(np.uint32))
    assert np.array_equal(storage(dkc), okc) and np.array_equal(dvc.cpu().numpy(), ovc)
    ref = Q.paged_attention_decode_quant(storage(c["q"]), okc, ovc, w.block_tables,
                                         w.context_lens, w.scale, q_dtype, fmt, **scales, **tok)
    check_attention(as_f64(out), ref, q_dtype, f"{fmt} {q_dtype} D{D} G{G} K{K} {attn_kw}")


def test_quant_rejects_bad_descriptions(ops):
    q = torch.zeros((1, 2, 128), dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros((2, 16, 1, 128), dtype=torch.uint8, device=DEV)
    bt = torch.zeros((1, 1), dtype=torch.int32, device=DEV)
    lens = torch.ones(1, dtype=torch.int32, device=DEV)
    with pytest.raises(ops.PagedKVError, match="scales"):
        ops.paged_attention_decode_quant(q, kc, kc, bt, lens, 0.1, ops.kv_quant("fp8", 0.0, 1.0))
    bad = ops.KvQuant()
    bad.format = 2                              # int8 without scale arrays
    with pytest.raises(ops.PagedKVError, match="scale"):
        ops.paged_attention_decode_quant(q, kc, kc, bt, lens, 0.1, bad)


@pytest.mark.parametrize("fmt", ["fp8", "int8"])
@pytest.mark.parametrize("kernel", [0, 1, 2])
def test_quant_rising_scores_rescale(ops, fmt, kernel):
    """Scores that rise along every sequence (and jump at its last token), so
    that the running exponent base of the one-byte tensor-core path is raised
    many times; the output must still be the oracle's softmax."""
    lens = [40, 700, 2048, 17]
    H_kv, G, D, K = 2, 4, 128, 16
    w = wl.build_decode("rising", lens, G * H_kv, H_kv, D, K, "bf16", seed=3)
    rng = np.random.default_rng(3)
    nb = w.num_blocks
    shape = (nb, K, H_kv, D)
    q = torch.ones((len(lens), G * H_kv, D), dtype=torch.bfloat16)
    # key value of position t of sequence s: 6 t / len, the last token 12
    kval = np.zeros((nb, K), np.float32)
    for s, L in enumerate(lens):
        t = np.arange(L)
        v = 6.0 * t / L
        v[-1] = 12.0
        kval[w.block_tables[s][t // K], t % K] = v
    if fmt == "fp8":
        vals = Q.e4m3_values()
        finite = np.array([i for i in range(256) if np.isfinite(vals[i])], np.uint8)
        fv = vals[finite]
        near = finite[np.abs(fv[None, :] - kval.reshape(-1, 1)).argmin(axis=1)].reshape(nb, K)
        kc = np.repeat(near[:, :, None, None], H_kv, 2).repeat(D, 3).astype(np.uint8)
        ok = np.array([i for i in range(256) if np.isfinite(vals[i]) and abs(vals[i]) <= 8],
                      np.uint8)
        vc = rng.choice(ok, size=shape).astype(np.uint8)
        qd = ops.kv_quant("fp8", 1.0, 0.75)
        extra = dict(k_scale=1.0, v_scale=0.75)
    else:
        kc = np.full(shape, 100, np.int8)
        kts = (kval.reshape(-1) / 100.0).astype(np.float32)
        vc = rng.integers(-127, 128, size=shape).astype(np.int8)
        vts = rng.uniform(0.002, 0.03, size=nb * K).astype(np.float32)
        qd = ops.kv_quant("int8", k_token_scales=torch.from_numpy(kts).to(DEV),
                          v_token_scales=torch.from_numpy(vts).to(DEV))
        extra = dict(k_tok_scales=kts, v_tok_scales=vts)
    out = ops.paged_attention_decode_quant(q.to(DEV), torch.from_numpy(kc).to(DEV),
                                           torch.from_numpy(vc).to(DEV),
                                           torch.from_numpy(w.block_tables).to(DEV),
                                           torch.tensor(lens, dtype=torch.int32, device=DEV),
                                           w.scale, qd, max_context_len=max(lens), kernel=kernel)
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    ref = Q.paged_attention_decode_quant(storage(q), kc, vc, w.block_tables, np.array(lens),
                                         w.scale, "bf16", fmt, **extra)
    check_attention(as_f64(out), ref, "bf16", f"rising {fmt} kernel={kernel}")
