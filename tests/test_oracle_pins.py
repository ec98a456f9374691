"""Pins of the CPU oracle against things other than itself.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with
what the pages or plain mathematics fix: the pages' worked examples
(``tests/golden``), closed forms, invariants, and scalar brute force on tiny
inputs.  ``test_mutations_are_caught`` plants plausible mistakes in the oracle
(on the CPU, through monkeypatching) and checks that some pin fails for each.
"""

import math

import numpy as np
import pytest

import oracle
import oracle.paged_attention as opa

RNG = np.random.default_rng(1234)


# --------------------------------------------------------------------------
# helpers (test-local, independent of the oracle)
# --------------------------------------------------------------------------

def append_tokens_p1(num_tokens, block_size, free_list):
    """Allocate blocks one token at a time the way ``BlockTable.append_token``
    does in "19.2 KV Cache 系统化管理" §19.2.3: a new block is popped from the
    end of the free list whenever the token opens a new logical block.
    Returns (block table, {position: (physical block, offset)})."""
    table, where = [], {}
    filled = 0
    for _ in range(num_tokens):
        blk_i, off = divmod(filled, block_size)
        if blk_i >= len(table):
            table.append(free_list.pop())
        where[filled] = (table[blk_i], off)
        filled += 1
    return table, where


def scalar_attention(q, keys, vals, scale):
    """Pure-Python scalar loops: softmax(scale * q.k) . v."""
    if not keys:
        return [0.0] * len(q)
    z = [scale * sum(qd * kd for qd, kd in zip(q, k)) for k in keys]
    m = max(z)
    e = [math.exp(x - m) for x in z]
    tot = sum(e)
    return [sum(e[t] * vals[t][d] for t in range(len(keys))) / tot
            for d in range(len(q))]


def random_paged_problem(rng, S, H_q, H_kv, D, K, lens, extra_blocks=3,
                         nan_fill=True):
    """Small f32 paged problem with blocks placed in random order, every
    unused slot and unused block set to NaN, and garbage past each table."""
    need = [-(-L // K) for L in lens]
    nb = sum(need) + extra_blocks
    order = rng.permutation(nb)
    maxB = max(max(need), 1) + 2
    bt = rng.integers(10**6, 10**7, size=(S, maxB)).astype(np.int64)  # garbage
    fill = np.nan if nan_fill else 0.0
    kc = np.full((nb, K, H_kv, D), fill, dtype=np.float32)
    vc = np.full((nb, K, H_kv, D), fill, dtype=np.float32)
    Kc = [rng.standard_normal((L, H_kv, D)).astype(np.float32) for L in lens]
    Vc = [rng.standard_normal((L, H_kv, D)).astype(np.float32) for L in lens]
    p = 0
    for s, L in enumerate(lens):
        for i in range(need[s]):
            bt[s, i] = order[p]
            p += 1
        for t in range(L):
            kc[bt[s, t // K], t % K] = Kc[s][t]
            vc[bt[s, t // K], t % K] = Vc[s][t]
    q = rng.standard_normal((S, H_q, D)).astype(np.float32)
    return q, kc, vc, bt, np.array(lens, dtype=np.int64), Kc, Vc


# --------------------------------------------------------------------------
# pins: decoding
# --------------------------------------------------------------------------

def pin_decode():
    bits = np.array([0x3F80, 0xC000, 0x7F80, 0xFF80, 0x0001, 0x3F81, 0x0000,
                     0x8000, 0x4049], dtype=np.uint16)
    want = [1.0, -2.0, np.inf, -np.inf, 2.0 ** -133, 1.0 + 2.0 ** -7, 0.0,
            -0.0, 3.140625]
    got = oracle.decode(bits, "bf16")
    assert got.dtype == np.float64
    for g, w in zip(got, want):
        assert g == w, (g, w)
    assert np.signbit(got[7])
    assert np.isnan(oracle.decode(np.array([0x7FC1], np.uint16), "bf16")[0])
    f = np.array([1.5, -2.25e-30, 3.4e38], dtype=np.float32)
    assert np.array_equal(oracle.decode(f, "f32"), f.astype(np.float64))
    assert np.array_equal(oracle.decode(f.view(np.uint32), "f32"), f.astype(np.float64))
    assert oracle.decode(np.array([0x3F800000], np.uint32), "f32")[0] == 1.0


# --------------------------------------------------------------------------
# pins: slot mapping
# --------------------------------------------------------------------------

def pin_slot_p3_example(g):
    K = g["block_size"]
    bt = np.array([g["block_table"]])
    for i, (lo, hi) in enumerate(g["logical_block_positions"]):
        for t in range(lo, hi + 1):
            slot = oracle.slot_mapping(bt, np.array([t]), K)[0]
            assert slot == g["block_table"][i] * K + (t - lo), (t, slot)
    tr = g["trace"]
    assert oracle.slot_mapping(bt, np.array([tr["position"]]), K)[0] == tr["slot"]


def pin_slot_p1_lifecycle(g):
    K = g["block_size"]
    bt = np.array([g["final_block_table"]])
    for step in g["decode"]:
        assert oracle.slot_mapping(bt, np.array([step["position"]]), K)[0] == step["slot"]
        assert step["slot"] == step["physical_block"] * K + step["offset"]


def pin_slot_p4(g):
    K = g["block_size"]
    bt = np.array([g["block_table"]])
    assert -(-g["num_tokens"] // K) == len(g["block_table"])
    d = g["derived"]
    assert oracle.slot_mapping(bt, np.array([d["position"]]), K)[0] == d["slot"]


def pin_slot_brute_force():
    rng = np.random.default_rng(7)
    for K in (1, 2, 4, 8, 16, 32):
        for L in (1, K - 1 if K > 1 else 1, K, K + 1, 3 * K + 2):
            free = list(rng.permutation(64))
            table, where = append_tokens_p1(L, K, free)
            bt = np.array([table + [999999] * 3])
            for t in range(L):
                slot = oracle.slot_mapping(bt, np.array([t]), K)[0]
                blk, off = where[t]
                assert slot == blk * K + off, (K, L, t)
    # padding entries
    assert oracle.slot_mapping(np.array([[3]]), np.array([-1]), 4)[0] == -1


# --------------------------------------------------------------------------
# pins: KV write and block copy (bit exact)
# --------------------------------------------------------------------------

def pin_kv_write_brute_force():
    rng = np.random.default_rng(11)
    nb, K, H, D = 6, 4, 2, 3
    canary = np.uint32(0x7FC0DEAD)  # NaN with a payload: must survive untouched
    kc = np.full((nb, K, H, D), canary, dtype=np.uint32)
    vc = np.full((nb, K, H, D), canary + 1, dtype=np.uint32)
    T = 7
    slots = rng.choice(nb * K, size=T, replace=False).astype(np.int64)
    slots[3] = -1
    k = rng.integers(0, 2**32, size=(T, H, D), dtype=np.uint32)
    v = rng.integers(0, 2**32, size=(T, H, D), dtype=np.uint32)
    nk, nv = oracle.kv_write(kc, vc, k, v, slots)
    for b in range(nb):
        for o in range(K):
            flat = b * K + o
            hits = [i for i in range(T) if slots[i] == flat]
            for h in range(H):
                for d in range(D):
                    if hits:
                        assert nk[b, o, h, d] == k[hits[0], h, d]
                        assert nv[b, o, h, d] == v[hits[0], h, d]
                    else:
                        assert nk[b, o, h, d] == canary
                        assert nv[b, o, h, d] == canary + 1
    assert np.all(kc == canary)  # inputs are not modified


def pin_block_copy_brute_force():
    rng = np.random.default_rng(12)
    nb, K, H, D = 8, 4, 2, 2
    kc = rng.integers(0, 2**16, size=(nb, K, H, D), dtype=np.uint16)
    vc = rng.integers(0, 2**16, size=(nb, K, H, D), dtype=np.uint16)
    pairs = np.array([[1, 5], [2, 6], [0, 7]], dtype=np.int64)
    nk, nv = oracle.kv_block_copy(kc, vc, pairs)
    for b in range(nb):
        src = {5: 1, 6: 2, 7: 0}.get(b, b)
        assert np.array_equal(nk[b], kc[src]) and np.array_equal(nv[b], vc[src])


def pin_cow_sequence():
    """§19.2.2 写时复制: two samples share a partially filled block (refcount
    2); the first writer gets a copy, then both write different tokens."""
    K, H, D = 4, 1, 2
    kc = np.zeros((4, K, H, D), dtype=np.float32)
    vc = np.zeros((4, K, H, D), dtype=np.float32)
    kc[2, :3] = np.arange(6, dtype=np.float32).reshape(3, H, D) + 1
    vc[2, :3] = -kc[2, :3]
    # sample A copies block 2 -> 3 then writes at offset 3; B writes in place
    kc, vc = oracle.kv_block_copy(kc, vc, np.array([[2, 3]]))
    a_new = np.full((1, H, D), 10.0, np.float32)
    b_new = np.full((1, H, D), 20.0, np.float32)
    kc, vc = oracle.kv_write(kc, vc, a_new, -a_new, np.array([3 * K + 3]))
    kc, vc = oracle.kv_write(kc, vc, b_new, -b_new, np.array([2 * K + 3]))
    assert np.array_equal(kc[3, :3], kc[2, :3])
    assert kc[3, 3, 0, 0] == 10.0 and kc[2, 3, 0, 0] == 20.0
    assert np.array_equal(vc[3, :3], vc[2, :3])


# --------------------------------------------------------------------------
# pins: attention
# --------------------------------------------------------------------------

def pin_p1_selfcheck(g):
    """The page's own check: paged attention equals dense attention on the
    same K/V (bound 1e-5 in fp32; the fp64 oracle must be far tighter)."""
    rng = np.random.default_rng(5)
    nb, K, H, D, L = (g["num_blocks"], g["block_size"], g["num_heads"],
                      g["head_dim"], g["num_tokens"])
    free = list(range(nb))
    table, where = append_tokens_p1(L, K, free)
    assert len(table) == g["blocks_used"]
    kc = np.zeros((nb, K, H, D), np.float32)
    vc = np.zeros((nb, K, H, D), np.float32)
    Kd = rng.standard_normal((L, H, D)).astype(np.float32)
    Vd = rng.standard_normal((L, H, D)).astype(np.float32)
    for t in range(L):
        b, o = where[t]
        kc[b, o], vc[b, o] = Kd[t], Vd[t]
    q = rng.standard_normal((1, H, D)).astype(np.float32)
    scale = 1.0 / math.sqrt(D)
    out = oracle.paged_attention_decode(q, kc, vc, np.array([table]),
                                        np.array([L]), scale, "f32")
    for h in range(H):
        dense = oracle.dense_attention(q[0, h].astype(np.float64),
                                       Kd[:, h].astype(np.float64),
                                       Vd[:, h].astype(np.float64), scale)
        err = np.abs(out[0, h] - dense).max()
        assert err < g["max_error_bound_fp32"]
        assert err < 1e-12


def pin_dense_vs_paged_random():
    rng = np.random.default_rng(21)
    for K in (1, 2, 4, 16):
        lens = [1, K, K + 1, 3 * K - 1, 37]
        q, kc, vc, bt, cl, Kc, Vc = random_paged_problem(rng, 5, 4, 2, 8, K, lens)
        out = oracle.paged_attention_decode(q, kc, vc, bt, cl, 0.3, "f32")
        for s, L in enumerate(lens):
            for h in range(4):
                ref = oracle.dense_attention(q[s, h].astype(np.float64),
                                             Kc[s][:, h // 2].astype(np.float64),
                                             Vc[s][:, h // 2].astype(np.float64), 0.3)
                assert np.abs(out[s, h] - ref).max() < 1e-12, (K, s, h)
        assert np.all(np.isfinite(out))  # NaN canaries were never read


def pin_permutation_invariance():
    rng = np.random.default_rng(22)
    K, H_kv, D = 4, 2, 8
    lens = [9, 14, 4]
    q, kc, vc, bt, cl, _, _ = random_paged_problem(rng, 3, 4, H_kv, D, K, lens)
    out1 = oracle.paged_attention_decode(q, kc, vc, bt, cl, 0.25, "f32")
    nb = kc.shape[0]
    perm = rng.permutation(nb)           # block b moves to perm[b]
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = bt.copy()
    for s, L in enumerate(lens):
        n = -(-L // K)
        bt2[s, :n] = perm[bt[s, :n]]
    out2 = oracle.paged_attention_decode(q, kc2, vc2, bt2, cl, 0.25, "f32")
    assert np.abs(out1 - out2).max() < 1e-13


def pin_gqa_equals_mha():
    rng = np.random.default_rng(23)
    K, H_q, H_kv, D = 4, 8, 2, 4
    lens = [6, 11]
    q, kc, vc, bt, cl, _, _ = random_paged_problem(rng, 2, H_q, H_kv, D, K, lens)
    out = oracle.paged_attention_decode(q, kc, vc, bt, cl, 0.5, "f32")
    G = H_q // H_kv
    kc_m = np.repeat(kc, G, axis=2)  # KV head j serves query heads j*G .. j*G+G-1
    vc_m = np.repeat(vc, G, axis=2)
    out_m = oracle.paged_attention_decode(q, kc_m, vc_m, bt, cl, 0.5, "f32")
    assert np.abs(out - out_m).max() < 1e-13


def pin_closed_forms():
    rng = np.random.default_rng(24)
    K, D = 4, 6
    # len = 1 -> out = v0 exactly
    q, kc, vc, bt, cl, Kc, Vc = random_paged_problem(rng, 1, 2, 2, D, K, [1])
    out = oracle.paged_attention_decode(q, kc, vc, bt, cl, 0.7, "f32")
    for h in range(2):
        assert np.array_equal(out[0, h], Vc[0][0, h].astype(np.float64))
    # q = 0 -> plain mean of V
    q, kc, vc, bt, cl, Kc, Vc = random_paged_problem(rng, 1, 2, 2, D, K, [7])
    q[:] = 0
    out = oracle.paged_attention_decode(q, kc, vc, bt, cl, 0.7, "f32")
    assert np.abs(out[0, 1] - Vc[0][:, 1].astype(np.float64).mean(0)).max() < 1e-14
    # all keys equal -> mean of V
    q, kc, vc, bt, cl, Kc, Vc = random_paged_problem(rng, 1, 2, 2, D, K, [9])
    for t in range(9):
        kc[bt[0, t // K], t % K] = kc[bt[0, 0], 0]
    out = oracle.paged_attention_decode(q, kc, vc, bt, cl, 0.7, "f32")
    assert np.abs(out[0, 0] - Vc[0][:, 0].astype(np.float64).mean(0)).max() < 1e-14
    # two tokens: out = v1 + (v0 - v1) * sigmoid(z0 - z1)
    q, kc, vc, bt, cl, Kc, Vc = random_paged_problem(rng, 1, 1, 1, D, K, [2])
    scale = 0.37
    q64 = q[0, 0].astype(np.float64)
    k0, k1 = Kc[0][0, 0].astype(np.float64), Kc[0][1, 0].astype(np.float64)
    v0, v1 = Vc[0][0, 0].astype(np.float64), Vc[0][1, 0].astype(np.float64)
    dz = scale * (q64 @ k0 - q64 @ k1)
    want = v1 + (v0 - v1) / (1.0 + math.exp(-dz))
    out = oracle.paged_attention_decode(q, kc, vc, bt, cl, scale, "f32")
    assert np.abs(out[0, 0] - want).max() < 1e-14
    # constant V -> that constant
    q, kc, vc, bt, cl, Kc, Vc = random_paged_problem(rng, 1, 2, 2, D, K, [10])
    for t in range(10):
        vc[bt[0, t // K], t % K] = 1.25
    out = oracle.paged_attention_decode(q, kc, vc, bt, cl, 0.7, "f32")
    assert np.abs(out - 1.25).max() < 1e-14
    # empty context -> zeros (reading)
    q, kc, vc, bt, cl, Kc, Vc = random_paged_problem(rng, 2, 2, 2, D, K, [0, 3])
    out = oracle.paged_attention_decode(q, kc, vc, bt, cl, 0.7, "f32")
    assert np.array_equal(out[0], np.zeros((2, D)))


def pin_streaming_matches_two_pass():
    rng = np.random.default_rng(25)
    for K in (1, 4, 16):
        lens = [1, 2 * K + 3, 50]
        q, kc, vc, bt, cl, _, _ = random_paged_problem(rng, 3, 4, 2, 8, K, lens)
        out = oracle.paged_attention_decode(q, kc, vc, bt, cl, 0.4, "f32")
        for s, L in enumerate(lens):
            st = oracle.paged_attention_streaming(q[s], kc, vc, bt[s], L, 0.4, "f32")
            assert np.abs(st - out[s]).max() < 1e-12


def pin_scalar_brute_force():
    rng = np.random.default_rng(26)
    for trial in range(30):
        K = int(rng.choice([1, 2, 4]))
        D = int(rng.integers(1, 5))
        H_kv = int(rng.choice([1, 2]))
        G = int(rng.choice([1, 2]))
        lens = [int(x) for x in rng.integers(1, 6, size=2)]
        q, kc, vc, bt, cl, Kc, Vc = random_paged_problem(rng, 2, H_kv * G, H_kv, D, K, lens)
        scale = float(rng.uniform(0.1, 1.5))
        out = oracle.paged_attention_decode(q, kc, vc, bt, cl, scale, "f32")
        for s in range(2):
            for h in range(H_kv * G):
                keys = [[float(x) for x in Kc[s][t, h // G]] for t in range(lens[s])]
                vals = [[float(x) for x in Vc[s][t, h // G]] for t in range(lens[s])]
                ref = scalar_attention([float(x) for x in q[s, h]], keys, vals, scale)
                assert np.abs(out[s, h] - np.array(ref)).max() < 1e-13, trial


def pin_decode_one():
    """The single-row oracle (the checker of the full-size GPU tests) against
    (a) a pure-Python scalar brute force that maps query head h to KV head
    h // G by itself, on tiny problems, and (b) the whole-batch oracle, row by
    row, over GQA ratios 1, 2, 4, 8 and block sizes 1, 4, 16 with NaN in every
    slot without history and garbage past each table row."""
    rng = np.random.default_rng(29)
    for G in (1, 2, 4, 8):
        for K in (1, 4, 16):
            H_kv = 2
            H_q = H_kv * G
            D = 3
            lens = [1, K + 2, 2 * K + 1, 0]
            q, kc, vc, bt, cl, Kc, Vc = random_paged_problem(rng, len(lens), H_q, H_kv, D, K,
                                                             lens)
            scale = float(rng.uniform(0.2, 1.2))
            whole = oracle.paged_attention_decode(q, kc, vc, bt, cl, scale, "f32")
            for s, L in enumerate(lens):
                for h in range(H_q):
                    one = oracle.paged_attention_decode_one(q, kc, vc, bt, cl, scale, s, h,
                                                            "f32")
                    kvh = h // G
                    keys = [[float(x) for x in Kc[s][t, kvh]] for t in range(L)]
                    vals = [[float(x) for x in Vc[s][t, kvh]] for t in range(L)]
                    ref = scalar_attention([float(x) for x in q[s, h]], keys, vals, scale)
                    assert np.abs(one - np.array(ref)).max() < 1e-13, (G, K, s, h)
                    assert np.abs(one - whole[s, h]).max() < 1e-13, (G, K, s, h)


def pin_attention_rows():
    """Several query rows at once, each up to its own inclusive key limit:
    equal to a pure-Python scalar brute force over keys 0 .. limit (tiny
    sizes), and a negative limit gives zeros."""
    rng = np.random.default_rng(30)
    for trial in range(25):
        L = int(rng.integers(1, 9))
        D = int(rng.integers(1, 5))
        R = int(rng.integers(1, 6))
        Kd = rng.standard_normal((L, D)) * 1.5
        Vd = rng.standard_normal((L, D))
        Qd = rng.standard_normal((R, D))
        lim = rng.integers(-1, L, size=R)
        scale = float(rng.uniform(0.2, 1.3))
        got = oracle.attention_rows(Qd, Kd, Vd, lim, scale)
        for i in range(R):
            n = int(lim[i]) + 1
            keys = [[float(x) for x in Kd[t]] for t in range(n)]
            vals = [[float(x) for x in Vd[t]] for t in range(n)]
            ref = scalar_attention([float(x) for x in Qd[i]], keys, vals, scale)
            assert np.abs(got[i] - np.array(ref)).max() < 1e-13, (trial, i)


def pin_bf16_path():
    """bf16 storage decodes exactly: the oracle on bf16 bit patterns equals
    the oracle on the same numbers stored as f32."""
    rng = np.random.default_rng(27)
    q, kc, vc, bt, cl, _, _ = random_paged_problem(rng, 2, 4, 2, 8, 4, [5, 9],
                                                   nan_fill=False)

    def to_bf16_bits(x):  # truncation gives some bf16 number; exactness is the point
        return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)

    qb, kb, vb = to_bf16_bits(q), to_bf16_bits(kc), to_bf16_bits(vc)
    back = lambda b: (b.astype(np.uint32) << 16).view(np.float32)
    out_b = oracle.paged_attention_decode(qb, kb, vb, bt, cl, 0.3, "bf16")
    out_f = oracle.paged_attention_decode(back(qb), back(kb), back(vb), bt, cl, 0.3, "f32")
    assert np.array_equal(out_b, out_f)


def pin_merge_identity():
    rng = np.random.default_rng(28)
    for trial in range(20):
        L = int(rng.integers(1, 60))
        D = 5
        q = rng.standard_normal(D)
        Kd = rng.standard_normal((L, D)) * 2
        Vd = rng.standard_normal((L, D))
        cuts = np.sort(rng.integers(0, L + 1, size=int(rng.integers(0, 5))))
        bounds = [0, *cuts.tolist(), L]
        parts = [oracle.partial_state(q, Kd[a:b], Vd[a:b], 0.6)
                 for a, b in zip(bounds[:-1], bounds[1:])]
        ms, ls, os_ = zip(*parts)
        merged = oracle.merge_partials(ms, ls, os_)
        ref = oracle.dense_attention(q, Kd, Vd, 0.6)
        assert np.abs(merged - ref).max() < 1e-12
    assert np.array_equal(oracle.merge_partials([-np.inf], [0.0], [np.zeros(3)]),
                          np.zeros(3))


# --------------------------------------------------------------------------
# tests
# --------------------------------------------------------------------------

def test_decode():
    pin_decode()


def test_slot_mapping_pins(golden):
    pin_slot_p3_example(golden("p3_block_table_example.json"))
    pin_slot_p1_lifecycle(golden("p1_lifecycle_example.json"))
    pin_slot_p4(golden("p4_35_tokens.json"))
    pin_slot_brute_force()


def test_write_and_copy_pins():
    pin_kv_write_brute_force()
    pin_block_copy_brute_force()
    pin_cow_sequence()


def test_attention_pins(golden):
    pin_p1_selfcheck(golden("p1_selfcheck.json"))
    pin_dense_vs_paged_random()
    pin_permutation_invariance()
    pin_gqa_equals_mha()
    pin_closed_forms()
    pin_streaming_matches_two_pass()
    pin_scalar_brute_force()
    pin_decode_one()
    pin_attention_rows()
    pin_bf16_path()


def test_merge_pins():
    pin_merge_identity()


def _all_attention_pins(golden):
    pin_p1_selfcheck(golden("p1_selfcheck.json"))
    pin_dense_vs_paged_random()
    pin_gqa_equals_mha()
    pin_closed_forms()
    pin_scalar_brute_force()


def _mut_gather_offset_swapped(cache, row, length, kv_head, K, dtype):
    t = np.arange(length, dtype=np.int64)
    phys = np.asarray(row, dtype=np.int64)[t % K]          # index mistake
    return opa.decode(cache[phys, t // K, kv_head, :], dtype) if K > 0 else None


def _mut_gqa_modulo(q, k_cache, v_cache, bt, cl, scale, dtype):
    S, H_q, D = q.shape
    H_kv = k_cache.shape[2]
    out = np.zeros((S, H_q, D))
    for s in range(S):
        for h in range(H_q):
            j = h % H_kv                                     # wrong head map
            Kj = opa.gather_kv(k_cache, bt[s], int(cl[s]), j, k_cache.shape[1], dtype)
            Vj = opa.gather_kv(v_cache, bt[s], int(cl[s]), j, k_cache.shape[1], dtype)
            out[s, h] = opa.dense_attention(opa.decode(q[s, h], dtype), Kj, Vj, scale)
    return out


def _mut_one_gqa_modulo(q, k_cache, v_cache, bt, cl, scale, s, h, dtype):
    H_kv = k_cache.shape[2]
    j = h % H_kv                                             # wrong head map
    Kj = opa.gather_kv(k_cache, bt[s], int(cl[s]), j, k_cache.shape[1], dtype)
    Vj = opa.gather_kv(v_cache, bt[s], int(cl[s]), j, k_cache.shape[1], dtype)
    return opa.dense_attention(opa.decode(q[s, h], dtype), Kj, Vj, scale)


def _mut_rows_exclusive(Q, K, V, limits, scale):
    lim = np.asarray(limits, np.int64) - 1                   # exclusive bound
    return _orig_attention_rows(Q, K, V, lim, scale)


_orig_attention_rows = opa.attention_rows


def _mut_dense_no_scale(q, K, V, scale):
    if K.shape[0] == 0:
        return np.zeros(V.shape[1])
    z = K @ np.asarray(q, np.float64)                        # dropped scale
    w = np.exp(z - z.max())
    return (w / w.sum()) @ V


def _mut_dense_kv_swapped(q, K, V, scale):
    if K.shape[0] == 0:
        return np.zeros(V.shape[1])
    z = scale * (V @ np.asarray(q, np.float64))              # transposed operands
    w = np.exp(z - z.max())
    return (w / w.sum()) @ K


def _mut_slot_wrong(bt, positions, K):
    out = np.empty(len(positions), np.int64)
    for s, t in enumerate(positions):
        out[s] = int(bt[s, t // K]) + (t % K) * K            # slot formula mistake
    return out


@pytest.mark.parametrize("target,replacement,check", [
    ("gather_kv", _mut_gather_offset_swapped, "attention"),
    ("paged_attention_decode", _mut_gqa_modulo, "gqa"),
    ("paged_attention_decode_one", _mut_one_gqa_modulo, "one"),
    ("attention_rows", _mut_rows_exclusive, "rows"),
    ("dense_attention", _mut_dense_no_scale, "attention"),
    ("dense_attention", _mut_dense_kv_swapped, "attention"),
    ("slot_mapping", _mut_slot_wrong, "slot"),
])
def test_mutations_are_caught(monkeypatch, golden, target, replacement, check):
    monkeypatch.setattr(opa, target, replacement)
    monkeypatch.setattr(oracle, target, replacement)
    with pytest.raises((AssertionError, IndexError)):
        if check == "attention":
            _all_attention_pins(golden)
        elif check == "gqa":
            pin_gqa_equals_mha()
        elif check == "one":
            pin_decode_one()
        elif check == "rows":
            pin_attention_rows()
        else:
            pin_slot_p3_example(golden("p3_block_table_example.json"))


# --------------------------------------------------------------------------
# block swap between pools in different memories
# ("19.2 KV Cache 系统化管理" §19.2.6 Swap; "企业官网建设流程全解析" §8.2)
# --------------------------------------------------------------------------

def _swap_brute(src, dst, pairs):
    """Element-by-element: every element of a destination block named in a
    pair equals the element at the same place in the named source block;
    every other element keeps its old value."""
    out = dst.copy()
    nb_dst = dst.shape[0]
    moved = {int(d): int(s) for s, d in pairs}
    it = np.nditer(dst, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        if idx[0] in moved:
            out[idx] = src[(moved[idx[0]],) + idx[1:]]
    assert out.shape[0] == nb_dst
    return out


def test_swap_brute_force_with_canaries():
    rng = np.random.default_rng(11)
    K, H, D = 4, 2, 3
    gpu_k = rng.standard_normal((9, K, H, D)).astype(np.float32)
    gpu_v = rng.standard_normal((9, K, H, D)).astype(np.float32)
    host_k = np.full((5, K, H, D), np.float32(-7.25))
    host_v = np.full((5, K, H, D), np.float32(13.5))
    out_pairs = np.array([[8, 0], [2, 3], [5, 4]], np.int64)
    hk, hv = oracle.kv_block_swap(gpu_k, gpu_v, host_k, host_v, out_pairs)
    assert np.array_equal(hk, _swap_brute(gpu_k, host_k, out_pairs))
    assert np.array_equal(hv, _swap_brute(gpu_v, host_v, out_pairs))
    assert np.all(hk[[1, 2]] == np.float32(-7.25)) and np.all(hv[[1, 2]] == np.float32(13.5))
    # the source pools are not touched
    assert np.array_equal(gpu_k, gpu_k.copy()) and hk is not host_k
    # order of pairs does not matter (the source is never written)
    hk2, hv2 = oracle.kv_block_swap(gpu_k, gpu_v, host_k, host_v, out_pairs[::-1])
    assert np.array_equal(hk, hk2) and np.array_equal(hv, hv2)


def test_swap_round_trip_restores_logical_view():
    """Preempt: copy a request's blocks out to host blocks; resume: copy them
    into freshly chosen GPU blocks and repoint the table.  Gathering the
    request's rows through the new table gives the rows it had before."""
    rng = np.random.default_rng(12)
    K, H, D, L = 4, 2, 5, 14
    nb = 12
    kc = rng.standard_normal((nb, K, H, D)).astype(np.float32)
    vc = rng.standard_normal((nb, K, H, D)).astype(np.float32)
    table = np.array([7, 2, 9, 4], np.int64)            # ceil(14 / 4) = 4 blocks
    before_k = [opa.gather_kv(kc, table, L, j, K, "f32") for j in range(H)]
    before_v = [opa.gather_kv(vc, table, L, j, K, "f32") for j in range(H)]
    host_ids = np.array([3, 0, 1, 2], np.int64)
    hk, hv = oracle.kv_block_swap(kc, vc, np.zeros((4, K, H, D), np.float32),
                                  np.zeros((4, K, H, D), np.float32),
                                  np.stack([table, host_ids], 1))
    # the GPU blocks are reused by someone else meanwhile
    kc2 = rng.standard_normal(kc.shape).astype(np.float32)
    vc2 = rng.standard_normal(vc.shape).astype(np.float32)
    new_table = np.array([0, 11, 5, 6], np.int64)
    kc3, vc3 = oracle.kv_block_swap(hk, hv, kc2, vc2, np.stack([host_ids, new_table], 1))
    for j in range(H):
        assert np.array_equal(opa.gather_kv(kc3, new_table, L, j, K, "f32"), before_k[j])
        assert np.array_equal(opa.gather_kv(vc3, new_table, L, j, K, "f32"), before_v[j])
    # blocks outside the new table keep the other user's data
    others = [b for b in range(nb) if b not in set(new_table.tolist())]
    assert np.array_equal(kc3[others], kc2[others])


def test_swap_within_one_pool_is_block_copy():
    rng = np.random.default_rng(13)
    kc = rng.integers(0, 2**16, size=(6, 4, 2, 8), dtype=np.uint16)
    vc = rng.integers(0, 2**16, size=(6, 4, 2, 8), dtype=np.uint16)
    pairs = np.array([[0, 5], [1, 3]], np.int64)
    a = oracle.kv_block_swap(kc, vc, kc, vc, pairs)
    b = oracle.kv_block_copy(kc, vc, pairs)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_swap_planted_mistake_is_caught(monkeypatch):
    """Plausible mistakes (K and V exchanged; the pair read as (dst, src))
    each fail a pin."""
    def kv_exchanged(src_k, src_v, dst_k, dst_v, pairs):
        dk, dv = dst_k.copy(), dst_v.copy()
        for s, d in np.asarray(pairs).reshape(-1, 2):
            dk[int(d)] = src_v[int(s)]
            dv[int(d)] = src_k[int(s)]
        return dk, dv

    def pair_reversed(src_k, src_v, dst_k, dst_v, pairs):
        dk, dv = dst_k.copy(), dst_v.copy()
        for d, s in np.asarray(pairs).reshape(-1, 2):
            if d < dk.shape[0] and s < src_k.shape[0]:
                dk[int(d)] = src_k[int(s)]
                dv[int(d)] = src_v[int(s)]
        return dk, dv

    # (exchanging K and V twice cancels, so the round trip alone misses it)
    for wrong, pins in ((kv_exchanged, (test_swap_brute_force_with_canaries,)),
                        (pair_reversed, (test_swap_brute_force_with_canaries,
                                         test_swap_round_trip_restores_logical_view))):
        monkeypatch.setattr(oracle, "kv_block_swap", wrong)
        for pin in pins:
            with pytest.raises(AssertionError):
                pin()
