"""Pins of the multi-query (prefill) oracle, oracle/prefill.py, against things
other than itself: the decode oracle at one new token, a scalar brute force,
causality, chunked = one-shot prefill, closed forms, planted mistakes."""

import math

import numpy as np
import pytest

import oracle
from oracle import prefill as P


def _problem(rng, lens, news, H_q=4, H_kv=2, D=6, K=4, dtype=np.float32):
    S = len(lens)
    nb = sum(-(-L // K) for L in lens) + 3
    order = rng.permutation(nb)
    maxb = max(-(-L // K) for L in lens) + 1
    bt = np.full((S, maxb), 10**6, np.int64)
    p = 0
    for s, L in enumerate(lens):
        for i in range(-(-L // K)):
            bt[s, i] = order[p]
            p += 1
    kc = rng.standard_normal((nb, K, H_kv, D)).astype(dtype)
    vc = rng.standard_normal((nb, K, H_kv, D)).astype(dtype)
    cu = np.concatenate([[0], np.cumsum(news)]).astype(np.int64)
    q = rng.standard_normal((int(cu[-1]), H_q, D)).astype(dtype)
    return q, kc, vc, bt, cu


def test_one_new_token_is_decode():
    rng = np.random.default_rng(1)
    lens = [5, 1, 13, 8]
    q, kc, vc, bt, cu = _problem(rng, lens, [1, 1, 1, 1])
    got = P.paged_attention_prefill(q, kc, vc, bt, cu, lens, 0.4, "f32")
    want = oracle.paged_attention_decode(q, kc, vc, bt, lens, 0.4, "f32")
    assert np.abs(got - want).max() < 1e-13


def _scalar_brute(q, kc, vc, bt, cu, lens, scale):
    """Pure-Python loops: position, gather, softmax, weighted sum."""
    T, H_q, D = q.shape
    K, H_kv = kc.shape[1], kc.shape[2]
    G = H_q // H_kv
    out = [[[0.0] * D for _ in range(H_q)] for _ in range(T)]
    for s in range(len(lens)):
        n = int(cu[s + 1] - cu[s])
        for i in range(n):
            t = int(cu[s]) + i
            last = lens[s] - n + i
            for h in range(H_q):
                j = h // G
                zs = []
                for x in range(last + 1):
                    b = int(bt[s][x // K])
                    z = sum(float(q[t, h, d]) * float(kc[b, x % K, j, d]) for d in range(D))
                    zs.append(z * scale)
                m = max(zs)
                ws = [math.exp(z - m) for z in zs]
                tot = sum(ws)
                for d in range(D):
                    acc = 0.0
                    for x in range(last + 1):
                        b = int(bt[s][x // K])
                        acc += ws[x] * float(vc[b, x % K, j, d])
                    out[t][h][d] = acc / tot
    return np.array(out)


def test_scalar_brute_force():
    rng = np.random.default_rng(2)
    lens, news = [7, 3, 10], [3, 3, 1]          # a fresh prompt (n = L), a chunk, a decode
    q, kc, vc, bt, cu = _problem(rng, lens, news, D=3)
    got = P.paged_attention_prefill(q, kc, vc, bt, cu, lens, 0.7, "f32")
    assert np.abs(got - _scalar_brute(q, kc, vc, bt, cu, lens, 0.7)).max() < 1e-12


def test_causality_and_sensitivity():
    rng = np.random.default_rng(3)
    lens, news = [11], [5]
    q, kc, vc, bt, cu = _problem(rng, lens, news)
    base = P.paged_attention_prefill(q, kc, vc, bt, cu, lens, 0.5, "f32")
    pos = P.query_positions(cu, lens)
    assert pos.tolist() == [6, 7, 8, 9, 10]
    K = kc.shape[1]
    for x in range(11):                          # change the token at position x
        k2, v2 = kc.copy(), vc.copy()
        b = bt[0][x // K]
        k2[b, x % K] += 1.0
        v2[b, x % K] -= 2.0
        out = P.paged_attention_prefill(q, k2, v2, bt, cu, lens, 0.5, "f32")
        for t in range(5):
            changed = np.abs(out[t] - base[t]).max() > 1e-9
            assert changed == (x <= pos[t]), (x, t)


def test_chunked_equals_one_shot():
    """A 10-token prompt as one prefill, and as chunks of 4 then 6 over the
    same cache: the same rows."""
    rng = np.random.default_rng(4)
    q, kc, vc, bt, cu = _problem(rng, [10], [10])
    one = P.paged_attention_prefill(q, kc, vc, bt, cu, [10], 0.3, "f32")
    a = P.paged_attention_prefill(q[:4], kc, vc, bt, [0, 4], [4], 0.3, "f32")
    b = P.paged_attention_prefill(q[4:], kc, vc, bt, [0, 6], [10], 0.3, "f32")
    assert np.abs(np.concatenate([a, b]) - one).max() < 1e-13


def test_closed_forms():
    rng = np.random.default_rng(5)
    q, kc, vc, bt, cu = _problem(rng, [6], [6])
    out = P.paged_attention_prefill(q, kc, vc, bt, cu, [6], 0.9, "f32")
    b0 = bt[0][0]
    # the first token of a fresh prompt sees only itself: its V row, exactly
    for h in range(4):
        assert np.array_equal(out[0, h], vc[b0, 0, h // 2].astype(np.float64))
    # q = 0: every row is the mean of the V rows it sees
    out = P.paged_attention_prefill(np.zeros_like(q), kc, vc, bt, cu, [6], 0.9, "f32")
    for t in range(6):
        rows = np.stack([vc[bt[0][x // 4], x % 4, 0] for x in range(t + 1)]).astype(np.float64)
        assert np.abs(out[t, 0] - rows.mean(0)).max() < 1e-14


def test_bad_counts_rejected():
    with pytest.raises(ValueError):
        P.query_positions([0, 5], [4])


def test_planted_mistakes_are_caught(monkeypatch):
    real = P.query_positions

    def exclusive(cu, lens):                 # sees 0 .. p - 1 (and row 0 sees itself)
        return np.maximum(real(cu, lens) - 1, 0)

    def from_start(cu, lens):                # positions 0 .. n - 1, ignoring the cache
        cu = np.asarray(cu)
        return np.concatenate([np.arange(cu[s + 1] - cu[s]) for s in range(len(cu) - 1)])

    for wrong in (exclusive, from_start):
        monkeypatch.setattr(P, "query_positions", wrong)
        with pytest.raises(AssertionError):
            test_scalar_brute_force()
        monkeypatch.setattr(P, "query_positions", real)

    real_decode = P.decode

    def swapped_heads(x, dtype):             # query head h reads h mod H_kv
        y = real_decode(x, dtype)
        return y[:, [0, 2, 1, 3], :] if y.ndim == 3 and y.shape[1] == 4 else y
    monkeypatch.setattr(P, "decode", swapped_heads)
    with pytest.raises(AssertionError):
        test_scalar_brute_force()
