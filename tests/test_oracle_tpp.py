"""Pins for oracle.tpp: the two-phase algorithm against the definition and the
invariants the pages fix (ChunkAttention, Knowls 2-3; Chunked Prefill, section 2).

* TPP over a shared tree equals plain per-sequence attention (1e-12).
* The shared-prefix result equals the unshared one: the same K/V inserted with
  distinct token ids (nothing shared) gives the same output.
* A tree with no shared chunk reduces to per-sequence attention.
* Chunked partial_attn + attn_reduce equals whole-block partial attention for
  every chunk size dividing the length.
* attn_reduce is order independent (up to rounding).
"""
import math

import numpy as np
import pytest

from oracle import attention as A
from oracle.tpp import attn_reduce, partial_attn, tpp_decode
from oracle.tree import PrefixTree


def _build(rng, c, hkv, d, prefix, tails, distinct_tokens=False, min_share=2):
    tree = PrefixTree(c, min_share=min_share)
    ptok = list(rng.integers(0, 1000, prefix))
    pk = rng.standard_normal((prefix, hkv, d))
    pv = rng.standard_normal((prefix, hkv, d))
    seq_kv = []
    for s, n in enumerate(tails):
        tok = ptok + [2000 + 100 * s + t for t in range(n)]
        if distinct_tokens:
            tok = [10_000 * (s + 1) + t for t in range(len(tok))]
        k = np.concatenate([pk, rng.standard_normal((n, hkv, d))])
        v = np.concatenate([pv, rng.standard_normal((n, hkv, d))])
        tree.insert(tok, k, v)
        seq_kv.append((k, v))
    return tree, seq_kv


@pytest.mark.parametrize("hq,hkv", [(1, 1), (4, 2), (8, 1)])
@pytest.mark.parametrize("c", [4, 8])
def test_tpp_equals_definition(hq, hkv, c):
    rng = np.random.default_rng(hq + 7 * c)
    d = 8
    tree, seq_kv = _build(rng, c, hkv, d, prefix=3 * c, tails=[5, c, 2 * c + 3, 1])
    order = tree.batch_order()
    q = rng.standard_normal((len(order), hq, d))
    got = tpp_decode(tree, q, hkv)
    ref = A.decode_attention([seq_kv[s] for s in order], q)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_tpp_multilevel_with_appends_and_removes():
    rng = np.random.default_rng(21)
    c, hkv, d, hq = 4, 2, 8, 4
    tree = PrefixTree(c)
    kv = {}
    base = list(rng.integers(0, 50, 8))
    bk, bv = rng.standard_normal((8, hkv, d)), rng.standard_normal((8, hkv, d))
    for s in range(6):
        mid = [100 + (s // 2)] * 4
        mk = rng.standard_normal((4, hkv, d)) if s % 2 == 0 else kv[s - 1][0][8:12]
        mv = rng.standard_normal((4, hkv, d)) if s % 2 == 0 else kv[s - 1][1][8:12]
        tail = list(rng.integers(0, 50, 3 + s))
        tail[0] = 500 + s
        tk, tv = rng.standard_normal((len(tail), hkv, d)), rng.standard_normal((len(tail), hkv, d))
        k = np.concatenate([bk, mk, tk])
        v = np.concatenate([bv, mv, tv])
        sid, _ = tree.insert(base + mid + tail, k, v)
        kv[sid] = (k, v)
    for step in range(7):
        for sid in list(tree.paths):
            kr, vr = rng.standard_normal((hkv, d)), rng.standard_normal((hkv, d))
            tree.append(sid, 900 + step, kr, vr)
            kv[sid] = (np.concatenate([kv[sid][0], kr[None]]), np.concatenate([kv[sid][1], vr[None]]))
        if step == 3:
            tree.remove(2)
    order = tree.batch_order()
    q = rng.standard_normal((len(order), hq, d))
    got = tpp_decode(tree, q, hkv)
    ref = A.decode_attention([kv[s] for s in order], q)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_shared_equals_unshared():
    rng1 = np.random.default_rng(5)
    rng2 = np.random.default_rng(5)
    c, hkv, d, hq = 4, 2, 8, 4
    t_shared, kv_s = _build(rng1, c, hkv, d, 12, [3, 6, 4])
    t_plain, kv_p = _build(rng2, c, hkv, d, 12, [3, 6, 4], distinct_tokens=True)
    assert len(t_shared.canonical_tables()[1]) > 0
    assert len(t_plain.canonical_tables()[1]) == 0
    for a, b in zip(kv_s, kv_p):
        assert np.array_equal(a[0], b[0])
    q = np.random.default_rng(6).standard_normal((3, hq, d))
    # insertion order == batch order in both trees (no sequence ends inside the prefix)
    assert t_shared.batch_order() == t_plain.batch_order() == [0, 1, 2]
    np.testing.assert_allclose(tpp_decode(t_shared, q, hkv), tpp_decode(t_plain, q, hkv), rtol=0, atol=1e-12)


def test_no_sharing_reduces_to_per_sequence():
    rng = np.random.default_rng(8)
    c, hkv, d, hq = 4, 1, 8, 1
    tree, seq_kv = _build(rng, c, hkv, d, 8, [1, 2, 9], min_share=10**9)
    assert tree.canonical_tables()[1] == []
    q = rng.standard_normal((3, hq, d))
    got = tpp_decode(tree, q, hkv)
    for u, s in enumerate(tree.batch_order()):
        np.testing.assert_allclose(got[u, 0], A.attend(q[u, 0], seq_kv[s][0][:, 0], seq_kv[s][1][:, 0], 1 / math.sqrt(d)),
                                   atol=1e-12)


@pytest.mark.parametrize("c", [1, 2, 3, 4, 6, 12])
def test_chunked_equals_whole_block(c):
    rng = np.random.default_rng(c)
    n, d, r = 12, 8, 3
    q, k, v = rng.standard_normal((r, d)), rng.standard_normal((n, d)), rng.standard_normal((n, d))
    o_w, m_w, n_w = partial_attn(q, k, v, 0.4)
    for row in range(r):
        o, m, s = np.zeros(d), -math.inf, 0.0
        for start in range(0, n, c):
            oc, mc, nc = partial_attn(q[row:row + 1], k[start:start + c], v[start:start + c], 0.4)
            o, m, s = attn_reduce(oc[0], float(mc[0]), float(nc[0]), o, m, s)
        assert m == pytest.approx(m_w[row], rel=1e-14, abs=1e-14)
        np.testing.assert_allclose(o / s, o_w[row] / n_w[row], rtol=0, atol=1e-13)
        np.testing.assert_allclose(s, n_w[row], rtol=1e-13)


def test_attn_reduce_order_independent():
    rng = np.random.default_rng(12)
    d = 16
    parts = []
    for _ in range(9):
        q, k, v = rng.standard_normal((1, d)), rng.standard_normal((5, d)), rng.standard_normal((5, d))
        o, m, n = partial_attn(q * rng.uniform(0.1, 4), k, v, 1.0)
        parts.append((o[0], float(m[0]), float(n[0])))
    outs = []
    for _ in range(20):
        o, m, s = np.zeros(d), -math.inf, 0.0
        for i in rng.permutation(len(parts)):
            o, m, s = attn_reduce(*parts[i], o, m, s)
        outs.append(o / s)
    for x in outs[1:]:
        np.testing.assert_allclose(x, outs[0], rtol=1e-13, atol=1e-15)


def test_attn_reduce_first_merge_from_empty():
    o, m, s = attn_reduce(np.array([2.0, 4.0]), 1.5, 2.0, np.zeros(2), -math.inf, 0.0)
    assert m == 1.5 and s == 2.0 and np.array_equal(o, [2.0, 4.0])
