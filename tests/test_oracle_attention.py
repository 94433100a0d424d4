"""Pins for oracle.attention: library routine, brute force, closed forms.

The definition softmax(q K^T / sqrt(d)) V (CachedAttention page, "Load-bearing
equations"; ChunkAttention, Knowl 3) is checked against torch's own
scaled_dot_product_attention in float64 on the CPU (including its GQA head
mapping and an explicit causal mask), against a 50-digit mpmath evaluation that
skips the max subtraction, and against closed forms.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _sdpa(q, k, v, mask=None, gqa=False):
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
        attn_mask=None if mask is None else torch.from_numpy(mask), enable_gqa=gqa).numpy()


@pytest.mark.parametrize("hq,hkv", [(1, 1), (4, 4), (4, 2), (8, 1), (32, 8)])
def test_decode_matches_torch_sdpa_fp64(hq, hkv):
    rng = np.random.default_rng(hq * 10 + hkv)
    d = 16
    lens = [1, 7, 33, 64]
    seq_kv = [(_rand(rng, n, hkv, d), _rand(rng, n, hkv, d)) for n in lens]
    q = _rand(rng, len(lens), hq, d)
    got = A.decode_attention(seq_kv, q)
    for u, (k, v) in enumerate(seq_kv):
        ref = _sdpa(q[u][:, None, :], k.transpose(1, 0, 2).copy(), v.transpose(1, 0, 2).copy(), gqa=hq != hkv)
        np.testing.assert_allclose(got[u], ref[:, 0, :], rtol=0, atol=1e-13)


def test_decode_rows_matches_full():
    rng = np.random.default_rng(5)
    seq_kv = [(_rand(rng, n, 2, 8), _rand(rng, n, 2, 8)) for n in (3, 9)]
    q = _rand(rng, 2, 4, 8)
    full = A.decode_attention(seq_kv, q)
    rows = [(1, 3), (0, 0), (1, 1)]
    got = A.decode_rows(seq_kv, q, rows)
    for i, (u, h) in enumerate(rows):
        assert np.array_equal(got[i], full[u, h])


@pytest.mark.parametrize("p0,w,hq,hkv", [(0, 5, 2, 2), (7, 4, 4, 2), (64, 9, 4, 1)])
def test_prefill_matches_torch_sdpa_causal(p0, w, hq, hkv):
    rng = np.random.default_rng(p0 + w)
    d = 8
    k = _rand(rng, p0 + w, hkv, d)
    v = _rand(rng, p0 + w, hkv, d)
    q = _rand(rng, w, hq, d)
    got = A.prefill_attention(k, v, q, p0)
    mask = np.zeros((w, p0 + w), dtype=bool)
    for t in range(w):
        mask[t, :p0 + t + 1] = True
    ref = _sdpa(q.transpose(1, 0, 2).copy(), k.transpose(1, 0, 2).copy(), v.transpose(1, 0, 2).copy(),
                mask=mask, gqa=hq != hkv)
    np.testing.assert_allclose(got, ref.transpose(1, 0, 2), rtol=0, atol=1e-13)


def test_brute_force_mpmath():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    rng = np.random.default_rng(11)
    for n, d in [(1, 1), (2, 3), (5, 4), (6, 2)]:
        q = _rand(rng, d) * 3
        k = _rand(rng, n, d)
        v = _rand(rng, n, d)
        got = A.attend(q, k, v, 1 / math.sqrt(d))
        sc = 1 / mpmath.sqrt(d)
        w = [mpmath.exp(sum(mpmath.mpf(q[i]) * mpmath.mpf(k[t, i]) for i in range(d)) * sc) for t in range(n)]
        z = sum(w)
        for i in range(d):
            ref = sum(w[t] * mpmath.mpf(v[t, i]) for t in range(n)) / z
            assert abs(float(ref) - got[i]) < 1e-14


def test_closed_forms():
    rng = np.random.default_rng(3)
    d, n = 8, 11
    k = _rand(rng, n, d)
    v = _rand(rng, n, d)
    # q = 0: uniform weights -> mean of V
    np.testing.assert_allclose(A.attend(np.zeros(d), k, v, 0.3), v.mean(axis=0), atol=1e-14)
    # one key: output is that key's value
    np.testing.assert_allclose(A.attend(_rand(rng, d), k[:1], v[:1], 0.3), v[0], atol=0)
    # all keys equal: mean of V
    np.testing.assert_allclose(A.attend(_rand(rng, d), np.repeat(k[:1], n, 0), v, 0.3), v.mean(0), atol=1e-14)
    # key t = lambda * q dominates all others -> V_t
    q = _rand(rng, d)
    k2 = k.copy()
    k2[4] = 200.0 * q
    np.testing.assert_allclose(A.attend(q, k2, v, 1.0), v[4], atol=1e-12)
    # two keys: weight of the first is the logistic of the score gap
    q = np.array([1.0, 0.0])
    kk = np.array([[2.0, 0.0], [0.0, 0.0]])
    vv = np.array([[1.0, 0.0], [0.0, 1.0]])
    sig = 1.0 / (1.0 + math.exp(-2.0 / math.sqrt(2.0)))
    np.testing.assert_allclose(A.attend(q, kk, vv, 1 / math.sqrt(2)), [sig, 1 - sig], atol=1e-15)


def test_invariances():
    rng = np.random.default_rng(4)
    d, n = 8, 13
    q, k, v = _rand(rng, d), _rand(rng, n, d), _rand(rng, n, d)
    base = A.attend(q, k, v, 0.5)
    perm = rng.permutation(n)
    np.testing.assert_allclose(A.attend(q, k[perm], v[perm], 0.5), base, atol=1e-14)
    # a common offset added to every key shifts all scores equally
    np.testing.assert_allclose(A.attend(q, k + _rand(rng, d), v, 0.5), base, atol=1e-13)
    # adding a constant vector to every value row adds it to the output
    c = _rand(rng, d)
    np.testing.assert_allclose(A.attend(q, k, v + c, 0.5), base + c, atol=1e-13)


def test_kv_head_mapping_special_cases():
    # g = 1: head h reads KV head h; g = Hq (multi-query): all read head 0
    assert [A.kv_head_of(h, 4, 4) for h in range(4)] == [0, 1, 2, 3]
    assert [A.kv_head_of(h, 8, 1) for h in range(8)] == [0] * 8
    assert [A.kv_head_of(h, 32, 8) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]


def test_chunked_prefill_is_bitwise_single_pass():
    """Chunked Prefill, sections 1-2: W-row causal blocks equal one pass, byte for byte."""
    from oracle.schedule import prefill_blocks
    rng = np.random.default_rng(9)
    p0, n, d = 70, 1137, 8
    k = _rand(rng, p0 + n, 1, d)
    v = _rand(rng, p0 + n, 1, d)
    q = _rand(rng, n, 2, d)
    one = A.prefill_attention(k, v, q, p0)
    for w in (512, 113, 1000):
        blk = A.chunked_prefill(k, v, q, p0, prefill_blocks(n, w))
        assert np.array_equal(one, blk)
