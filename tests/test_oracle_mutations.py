"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin catches each.

Each mutation is applied with monkeypatch to the oracle itself; the pin tests
are then re-run and at least one must fail.
"""
import math

import numpy as np
import pytest

from oracle import attention as A
from oracle import schedule as S
from oracle import theory as T
from oracle import tpp as P
from oracle import tree as TR

from tests import test_oracle_attention as TA
from tests import test_oracle_tpp as TT
from tests import test_oracle_tree as TRT


def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


def test_dropped_scale(monkeypatch):
    monkeypatch.setattr(A, "default_scale", lambda d: 1.0)
    assert _fails(TA.test_decode_matches_torch_sdpa_fp64, 4, 2)


def test_wrong_gqa_mapping(monkeypatch):
    monkeypatch.setattr(A, "kv_head_of", lambda h, hq, hkv: h % hkv)
    assert _fails(TA.test_decode_matches_torch_sdpa_fp64, 4, 2)
    assert _fails(TA.test_kv_head_mapping_special_cases)


def test_swapped_key_value(monkeypatch):
    orig = A.attend
    monkeypatch.setattr(A, "attend", lambda q, k, v, s: orig(q, v, k, s))
    assert _fails(TA.test_decode_matches_torch_sdpa_fp64, 1, 1)


def test_causal_off_by_one(monkeypatch):
    def bad(k_all, v_all, q_blk, p0, scale=None):
        q_blk = np.asarray(q_blk, np.float64)
        w, hq, d = q_blk.shape
        out = np.empty((w, hq, d))
        for t in range(w):
            n_vis = max(1, p0 + t)
            for h in range(hq):
                kv = A.kv_head_of(h, hq, k_all.shape[1])
                out[t, h] = A.attend(q_blk[t, h], k_all[:n_vis, kv], v_all[:n_vis, kv], 1 / math.sqrt(d))
        return out
    monkeypatch.setattr(A, "prefill_attention", bad)
    assert _fails(TA.test_prefill_matches_torch_sdpa_causal, 7, 4, 4, 2)


def test_reduce_wrong_weight(monkeypatch):
    def bad(o_c, m_c, n_c, o_u, m_u, n_u):
        mx = max(m_c, m_u)
        x = math.exp(m_c - mx)
        y = 0.0 if m_u == -math.inf else math.exp(m_c - mx)
        return x * o_c + y * o_u, mx, x * n_c + y * n_u
    monkeypatch.setattr(P, "attn_reduce", bad)
    assert _fails(TT.test_tpp_equals_definition, 4, 2, 4)


def test_partial_attn_missing_max(monkeypatch):
    def bad(q_rows, k, v, scale):
        w = (q_rows @ k.T) * scale
        m = np.max(w, axis=1)
        e = np.exp(w)
        return e @ v, m, np.sum(e, axis=1)
    monkeypatch.setattr(P, "partial_attn", bad)
    assert _fails(TT.test_tpp_equals_definition, 4, 2, 4)


def test_children_visited_in_reverse(monkeypatch):
    orig = TR.PrefixTree._dfs

    def bad(self):
        for n in self.live_nodes() + [self.root]:
            n.children.reverse()
        try:
            return orig(self)
        finally:
            for n in self.live_nodes() + [self.root]:
                n.children.reverse()
    monkeypatch.setattr(TR.PrefixTree, "_dfs", bad)
    assert _fails(TRT.test_batch_order_tie_breaks_hand_worked)


def test_share_threshold_strict(monkeypatch):
    monkeypatch.setattr(TR.PrefixTree, "is_shared", lambda self, rng: rng[1] - rng[0] > self.min_share)
    assert _fails(TRT.test_min_share_threshold)


def test_partial_chunks_matched(monkeypatch):
    def bad(self, parent, chunk):
        for ch in parent.children:
            if ch.tokens == chunk[:len(ch.tokens)]:
                return ch
        return None
    monkeypatch.setattr(TR.PrefixTree, "_find_full_child", bad)
    assert _fails(TRT.test_appends_fill_leaf_then_branch) or _fails(TRT.test_random_histories, 0)


def test_split_evenly(monkeypatch):
    monkeypatch.setattr(S, "prefill_blocks", lambda n, w: [math.ceil(n / math.ceil(n / w))] * math.ceil(n / w))
    monkeypatch.setattr(TRT, "prefill_blocks", S.prefill_blocks)
    assert _fails(TRT.test_prefill_split_golden)


def test_fragmentation_bound_too_tight(monkeypatch):
    monkeypatch.setattr(T, "fragmentation_bound", lambda c, n: (c - 2) / n)
    assert _fails(TRT.test_fragmentation_bound, 16)
