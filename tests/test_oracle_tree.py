"""Pins for oracle.tree and oracle.theory (ChunkAttention, Knowls 1, 4 and 5).

* Closed-form chunk counts and shared-chunk tables for every benchmark tree.
* Contiguity (Knowl 1): every node's covering sequences form one batch range,
  checked by brute force over the paths.
* Prefix match equals a brute-force longest full-chunk agreement with any live
  sequence (insert/remove histories, where no two siblings can be equal).
* Pool accounting: after any history the live chunk count equals the chunks on
  live paths; after removing everything nothing is left.
* Knowl 4 closed forms: per-sequence waste <= c - 1 tokens, i.e. memory loss
  <= (c - 1) / n; the shared/unshared chunk ratio approaches 1 / (1 - r).
* Batch-order tie-breaks on a small hand-worked history.
"""
import math

import numpy as np
import pytest

from oracle import theory as T
from oracle.schedule import prefill_blocks
from oracle.tree import PrefixTree


def _tree_from_levels(levels, c, min_share=2):
    """Token-only tree with the segment structure of ``levels`` (as the workloads build it)."""
    tree = PrefixTree(c, min_share)
    seg = [0]

    def seg_tokens(n):
        seg[0] += 1
        return [32000 + seg[0]] + [7] * (n - 1)

    def grow(depth, prefix):
        n, fan = levels[depth]
        for _ in range(fan):
            toks = prefix + seg_tokens(n)
            if depth + 1 == len(levels):
                tree.insert(toks)
            else:
                grow(depth + 1, toks)
    grow(0, [])
    return tree


SHAPES = {
    # name: (levels, c, shared table summary {(i, j): count}, private chunks per seq, used chunks)
    "tiny": (((128, 1), (32, 4)), 32, {(0, 4): 4}, 1, 8),
    "share1k": (((1024, 1), (512, 32)), 64, {(0, 32): 16}, 8, 272),
    "share4k": (((4096, 1), (512, 64)), 64, {(0, 64): 64}, 8, 576),
    "noshare": (((2048, 64),), 64, {}, 32, 2048),
    "gqa_tree": (((2048, 1), (512, 16), (256, 16)), 64,
                 dict([((0, 256), 32)] + [((16 * b, 16 * b + 16), 8) for b in range(16)]), 4, 32 + 128 + 1024),
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_benchmark_tree_closed_forms(name):
    levels, c, shared_expect, priv, used = SHAPES[name]
    tree = _tree_from_levels(levels, c)
    order, shared, per_seq = tree.canonical_tables()
    got = {}
    for depth, i, j, ntok in shared:
        assert ntok == c
        got[(i, j)] = got.get((i, j), 0) + 1
    assert got == shared_expect
    assert all(sum(1 for _, kind in e if kind == 0) == priv for e in per_seq)
    assert tree.used_chunks() == used
    assert order == list(range(len(order)))


def test_share1k_capacity_matches_formula():
    tree = _tree_from_levels(((1024, 1), (512, 32)), 64)
    assert tree.used_chunks() == T.chunks_shared(32, 1536, 1024, 64) == 272
    assert T.chunks_unshared(32, 1536, 64) == 768


def test_capacity_multiplier_limit():
    n_s, n, c = 1024, 1536, 64
    r = T.sharing_ratio(n_s, n)
    target = T.capacity_multiplier(r)
    assert target == pytest.approx(3.0)
    prev = 0.0
    for b in (1, 2, 8, 64, 1024, 1 << 16):
        ratio = T.chunks_unshared(b, n, c) / T.chunks_shared(b, n, n_s, c)
        assert prev <= ratio <= target
        assert target - ratio <= target * (n_s / c) / (b * (n - n_s) / c) + 1e-12
        prev = ratio


@pytest.mark.parametrize("c", [1, 16, 32, 64, 128])
def test_fragmentation_bound(c):
    for n in range(1, 400):
        w = T.wasted_slots(n, c)
        assert 0 <= w <= c - 1
        assert w / n <= T.fragmentation_bound(c, n) + 1e-15
        tree = PrefixTree(c)
        tree.insert(list(range(n)))
        assert tree.used_chunks() * c - n == w


def _covering(tree):
    order, ranges, preorder = tree.node_ranges()
    pos = {sid: u for u, sid in enumerate(order)}
    for node in preorder:
        us = sorted(pos[s] for s, p in tree.paths.items() if any(x is node for x in p))
        i, j = ranges[id(node)]
        assert us == list(range(i, j)), "covering set is not the node's contiguous range"
        assert node.refs == len(us)


def _brute_match(tree, tokens, c):
    best = 0
    for sid in tree.paths:
        st = tree.seq_tokens(sid)
        full = (len(st) // c) * c
        m = 0
        while m + c <= min(full, len(tokens)) and st[m:m + c] == list(tokens[m:m + c]):
            m += c
        best = max(best, m)
    return best


@pytest.mark.parametrize("seed", range(6))
def test_random_histories(seed):
    rng = np.random.default_rng(seed)
    c = int(rng.choice([2, 3, 4]))
    tree = PrefixTree(c, min_share=int(rng.choice([2, 3])))
    prefixes = [list(rng.integers(0, 3, int(rng.integers(0, 12)))) for _ in range(4)]
    for step in range(60):
        op = rng.random()
        if op < 0.55 or not tree.paths:
            toks = prefixes[int(rng.integers(0, 4))] + list(rng.integers(0, 3, int(rng.integers(1, 9))))
            assert tree.match(toks) == _brute_match(tree, toks, c)
            sid, m = tree.insert(toks)
            assert tree.seq_tokens(sid) == [int(t) for t in toks]
        else:
            sid = int(rng.choice(sorted(tree.paths)))
            tree.remove(sid)
        _covering(tree)
        live = {id(n) for p in tree.paths.values() for n in p}
        assert tree.used_chunks() == len(live)
        order = tree.batch_order()
        assert sorted(order) == sorted(tree.paths)
        for sid, ln in tree.lengths.items():
            assert len(tree.paths[sid]) == math.ceil(ln / c)
    for sid in list(tree.paths):
        tree.remove(sid)
    assert tree.used_chunks() == 0 and tree.batch_order() == []


def test_appends_fill_leaf_then_branch():
    c = 4
    tree = PrefixTree(c)
    a, _ = tree.insert([1, 2, 3, 4, 5, 6])
    b, m = tree.insert([1, 2, 3, 4, 5, 6])
    assert m == 4                       # only the full chunk is matched
    assert tree.used_chunks() == 3      # shared chunk + two private partial chunks
    for t in (7, 8):
        tree.append(a, t)
    assert tree.used_chunks() == 3      # leaf of a filled in place
    tree.append(a, 9)
    assert tree.used_chunks() == 4      # new chunk under a's full leaf
    c2, m2 = tree.insert([1, 2, 3, 4, 5, 6, 7, 8, 10])
    assert m2 == 8                      # a chunk that filled by append is matchable
    assert len(tree.paths[c2]) == 3
    d1, _ = tree.insert([9, 9])
    d2, m3 = tree.insert([9, 9, 9, 9, 1])
    assert m3 == 0                      # a partial chunk is never matched, even as a prefix
    assert tree.seq_tokens(d2) == [9, 9, 9, 9, 1] and tree.seq_tokens(d1) == [9, 9]


def test_batch_order_tie_breaks_hand_worked():
    """Reading of the depth-first order: sequences ending at a node come first
    (by id), then children in creation order."""
    c = 2
    tree = PrefixTree(c)
    s0, _ = tree.insert([1, 1, 2, 2])        # root R=[1,1] -> X=[2,2]
    s1, _ = tree.insert([1, 1, 3])           # R -> Y=[3]
    s2, _ = tree.insert([1, 1])              # ends at R
    s3, _ = tree.insert([1, 1, 2, 2, 4])     # X -> Z=[4]
    s4, _ = tree.insert([5, 5])              # second root
    s5, _ = tree.insert([1, 1, 2, 2])        # ends at X
    assert tree.batch_order() == [s2, s0, s5, s3, s1, s4]
    order, shared, per_seq = tree.canonical_tables()
    # R covers s2,s0,s5,s3,s1 -> [0,5); X covers s0,s5,s3 -> [1,4)
    assert shared == [(0, 0, 5, 2), (1, 1, 4, 2)]
    assert per_seq[0] == [(0, 1)]
    assert per_seq[3] == [(0, 1), (1, 1), (2, 0)]
    tree.remove(s0)
    assert tree.batch_order() == [s2, s5, s3, s1, s4]


def test_prefill_split_golden():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "prefill_splits.txt")
    rows = [l for l in open(path) if l.strip() and not l.startswith("#")]
    assert len(rows) == 2
    for line in rows:
        lhs, rhs = line.split("->")
        n, w = map(int, lhs.split())
        assert prefill_blocks(n, w) == list(map(int, rhs.split()))
    assert prefill_blocks(512, 512) == [512]
    assert prefill_blocks(5, 512) == [5]
    assert prefill_blocks(0, 512) == []


def test_min_share_threshold():
    """Knowl 2: phase 1 takes chunks covered by multiple sequences -- two is enough."""
    for min_share, expect in ((2, [(0, 0, 2, 2)]), (3, [])):
        tree = PrefixTree(2, min_share)
        tree.insert([1, 1, 2])
        tree.insert([1, 1, 3])
        assert tree.canonical_tables()[1] == expect
