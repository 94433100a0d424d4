"""The two-phase partition (TPP) decode algorithm, replayed over the tree model.

ChunkAttention, Knowl 2 (algorithm) and Knowl 3 (equations), in their order:

Phase 1 (chunk-first): for every chunk covered by several sequences, take the
stacked queries of its batch range [i, j) and compute partial_attn against the
chunk's K/V; keep (O, m, n) per row.
Phase 2 (sequence-first): per sequence u, start from o = 0, m = -inf, n = 0;
fold in the saved partial rows of every shared chunk on its path (root to
leaf) with attn_reduce; then, for each of its own chunks, partial_attn of q_u
and attn_reduce; finally O_u = o_u / n_u.

The 1/sqrt(d) scale is applied to the scores before the row max (the reading
taken in ``oracle.attention``).  With GQA, the rows of a KV head are the
(sequence, query head) pairs of its group, sequence-major.
"""
from __future__ import annotations

import math
from typing import Dict, Tuple

import numpy as np

from .attention import kv_head_of


def partial_attn(q_rows: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float):
    """Knowl 3: W = Q K^T (scaled); m = rowmax W; E = exp(W - m); n = rowsum E; O = E V.

    q_rows: [r][d]; k, v: [c][d].  Returns (O [r][d], m [r], n [r]).
    """
    w = (np.asarray(q_rows, np.float64) @ np.asarray(k, np.float64).T) * scale
    m = np.max(w, axis=1)
    e = np.exp(w - m[:, None])
    n = np.sum(e, axis=1)
    o = e @ np.asarray(v, np.float64)
    return o, m, n


def attn_reduce(o_c, m_c, n_c, o_u, m_u, n_u):
    """Knowl 3 online-softmax merge of a chunk partial (o_c, m_c, n_c) into (o_u, m_u, n_u).

    x = exp(m_c - max), y = exp(m_u - max); o = x o_c + y o_u; n = x n_c + y n_u;
    m = max.  When the running max is still -inf (nothing merged yet) its
    weight y is 0.
    """
    mx = max(m_c, m_u)
    x = math.exp(m_c - mx)
    y = 0.0 if m_u == -math.inf else math.exp(m_u - mx)
    return x * o_c + y * o_u, mx, x * n_c + y * n_u


def tpp_decode(tree, q: np.ndarray, n_kv_heads: int, scale: float | None = None) -> np.ndarray:
    """Decode attention for every live sequence of ``tree`` by the two-phase algorithm.

    q: [B][Hq][d] in the tree's batch order.  The tree must carry K/V rows.
    """
    q = np.asarray(q, np.float64)
    b, hq, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    g = hq // n_kv_heads
    order, ranges, preorder = tree.node_ranges()
    assert len(order) == b

    # Phase 1: chunk-first over shared chunks.
    saved: Dict[Tuple[int, int, int], Tuple[np.ndarray, float, float]] = {}
    for node in preorder:
        i, j = ranges[id(node)]
        if not tree.is_shared((i, j)):
            continue
        k_c = np.stack(node.k)  # [c][Hkv][d]
        v_c = np.stack(node.v)
        for kv in range(n_kv_heads):
            rows = [(u, kv * g + hg) for u in range(i, j) for hg in range(g)]
            q_rows = np.stack([q[u, h] for (u, h) in rows])
            o, m, n = partial_attn(q_rows, k_c[:, kv, :], v_c[:, kv, :], scale)
            for r, (u, h) in enumerate(rows):
                saved[(id(node), u, h)] = (o[r], float(m[r]), float(n[r]))

    # Phase 2: sequence-first.
    out = np.empty((b, hq, d), np.float64)
    for u, sid in enumerate(order):
        path = tree.paths[sid]
        for h in range(hq):
            kv = kv_head_of(h, hq, n_kv_heads)
            o_u, m_u, n_u = np.zeros(d), -math.inf, 0.0
            for node in path:
                if tree.is_shared(ranges[id(node)]):
                    o_c, m_c, n_c = saved[(id(node), u, h)]
                else:
                    k_c = np.stack(node.k)[:, kv, :]
                    v_c = np.stack(node.v)[:, kv, :]
                    o, m, n = partial_attn(q[u, h][None, :], k_c, v_c, scale)
                    o_c, m_c, n_c = o[0], float(m[0]), float(n[0])
                o_u, m_u, n_u = attn_reduce(o_c, m_c, n_c, o_u, m_u, n_u)
            out[u, h] = o_u / n_u
    return out
