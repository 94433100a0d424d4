"""Exact softmax attention in fp64 -- the definition the method must reproduce.

ChunkAttention's two-phase partition (Knowl 2) with partial_attn / attn_reduce
(Knowl 3) composes to plain softmax attention over each sequence's whole KV.
Knowl 3 writes the scores as Q K^T without a scale; the textbook definition on
the CachedAttention page ("Load-bearing equations") divides by sqrt(d_K), and
that is the reading taken here: scores = q . k / sqrt(d).

Grouped-query attention is not on the pages.  Query head h reads KV head
floor(h * Hkv / Hq): heads are split into Hkv contiguous groups of g = Hq/Hkv.

Inputs are numpy arrays already rounded to the workload dtype; they are
up-cast exactly to float64 here.
"""
from __future__ import annotations

import math
from typing import List, Sequence, Tuple

import numpy as np


def kv_head_of(h: int, n_q_heads: int, n_kv_heads: int) -> int:
    """KV head read by query head ``h`` (contiguous groups)."""
    return h * n_kv_heads // n_q_heads


def attend(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """softmax(q k^T * scale) v for one query row.

    q: [d]; k, v: [n][d] (n >= 1).  Max-subtracted before exponentiation.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    s = (k @ q) * scale
    m = np.max(s)
    e = np.exp(s - m)
    return (e @ v) / np.sum(e)


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)


def decode_attention(seq_kv: Sequence[Tuple[np.ndarray, np.ndarray]], q: np.ndarray,
                     scale: float | None = None) -> np.ndarray:
    """Decode attention for a batch, every sequence over its own full KV.

    seq_kv: per batch row u, (K_u, V_u) each [n_u][Hkv][d] -- the rows the
            caller supplied for every token of the sequence, in position order,
            with no sharing.
    q:      [B][Hq][d], row u belongs to seq_kv[u].
    Returns [B][Hq][d] float64.  The query attends to all n_u cached tokens
    (its own token's K/V is appended before attention; no mask in decode).
    """
    q = np.asarray(q, dtype=np.float64)
    b, hq, d = q.shape
    if scale is None:
        scale = default_scale(d)
    out = np.empty((b, hq, d), dtype=np.float64)
    for u in range(b):
        k_u, v_u = seq_kv[u]
        k_u = np.asarray(k_u, dtype=np.float64)
        v_u = np.asarray(v_u, dtype=np.float64)
        hkv = k_u.shape[1]
        for h in range(hq):
            kv = kv_head_of(h, hq, hkv)
            out[u, h] = attend(q[u, h], k_u[:, kv, :], v_u[:, kv, :], scale)
    return out


def decode_rows(seq_kv: Sequence[Tuple[np.ndarray, np.ndarray]], q: np.ndarray,
                rows: List[Tuple[int, int]], scale: float | None = None) -> np.ndarray:
    """Like ``decode_attention`` but only for the listed (u, h) rows -> [len(rows)][d]."""
    q = np.asarray(q, dtype=np.float64)
    _, hq, d = q.shape
    if scale is None:
        scale = default_scale(d)
    out = np.empty((len(rows), d), dtype=np.float64)
    for i, (u, h) in enumerate(rows):
        k_u = np.asarray(seq_kv[u][0], dtype=np.float64)
        v_u = np.asarray(seq_kv[u][1], dtype=np.float64)
        kv = kv_head_of(h, hq, k_u.shape[1])
        out[i] = attend(q[u, h], k_u[:, kv, :], v_u[:, kv, :], scale)
    return out


def prefill_attention(k_all: np.ndarray, v_all: np.ndarray, q_blk: np.ndarray, p0: int,
                      scale: float | None = None) -> np.ndarray:
    """Causal attention of a W-row query block at absolute positions [p0, p0+W).

    k_all, v_all: [>= p0+W][Hkv][d] -- the sequence's cache after the block's
    own rows were appended (Chunked Prefill, section 1: the cache is
    append-only).  Row t sees keys [0, p0 + t] (section 2: the causal mask).
    Returns [W][Hq][d] float64.
    """
    q_blk = np.asarray(q_blk, dtype=np.float64)
    w, hq, d = q_blk.shape
    if scale is None:
        scale = default_scale(d)
    k_all = np.asarray(k_all, dtype=np.float64)
    v_all = np.asarray(v_all, dtype=np.float64)
    hkv = k_all.shape[1]
    out = np.empty((w, hq, d), dtype=np.float64)
    for t in range(w):
        n_vis = p0 + t + 1
        for h in range(hq):
            kv = kv_head_of(h, hq, hkv)
            out[t, h] = attend(q_blk[t, h], k_all[:n_vis, kv, :], v_all[:n_vis, kv, :], scale)
    return out


def chunked_prefill(k_all: np.ndarray, v_all: np.ndarray, q_all: np.ndarray, p0: int,
                    blocks: Sequence[int], scale: float | None = None) -> np.ndarray:
    """Run a prompt of sum(blocks) rows as consecutive causal blocks.

    Block b covers absolute positions [p0 + off_b, p0 + off_b + W_b); only the
    cache rows up to the block's end are handed to it, as in an append-only
    cache that the block has just extended.
    """
    outs = []
    off = 0
    for w in blocks:
        end = p0 + off + w
        outs.append(prefill_attention(k_all[:end], v_all[:end], q_all[off:off + w], p0 + off, scale))
        off += w
    return np.concatenate(outs, axis=0)
