"""Independent model of the prefix-aware KV cache (PAKV) tree.

ChunkAttention, Knowl 1: the cached K/V of live sequences form a forest of
chunks of c tokens; each root-to-leaf path is one sequence; the sequences that
pass through a node occupy a contiguous range of batch indices.  Arrival does a
prefix lookup and shares matched chunks, decode appends to the leaf chunk until
it is full, departure prunes the path and frees chunks nobody uses.
Knowl 5: the kernel is driven by (C, i, j) tuples -- a chunk and the batch
range it covers.

Readings where the pages leave a step open (the same ones the library takes):

* Only full chunks are matched or shared, and only by equality of all c token
  ids under an already matched parent; the first matching child in creation
  order wins.  A partial chunk always belongs to one sequence; a chunk that
  fills up by append is not merged with an equal sibling.
* Batch order is a depth-first preorder from a virtual root, children in
  creation order; at each node the sequences whose path ends there come first
  (in sequence-id order), then the children's subtrees.
* Ranges are half-open [i, j), 0-based.
* "Shared" means covered by at least ``min_share`` live sequences (default 2).
* Sequence ids count up from 0 in insertion order and are never reused.
* A node with no live sequence through it is deleted at once.

The model also keeps, per node, the K/V rows that were supplied when its
tokens were written (up-cast to float64) so the two-phase algorithm can be
replayed over the tree in ``oracle.tpp``.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Tuple

import numpy as np


class Node:
    __slots__ = ("parent", "depth", "tokens", "children", "refs", "ending", "k", "v", "serial")

    def __init__(self, parent: Optional["Node"], depth: int, serial: int):
        self.parent = parent
        self.depth = depth
        self.tokens: List[int] = []
        self.children: List[Node] = []
        self.refs = 0
        self.ending: List[int] = []
        self.k: List[np.ndarray] = []  # per token: [Hkv][d]
        self.v: List[np.ndarray] = []
        self.serial = serial


class PrefixTree:
    def __init__(self, chunk_size: int, min_share: int = 2):
        if chunk_size < 1:
            raise ValueError("chunk_size must be positive")
        self.c = chunk_size
        self.min_share = min_share
        self.root = Node(None, -1, -1)
        self.paths: Dict[int, List[Node]] = {}
        self.lengths: Dict[int, int] = {}
        self.next_id = 0
        self._serial = 0

    # ---------------------------------------------------------------- helpers
    def _new_node(self, parent: Node) -> Node:
        node = Node(parent, parent.depth + 1, self._serial)
        self._serial += 1
        parent.children.append(node)
        return node

    def _find_full_child(self, parent: Node, chunk: List[int]) -> Optional[Node]:
        for ch in parent.children:
            if len(ch.tokens) == self.c and ch.tokens == chunk:
                return ch
        return None

    # ------------------------------------------------------------- operations
    def match(self, tokens) -> int:
        """Number of leading tokens covered by existing full chunks."""
        tokens = [int(t) for t in tokens]
        cur, m = self.root, 0
        for k in range(len(tokens) // self.c):
            nxt = self._find_full_child(cur, tokens[k * self.c:(k + 1) * self.c])
            if nxt is None:
                break
            cur, m = nxt, m + self.c
        return m

    def insert(self, tokens, k=None, v=None) -> Tuple[int, int]:
        """Sequence arrival; returns (seq_id, n_matched).

        k, v (optional): [n][Hkv][d] rows for every token; rows below n_matched
        are not read.
        """
        tokens = [int(t) for t in tokens]
        n = len(tokens)
        if n == 0:
            raise ValueError("empty sequence")
        path: List[Node] = []
        cur = self.root
        pos = 0
        while pos + self.c <= n:
            nxt = self._find_full_child(cur, tokens[pos:pos + self.c])
            if nxt is None:
                break
            path.append(nxt)
            cur = nxt
            pos += self.c
        n_matched = pos
        while pos < n:
            node = self._new_node(cur)
            end = min(pos + self.c, n)
            node.tokens = tokens[pos:end]
            if k is not None:
                node.k = [np.asarray(k[t], dtype=np.float64) for t in range(pos, end)]
                node.v = [np.asarray(v[t], dtype=np.float64) for t in range(pos, end)]
            path.append(node)
            cur = node
            pos = end
        for node in path:
            node.refs += 1
        sid = self.next_id
        self.next_id += 1
        self.paths[sid] = path
        self.lengths[sid] = n
        path[-1].ending.append(sid)
        return sid, n_matched

    def append(self, sid: int, token: int, k_row=None, v_row=None) -> None:
        """One decode step's token: into the leaf if it has room, else a new chunk."""
        path = self.paths[sid]
        leaf = path[-1]
        if len(leaf.tokens) < self.c:
            target = leaf
        else:
            target = self._new_node(leaf)
            target.refs = 1
            leaf.ending.remove(sid)
            target.ending.append(sid)
            path.append(target)
        target.tokens.append(int(token))
        if k_row is not None:
            target.k.append(np.asarray(k_row, dtype=np.float64))
            target.v.append(np.asarray(v_row, dtype=np.float64))
        self.lengths[sid] += 1

    def remove(self, sid: int) -> None:
        """Sequence departure: prune the path; chunks nobody covers are freed."""
        path = self.paths.pop(sid)
        del self.lengths[sid]
        path[-1].ending.remove(sid)
        for node in path:
            node.refs -= 1
        for node in path:
            if node.refs == 0 and node in node.parent.children:
                node.parent.children.remove(node)

    # ----------------------------------------------------------------- views
    def live_nodes(self) -> List[Node]:
        out: List[Node] = []

        def walk(n: Node):
            for ch in n.children:
                out.append(ch)
                walk(ch)
        walk(self.root)
        return out

    def batch_order(self) -> List[int]:
        order, _ = self._dfs()
        return order

    def _dfs(self):
        order: List[int] = []
        ranges: Dict[int, Tuple[int, int]] = {}
        preorder: List[Node] = []

        def visit(n: Node):
            i = len(order)
            order.extend(sorted(n.ending))
            if n is not self.root:
                preorder.append(n)
            for ch in n.children:
                visit(ch)
            ranges[id(n)] = (i, len(order))
        visit(self.root)
        return order, (ranges, preorder)

    def node_ranges(self):
        """(batch order, {id(node): (i, j)}, nodes in DFS preorder)."""
        order, (ranges, preorder) = self._dfs()
        return order, ranges, preorder

    def is_shared(self, rng: Tuple[int, int]) -> bool:
        return rng[1] - rng[0] >= self.min_share

    def canonical_tables(self):
        """Tables in the canonical, chunk-id-free form.

        Returns (batch order,
                 shared rows: [(depth, i, j, n_tokens)] for every shared node in
                 DFS preorder,
                 per batch row u: [(depth, kind)] root->leaf, kind 1 = shared).
        """
        order, ranges, preorder = self.node_ranges()
        shared = []
        for n in preorder:
            i, j = ranges[id(n)]
            if self.is_shared((i, j)):
                shared.append((n.depth, i, j, len(n.tokens)))
        per_seq = []
        for sid in order:
            per_seq.append([(n.depth, 1 if self.is_shared(ranges[id(n)]) else 0) for n in self.paths[sid]])
        return order, shared, per_seq

    def used_chunks(self) -> int:
        return len(self.live_nodes())

    def unique_tokens(self) -> int:
        return sum(len(n.tokens) for n in self.live_nodes())

    def seq_tokens(self, sid: int) -> List[int]:
        out: List[int] = []
        for n in self.paths[sid]:
            out.extend(n.tokens)
        return out

    def seq_kv(self, sid: int) -> Tuple[np.ndarray, np.ndarray]:
        ks, vs = [], []
        for n in self.paths[sid]:
            ks.extend(n.k)
            vs.extend(n.v)
        return np.stack(ks), np.stack(vs)
