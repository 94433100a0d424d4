"""Seeded synthetic workloads shaped like the ChunkAttention microkernel benchmarks.

This module only draws random numbers and token ids; it holds none of the
method's arithmetic.  Both the CUDA path (through the tests and ``bench.py``)
and the CPU oracle consume what it produces.

A workload is a prefix tree of *segments*.  ``levels`` lists, root first, the
token count of each segment at that depth and how many children every segment
of the level above has (the first level's fan-out is the number of roots).
Every root-to-leaf path is one sequence; sequences are numbered in depth-first
order of their leaves, which is also their insertion order.

Recipe (one ``torch.Generator`` seeded with ``seed``; draws happen in this
order, segments visited depth-first in creation order):

* per segment: token ids uniform in ``[0, 32000)``, then its first token is
  overwritten with ``32000 + segment index`` so that two different segments can
  never match by accident; then K and V, each ``[n][n_kv_heads][head_dim]``
  standard normal in fp32, rounded once to the workload dtype;
* then Q ``[B][n_q_heads][head_dim]`` standard normal, rounded once;
* then, when a prefill step is configured, the new prompt tokens (first one
  forced unique the same way), their K and V, and the query block rows.

Segment lengths are multiples of the chunk size, so segment boundaries fall on
chunk boundaries and the prefix tree built from the token ids has exactly the
segment structure (ChunkAttention, Knowl 1: the tree is keyed by chunk tokens).

When ``device`` is a CUDA device the draws come from a CUDA generator with the
same seed: values then differ from the CPU draws but are fixed for a given seed
and GPU.  Small workloads are drawn on the CPU so every machine sees the same
numbers.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import torch

TOKEN_VOCAB = 32000

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
DTYPE_CODES = {"f16": 0, "bf16": 1, "f32": 2}


@dataclass(frozen=True)
class WorkloadSpec:
    name: str
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    chunk_size: int
    dtype: str
    levels: Tuple[Tuple[int, int], ...]  # ((tokens, fanout), ...), root level first
    seed: int
    prefill_prompt: int = 0  # new prompt tokens after the first root segment
    prefill_width: int = 0   # W rows per causal query block

    @property
    def n_sequences(self) -> int:
        b = 1
        for _, fan in self.levels:
            b *= fan
        return b

    @property
    def seq_len(self) -> int:
        return sum(n for n, _ in self.levels)

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    def bytes_per_token(self) -> int:
        """K and V bytes of one token over all KV heads."""
        return 2 * self.n_kv_heads * self.head_dim * torch.tensor([], dtype=DTYPES[self.dtype]).element_size()

    def unique_tokens(self) -> int:
        total, mult = 0, 1
        for n, fan in self.levels:
            mult *= fan
            total += mult * n
        return total

    def unique_kv_bytes(self) -> int:
        return self.unique_tokens() * self.bytes_per_token()

    def logical_kv_bytes(self) -> int:
        return self.n_sequences * self.seq_len * self.bytes_per_token()


# The five benchmark shapes.  Seeds are 1000 + index.
SPECS = {
    "tiny": WorkloadSpec("tiny", 1, 1, 64, 32, "f32", ((128, 1), (32, 4)), 1000),
    "share1k": WorkloadSpec("share1k", 32, 32, 128, 64, "f16", ((1024, 1), (512, 32)), 1001),
    "share4k": WorkloadSpec("share4k", 32, 32, 128, 64, "f16", ((4096, 1), (512, 64)), 1002),
    "noshare": WorkloadSpec("noshare", 32, 32, 128, 64, "f16", ((2048, 64),), 1003),
    "gqa_tree": WorkloadSpec("gqa_tree", 32, 8, 128, 64, "bf16", ((2048, 1), (512, 16), (256, 16)), 1004,
                             prefill_prompt=1137, prefill_width=512),
}

DESCRIPTIONS = {
    "tiny": "4 seqs, 1 head, d=64, fp32, 128 shared + 32 private tokens, chunk 32",
    "share1k": "7B-shaped decode attention: 32 heads, d=128, fp16, batch 32, 1024 shared + 512 private, chunk 64",
    "share4k": "32 heads, d=128, fp16, batch 64, 4096 shared + 512 private, chunk 64",
    "noshare": "no-sharing control: 32 heads, d=128, fp16, batch 64, 2048 private, chunk 64",
    "gqa_tree": "GQA 32q/8kv, d=128, bf16, 256 seqs: 2048 root -> 16x512 branches -> 16x256 leaves, chunk 64; "
                "plus a 1137-token prefill in W=512 causal blocks over the root prefix",
}


# Batch-scaling family (ChunkAttention, Knowl 9: n_s = 2048 shared tokens,
# n_c = 64 per sequence, b from 16 to 96): the chunk-first phase's stacked rows
# grow with the batch.
BATCH_FAMILY = tuple(f"batch{b}" for b in (16, 32, 48, 64, 80, 96))
for _b in (16, 32, 48, 64, 80, 96):
    SPECS[f"batch{_b}"] = WorkloadSpec(f"batch{_b}", 32, 32, 128, 64, "f16", ((2048, 1), (64, _b)), 1100 + _b)
    DESCRIPTIONS[f"batch{_b}"] = f"32 heads, d=128, fp16, batch {_b}, 2048 shared + 64 private, chunk 64"

# Divergence family (ChunkAttention, Knowl 8: b = 32, c = 64, fp16, the
# (n_s, n_c) pairs it reports): as completions n_c grow, the shared share of
# the KV cache falls.
DIVERGENCE_GRID = ((1024, 256), (1024, 512), (1024, 1024), (2048, 512), (2048, 1024), (2048, 2048),
                   (4096, 512), (4096, 4096))
DIVERGENCE_FAMILY = tuple(f"div_s{ns}_c{nc}" for ns, nc in DIVERGENCE_GRID)
for _i, (_ns, _nc) in enumerate(DIVERGENCE_GRID):
    _name = f"div_s{_ns}_c{_nc}"
    SPECS[_name] = WorkloadSpec(_name, 32, 32, 128, 64, "f16", ((_ns, 1), (_nc, 32)), 1300 + _i)
    DESCRIPTIONS[_name] = f"32 heads, d=128, fp16, batch 32, {_ns} shared + {_nc} private, chunk 64"

# Head-dim / chunk-size generality (ChunkAttention, Knowl 10: the kernel is
# specialised for common head dims, and porting it to others is listed as a
# limitation): the share1k tree (32 heads, fp16, batch 32, 1024 shared + 512
# private) at d in {64, 128} and c in {16, 32, 64, 128}.
GENERALITY_GRID = tuple((d, c) for d in (128, 64) for c in (16, 32, 64, 128))
GENERALITY_FAMILY = tuple(f"gen_d{d}_c{c}" for d, c in GENERALITY_GRID)
for _i, (_d, _c) in enumerate(GENERALITY_GRID):
    _name = f"gen_d{_d}_c{_c}"
    SPECS[_name] = WorkloadSpec(_name, 32, 32, _d, _c, "f16", ((1024, 1), (512, 32)), 1400 + _i)
    DESCRIPTIONS[_name] = f"32 heads, d={_d}, fp16, batch 32, 1024 shared + 512 private, chunk {_c}"


@dataclass
class Segment:
    index: int
    parent: int          # -1 for a root segment
    depth: int
    tokens: torch.Tensor  # int32 [n]
    k: torch.Tensor       # [n][Hkv][d] workload dtype
    v: torch.Tensor


@dataclass
class Workload:
    spec: WorkloadSpec
    segments: List[Segment]
    seq_paths: List[List[int]]     # per sequence: segment indices root->leaf
    q: torch.Tensor                # [B][Hq][d]
    prefill_tokens: Optional[torch.Tensor] = None  # int32 [prompt]
    prefill_k: Optional[torch.Tensor] = None       # [prompt][Hkv][d]
    prefill_v: Optional[torch.Tensor] = None
    prefill_q: Optional[torch.Tensor] = None       # [prompt][Hq][d]
    extra: dict = field(default_factory=dict)

    def seq_tokens(self, s: int) -> torch.Tensor:
        return torch.cat([self.segments[i].tokens for i in self.seq_paths[s]])

    def seq_k(self, s: int) -> torch.Tensor:
        return torch.cat([self.segments[i].k for i in self.seq_paths[s]])

    def seq_v(self, s: int) -> torch.Tensor:
        return torch.cat([self.segments[i].v for i in self.seq_paths[s]])

    @property
    def n_sequences(self) -> int:
        return len(self.seq_paths)


def _normal(gen: torch.Generator, shape, dtype, device) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32, device=device)
    return x.to(dtype)


def generate(spec: WorkloadSpec, device: str = "cpu", q_scale: float = 1.0) -> Workload:
    """Draw the workload described by ``spec`` (see the module docstring)."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(spec.seed)
    dt = DTYPES[spec.dtype]
    hkv, d = spec.n_kv_heads, spec.head_dim
    segments: List[Segment] = []
    seq_paths: List[List[int]] = []

    def make_segment(parent: int, depth: int) -> int:
        n = spec.levels[depth][0]
        idx = len(segments)
        tok = torch.randint(0, TOKEN_VOCAB, (n,), generator=gen, dtype=torch.int64, device=dev)
        tok[0] = TOKEN_VOCAB + idx
        k = _normal(gen, (n, hkv, d), dt, dev)
        v = _normal(gen, (n, hkv, d), dt, dev)
        segments.append(Segment(idx, parent, depth, tok.to(torch.int32), k, v))
        return idx

    def grow(parent: int, depth: int, path: List[int]) -> None:
        fan = spec.levels[depth][1]
        for _ in range(fan):
            idx = make_segment(parent, depth)
            p = path + [idx]
            if depth + 1 == len(spec.levels):
                seq_paths.append(p)
            else:
                grow(idx, depth + 1, p)

    grow(-1, 0, [])
    b = len(seq_paths)
    q = _normal(gen, (b, spec.n_q_heads, d), dt, dev)
    if q_scale != 1.0:
        q = (q.float() * q_scale).to(dt)
    wl = Workload(spec, segments, seq_paths, q)
    if spec.prefill_prompt:
        n = spec.prefill_prompt
        tok = torch.randint(0, TOKEN_VOCAB, (n,), generator=gen, dtype=torch.int64, device=dev)
        tok[0] = TOKEN_VOCAB + len(segments)
        wl.prefill_tokens = tok.to(torch.int32)
        wl.prefill_k = _normal(gen, (n, hkv, d), dt, dev)
        wl.prefill_v = _normal(gen, (n, hkv, d), dt, dev)
        wl.prefill_q = _normal(gen, (n, spec.n_q_heads, d), dt, dev)
    return wl


def random_tree_spec(seed: int, dtype: str = "f16", head_dim: int = 128, chunk_size: int = 64,
                     n_q_heads: int = 4, n_kv_heads: int = 2) -> WorkloadSpec:
    """A small random multi-level tree (ragged lengths are added by the callers)."""
    g = torch.Generator().manual_seed(seed)
    depth = int(torch.randint(1, 4, (1,), generator=g))
    levels = []
    for lvl in range(depth):
        n = chunk_size * int(torch.randint(1, 4, (1,), generator=g))
        fan = int(torch.randint(1, 4, (1,), generator=g)) if lvl else 1
        levels.append((n, fan))
    return WorkloadSpec(f"rand{seed}", n_q_heads, n_kv_heads, head_dim, chunk_size, dtype, tuple(levels), seed)


def ragged_sequences(seed: int, n_seqs: int, prefix_len: int, tail_lens: List[int], n_kv_heads: int,
                     head_dim: int, dtype: str, n_q_heads: int):
    """Sequences sharing a prefix of ``prefix_len`` tokens with tails of the given (ragged) lengths.

    Returns (tokens list, k list, v list, q) with every sequence's K/V rows for
    its full length; the shared prefix rows are identical across sequences.
    """
    gen = torch.Generator().manual_seed(seed)
    dt = DTYPES[dtype]
    ptok = torch.randint(0, TOKEN_VOCAB, (prefix_len,), generator=gen, dtype=torch.int64)
    pk = _normal(gen, (prefix_len, n_kv_heads, head_dim), dt, "cpu")
    pv = _normal(gen, (prefix_len, n_kv_heads, head_dim), dt, "cpu")
    toks, ks, vs = [], [], []
    for s, n in enumerate(tail_lens[:n_seqs]):
        t = torch.randint(0, TOKEN_VOCAB, (n,), generator=gen, dtype=torch.int64)
        if n:
            t[0] = TOKEN_VOCAB + s
        k = _normal(gen, (n, n_kv_heads, head_dim), dt, "cpu")
        v = _normal(gen, (n, n_kv_heads, head_dim), dt, "cpu")
        toks.append(torch.cat([ptok, t]).to(torch.int32))
        ks.append(torch.cat([pk, k]))
        vs.append(torch.cat([pv, v]))
    q = _normal(gen, (n_seqs, n_q_heads, head_dim), dt, "cpu")
    return toks, ks, vs, q


def insert_all(pool, wl: Workload, stream=None, nan_matched: bool = False, device: str = "cuda"):
    """Insert every sequence of ``wl`` into ``pool`` (insertion order = leaf DFS order).

    Each call passes the sequence's full K/V rows on ``device``; when
    ``nan_matched`` is set, the rows the pool will not read (the matched
    prefix) are overwritten with NaN first.  Returns the sequence ids.
    """
    ids = []
    for s in range(wl.n_sequences):
        toks = wl.seq_tokens(s).cpu()
        k = wl.seq_k(s).to(device)
        v = wl.seq_v(s).to(device)
        if nan_matched:
            m = pool.match(toks)
            if m:
                k = k.clone()
                v = v.clone()
                k[:m] = float("nan")
                v[:m] = float("nan")
        sid, _ = pool.insert(toks, k, v, stream)
        ids.append(sid)
    return ids
