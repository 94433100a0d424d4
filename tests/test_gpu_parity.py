"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Tolerances: max |gpu - oracle| <= 2e-3 for fp16/bf16
K/V, <= 1e-5 for fp32.  Outputs are rounded to the pool dtype, so cases with
large outputs (a handful of keys) add half an output ulp at |oracle| to the
bound: rounding the exact answer to bf16 alone can exceed 2e-3 once |o| > 0.5.
Byte work (K/V scatter into the chunk pool) is checked bit-exactly.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle.schedule import prefill_blocks
from prefix_shared_kv_tree_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"f16": 2e-3, "bf16": 2e-3, "f32": 1e-5}
ULP_BITS = {"f16": 10, "bf16": 7, "f32": 23}


@pytest.fixture(scope="module")
def pst():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from prefix_shared_kv_tree_gb300 import build
    build.build_library()
    from prefix_shared_kv_tree_gb300 import pst as mod
    return mod


def _f64(t):
    return t.detach().float().cpu().double().numpy()


def _bound(ref, dtype, with_ulp):
    tol = TOL[dtype]
    if not with_ulp:
        return tol
    mag = np.maximum(np.abs(ref), 1e-30)
    half_ulp = 0.5 * 2.0 ** (np.floor(np.log2(mag)) - ULP_BITS[dtype])
    return tol + half_ulp


def _assert_close(got, ref, dtype, with_ulp=False, what=""):
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref)
    bound = _bound(ref, dtype, with_ulp)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    bad = err > bound
    assert not bad.any(), f"{what}: max err {err.max():.3e} (bound {np.max(bound):.3e}) at {np.argwhere(bad)[:3]}"
    return float(err.max())


def _pool(pst, spec, max_chunks=None, min_share=0, flags=0):
    if max_chunks is None:
        max_chunks = W_chunks(spec) + 64
    return pst.Pool(spec.n_q_heads, spec.n_kv_heads, spec.head_dim, spec.chunk_size, max_chunks, spec.dtype,
                    min_share, 0, flags, device=0)


def W_chunks(spec):
    total, mult = 0, 1
    for n, fan in spec.levels:
        mult *= fan
        total += mult * math.ceil(n / spec.chunk_size)
    return total


def _decode(pool, q):
    out = torch.empty_like(q)
    pool.decode_attention(q, out)
    torch.cuda.synchronize()
    assert pool.check_device() == 0
    return out


# --------------------------------------------------------------- byte work
@pytest.mark.parametrize("dtype,d,c", [("f16", 128, 64), ("bf16", 64, 64), ("f32", 64, 32), ("f16", 64, 32)])
def test_scatter_gather_bit_exact(pst, dtype, d, c):
    g = torch.Generator().manual_seed(7)
    hkv = 2
    pool = pst.Pool(4, hkv, d, c, 64, dtype, 0, 0, 0, device=0)
    dt = W.DTYPES[dtype]
    seqs = {}
    prefix = torch.randint(0, 100, (2 * c,), generator=g, dtype=torch.int32)
    pk = torch.randn(2 * c, hkv, d, generator=g).to(dt)
    pv = torch.randn(2 * c, hkv, d, generator=g).to(dt)
    for s, tail in enumerate([1, c - 1, c, 2 * c + 5, 0]):
        toks = torch.cat([prefix, torch.arange(tail, dtype=torch.int32) + 1000 * (s + 1)])
        k = torch.cat([pk, torch.randn(tail, hkv, d, generator=g).to(dt)])
        v = torch.cat([pv, torch.randn(tail, hkv, d, generator=g).to(dt)])
        sid, _ = pool.insert(toks, k.cuda(), v.cuda())
        seqs[sid] = (k, v)
    for step in range(c + 3):  # appends cross chunk boundaries
        ids = sorted(seqs)
        k = torch.randn(len(ids), hkv, d, generator=g).to(dt)
        v = torch.randn(len(ids), hkv, d, generator=g).to(dt)
        pool.append_batch(ids, [5] * len(ids), k.cuda(), v.cuda())
        for i, sid in enumerate(ids):
            seqs[sid] = (torch.cat([seqs[sid][0], k[i:i + 1]]), torch.cat([seqs[sid][1], v[i:i + 1]]))
    for sid, (k, v) in seqs.items():
        n = pool.seq_length(sid)
        assert n == k.shape[0]
        ko = torch.empty(n, hkv, d, dtype=dt, device="cuda")
        vo = torch.empty_like(ko)
        pool.gather_kv(sid, ko, vo)
        torch.cuda.synchronize()
        assert torch.equal(ko.cpu().view(torch.uint8), k.view(torch.uint8))
        assert torch.equal(vo.cpu().view(torch.uint8), v.view(torch.uint8))


# ------------------------------------------------------------- small trees
def test_tiny_config_all_rows(pst):
    spec = W.SPECS["tiny"]
    wl = W.generate(spec)
    pool = _pool(pst, spec)
    W.insert_all(pool, wl)
    assert pool.batch_order() == list(range(4))
    out = _decode(pool, wl.q.cuda())
    ref = A.decode_attention([(_f64(wl.seq_k(s)), _f64(wl.seq_v(s))) for s in range(4)], _f64(wl.q))
    _assert_close(_f64(out), ref, "f32", what="tiny")


CASES = [
    # dtype, Hq, Hkv, d, c, flags, min_share
    ("f16", 4, 4, 128, 64, 0, 0),
    ("f16", 4, 1, 128, 64, 0, 0),
    ("bf16", 8, 2, 128, 64, 0, 0),
    ("bf16", 8, 1, 64, 64, 0, 0),
    ("f16", 2, 2, 64, 64, 0, 0),
    ("f16", 4, 2, 128, 64, 1, 0),          # chunk-first phase on the CUDA-core kernel
    ("bf16", 8, 2, 128, 64, 2, 0),          # both phases at once on disjoint SMs
    ("bf16", 8, 2, 128, 64, 0, 2**31 - 1),  # sequence-first only
    ("f16", 4, 2, 128, 32, 0, 0),           # c = 32: CUDA-core path for both phases
    ("f32", 2, 1, 64, 32, 0, 0),
    ("f32", 8, 1, 128, 64, 0, 3),
    # c = 128: the tensor-core kernel takes each chunk as two 64-key tiles;
    # two 128-byte key blocks per 16-bit V^T row in the CUDA-core kernel
    ("f16", 4, 2, 128, 128, 0, 0),
    ("bf16", 8, 1, 64, 128, 0, 0),
    ("bf16", 8, 2, 128, 128, 1, 0),         # chunk-first phase on the CUDA-core kernel
    ("f16", 2, 2, 128, 128, 0, 2**31 - 1),
    ("f32", 8, 2, 128, 128, 0, 0),          # one fp32 accumulator pair per key
    ("f32", 8, 1, 128, 128, 0, 0),
    # c = 16: one 16-key tile per chunk (16-bit), half a warp of keys (fp32)
    ("f16", 4, 4, 128, 16, 0, 0),
    ("bf16", 8, 2, 64, 16, 0, 0),
    ("bf16", 8, 1, 128, 16, 0, 2**31 - 1),
    ("f32", 4, 2, 128, 16, 0, 0),
    ("f32", 2, 2, 64, 16, 0, 0),
]


def _ragged_tree(seed, dtype, hq, hkv, d, c, n_seqs=7):
    """Sequences over a 3-level prefix tree with ragged, non-aligned lengths."""
    g = torch.Generator().manual_seed(seed)
    dt = W.DTYPES[dtype]
    root_n = 3 * c + 5 if c <= 64 else c
    root_t = torch.randint(0, 50, (root_n,), generator=g, dtype=torch.int32)
    root_k = torch.randn(root_n, hkv, d, generator=g).to(dt)
    root_v = torch.randn(root_n, hkv, d, generator=g).to(dt)
    br = []
    for b in range(2):
        n = c * (b + 1) + 3
        t = torch.randint(0, 50, (n,), generator=g, dtype=torch.int32)
        t[0] = 900 + b
        br.append((t, torch.randn(n, hkv, d, generator=g).to(dt), torch.randn(n, hkv, d, generator=g).to(dt)))
    seqs = []
    for s in range(n_seqs):
        b = s % 2
        # branch sequences share the root's full chunks (root_n is not chunk aligned,
        # so the partial last root chunk stays private to each sequence)
        tail = int(torch.randint(1, 2 * c + 7, (1,), generator=g))
        t = torch.randint(0, 50, (tail,), generator=g, dtype=torch.int32)
        t[0] = 2000 + s
        toks = torch.cat([root_t, br[b][0], t]) if s < n_seqs - 1 else root_t[: c * 2].clone()
        if s < n_seqs - 1:
            k = torch.cat([root_k, br[b][1], torch.randn(tail, hkv, d, generator=g).to(dt)])
            v = torch.cat([root_v, br[b][2], torch.randn(tail, hkv, d, generator=g).to(dt)])
        else:
            k, v = root_k[: c * 2].clone(), root_v[: c * 2].clone()
        seqs.append((toks, k, v))
    q = torch.randn(n_seqs, hq, d, generator=g).to(dt)
    return seqs, q


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_ragged_tree_all_rows(pst, case):
    dtype, hq, hkv, d, c, flags, min_share = case
    seqs, q = _ragged_tree(11, dtype, hq, hkv, d, c)
    pool = pst.Pool(hq, hkv, d, c, 512, dtype, min_share, 0, flags, device=0)
    ids = [pool.insert(t, k.cuda(), v.cuda())[0] for (t, k, v) in seqs]
    order = pool.batch_order()
    assert sorted(order) == ids
    qb = q[order]
    out = _decode(pool, qb.cuda())
    ref = A.decode_attention([(_f64(seqs[s][1]), _f64(seqs[s][2])) for s in order], _f64(qb))
    _assert_close(_f64(out), ref, dtype, with_ulp=True, what=str(case))


@pytest.mark.parametrize("dtype,hq,hkv,c", [("f16", 4, 2, 64), ("bf16", 8, 2, 64), ("f32", 2, 2, 32),
                                            ("f16", 4, 2, 16), ("bf16", 4, 4, 128)])
def test_dynamic_tree_appends_and_removes(pst, dtype, hq, hkv, c):
    d = 128
    seqs, q = _ragged_tree(5, dtype, hq, hkv, d, c, n_seqs=6)
    pool = pst.Pool(hq, hkv, d, c, 512, dtype, 0, 0, 0, device=0)
    kv = {}
    for (t, k, v) in seqs:
        sid, _ = pool.insert(t, k.cuda(), v.cuda())
        kv[sid] = (k, v)
    g = torch.Generator().manual_seed(3)
    dt = W.DTYPES[dtype]
    for step in range(c + 9):
        ids = sorted(kv)
        k = torch.randn(len(ids), hkv, d, generator=g).to(dt)
        v = torch.randn(len(ids), hkv, d, generator=g).to(dt)
        pool.append_batch(ids, [7] * len(ids), k.cuda(), v.cuda())
        for i, sid in enumerate(ids):
            kv[sid] = (torch.cat([kv[sid][0], k[i:i + 1]]), torch.cat([kv[sid][1], v[i:i + 1]]))
        if step in (5, 40):
            victim = ids[len(ids) // 2]
            pool.remove(victim)
            del kv[victim]
        if step % 17 == 0 or step == c + 8:
            order = pool.batch_order()
            qq = torch.randn(len(order), hq, d, generator=g).to(dt)
            out = _decode(pool, qq.cuda())
            ref = A.decode_attention([(_f64(kv[s][0]), _f64(kv[s][1])) for s in order], _f64(qq))
            _assert_close(_f64(out), ref, dtype, with_ulp=True, what=f"step {step}")


def test_nan_in_matched_rows_is_ignored(pst):
    spec = W.WorkloadSpec("nan", 4, 2, 128, 64, "f16", ((256, 1), (128, 3)), 77)
    wl = W.generate(spec)
    pool_a = _pool(pst, spec)
    W.insert_all(pool_a, wl, nan_matched=True)
    pool_b = _pool(pst, spec)
    W.insert_all(pool_b, wl, nan_matched=False)
    qa = wl.q.cuda()
    oa, ob = _decode(pool_a, qa), _decode(pool_b, qa)
    assert torch.equal(oa, ob)
    ref = A.decode_attention([(_f64(wl.seq_k(s)), _f64(wl.seq_v(s))) for s in range(wl.n_sequences)], _f64(wl.q))
    _assert_close(_f64(oa), ref, "f16")


def test_empty_batch_and_host_api(pst):
    spec = W.WorkloadSpec("hostapi", 8, 2, 128, 64, "bf16", ((128, 1), (64, 5)), 78)
    wl = W.generate(spec)
    pool = _pool(pst, spec)
    q0 = torch.empty(0, 8, 128, dtype=torch.bfloat16, device="cuda")
    pool.decode_attention(q0, torch.empty_like(q0))  # no live sequences: no-op
    W.insert_all(pool, wl)
    q = wl.q.cuda()
    out_dev = _decode(pool, q)
    q_host = wl.q.clone().pin_memory()
    out_host = torch.empty_like(q_host).pin_memory()
    pool.decode_attention_host(q_host, out_host)
    assert torch.equal(out_host, out_dev.cpu())


def test_pool_filled_to_capacity(pst):
    spec = W.WorkloadSpec("full", 4, 4, 64, 64, "f16", ((128, 1), (192, 4)), 79)
    wl = W.generate(spec)
    cap = W_chunks(spec)
    pool = _pool(pst, spec, max_chunks=cap)
    W.insert_all(pool, wl)
    assert pool.stats()["free_chunks"] == 0
    with pytest.raises(pst.PstError):
        pool.append(0, 1, torch.zeros(4, 64, dtype=torch.float16, device="cuda"),
                    torch.zeros(4, 64, dtype=torch.float16, device="cuda"))
    out = _decode(pool, wl.q.cuda())
    ref = A.decode_attention([(_f64(wl.seq_k(s)), _f64(wl.seq_v(s))) for s in range(wl.n_sequences)], _f64(wl.q))
    _assert_close(_f64(out), ref, "f16")


# ----------------------------------------------------------- full configs
def _sample_rows(b, hq, n, seed):
    rng = np.random.default_rng(seed)
    rows = {(0, 0), (b - 1, hq - 1), (b // 2, hq // 2)}
    while len(rows) < n:
        rows.add((int(rng.integers(0, b)), int(rng.integers(0, hq))))
    return sorted(rows)


@pytest.mark.parametrize("name", ["share1k", "share4k", "noshare", "gqa_tree", "batch96", "div_s1024_c1024",
                                  "gen_d128_c128", "gen_d64_c16"])
def test_full_config_sampled_rows(pst, name):
    spec = W.SPECS[name]
    wl = W.generate(spec, device="cuda")
    pool = _pool(pst, spec)
    W.insert_all(pool, wl)
    order = pool.batch_order()
    assert order == list(range(spec.n_sequences))
    st = pool.stats()
    assert st["used_chunks"] == W_chunks(spec)
    q = wl.q
    out = _decode(pool, q)
    rows = _sample_rows(spec.n_sequences, spec.n_q_heads, 24, spec.seed)
    seq_cache = {}

    def kv(u):
        if u not in seq_cache:
            seq_cache[u] = (_f64(wl.seq_k(u)), _f64(wl.seq_v(u)))
        return seq_cache[u]
    ref = A.decode_rows({u: kv(u) for u, _ in rows}, _f64(q), rows)
    got = np.stack([_f64(out[u, h]) for u, h in rows])
    _assert_close(got, ref, spec.dtype, what=name)
    # at any size: the sequence-first-only path gives the same answer
    pool2 = _pool(pst, spec, min_share=2**31 - 1)
    W.insert_all(pool2, wl)
    out2 = _decode(pool2, q)
    diff = (out.float() - out2.float()).abs().max().item()
    assert diff <= 2 * TOL[spec.dtype], diff


def test_gqa_tree_chunked_prefill(pst):
    spec = W.SPECS["gqa_tree"]
    wl = W.generate(spec, device="cuda")
    pool = _pool(pst, spec, max_chunks=W_chunks(spec) + 200)
    W.insert_all(pool, wl)
    root = wl.segments[0]
    n0 = root.tokens.shape[0]
    sid, m = pool.insert(root.tokens.cpu())          # fully matched: shares the 2048-token root
    assert m == n0
    blocks = prefill_blocks(spec.prefill_prompt, spec.prefill_width)
    assert blocks == [512, 512, 113]
    outs = []
    off = 0
    for w in blocks:
        out = torch.empty(w, spec.n_q_heads, spec.head_dim, dtype=W.DTYPES[spec.dtype], device="cuda")
        pool.prefill_attend(sid, wl.prefill_tokens[off:off + w].cpu(), wl.prefill_q[off:off + w].contiguous(),
                            wl.prefill_k[off:off + w].contiguous(), wl.prefill_v[off:off + w].contiguous(), out)
        outs.append(out)
        off += w
    torch.cuda.synchronize()
    assert pool.check_device() == 0
    out = torch.cat(outs)
    k_all = torch.cat([root.k, wl.prefill_k])
    v_all = torch.cat([root.v, wl.prefill_v])
    rows = [0, 1, 511, 512, 700, 1023, 1024, 1100, 1136]
    ref = np.concatenate([A.prefill_attention(_f64(k_all[:n0 + t + 1]), _f64(v_all[:n0 + t + 1]),
                                              _f64(wl.prefill_q[t:t + 1]), n0 + t) for t in rows])
    _assert_close(_f64(out[rows]), ref, spec.dtype, what="prefill")
    # the cache now holds the appended prompt, byte for byte
    n = pool.seq_length(sid)
    assert n == n0 + spec.prefill_prompt
    ko = torch.empty(n, spec.n_kv_heads, spec.head_dim, dtype=W.DTYPES[spec.dtype], device="cuda")
    vo = torch.empty_like(ko)
    pool.gather_kv(sid, ko, vo)
    assert torch.equal(ko.view(torch.int16), k_all.view(torch.int16))
    # single pass over the whole prompt agrees with the blocked run
    pool2 = _pool(pst, spec, max_chunks=W_chunks(spec) + 200)
    W.insert_all(pool2, wl)
    sid2, _ = pool2.insert(root.tokens.cpu())
    one = torch.empty_like(out)
    pool2.prefill_attend(sid2, wl.prefill_tokens.cpu(), wl.prefill_q.contiguous(), wl.prefill_k.contiguous(),
                         wl.prefill_v.contiguous(), one)
    torch.cuda.synchronize()
    assert (one.float() - out.float()).abs().max().item() <= 2 * TOL[spec.dtype]


PREFILL_CASES = [
    ("f16", 4, 2, 128, 64, 0, 0, [5, 64, 1, 130]),
    ("bf16", 8, 8, 64, 64, 0, 70, [200]),
    ("f16", 4, 1, 128, 64, 1, 33, [3, 61]),       # CUDA-core prefill
    ("f32", 2, 1, 64, 32, 0, 31, [33, 2, 40]),
    ("bf16", 8, 2, 128, 128, 0, 100, [130, 7]),   # c = 128: two tiles per chunk, the last one partial
    ("f16", 4, 4, 128, 128, 0, 0, [50, 20]),      # c = 128: a tile with no valid key
    ("bf16", 8, 2, 64, 128, 1, 40, [100]),        # c = 128: CUDA-core prefill
    ("f16", 4, 4, 64, 16, 0, 20, [40, 1, 77]),    # c = 16: runs of more than four chunks
    ("f32", 2, 1, 64, 16, 0, 5, [17, 30]),
]


@pytest.mark.parametrize("case", PREFILL_CASES, ids=lambda c: "-".join(map(str, c[:7])))
def test_prefill_blocks_all_rows(pst, case):
    dtype, hq, hkv, d, c, flags, p0, blocks = case
    g = torch.Generator().manual_seed(p0 + len(blocks))
    dt = W.DTYPES[dtype]
    n = p0 + sum(blocks)
    toks = torch.randint(0, 100, (n,), generator=g, dtype=torch.int32)
    k = torch.randn(n, hkv, d, generator=g).to(dt)
    v = torch.randn(n, hkv, d, generator=g).to(dt)
    q = torch.randn(n, hq, d, generator=g).to(dt)
    pool = pst.Pool(hq, hkv, d, c, 256, dtype, 0, 0, flags, device=0)
    start = max(p0, 1)
    sid, _ = pool.insert(toks[:start], k[:start].cuda(), v[:start].cuda())
    outs = []
    pos = start
    for w in ([blocks[0] - (start - p0)] if start > p0 else []) + (blocks[1:] if start > p0 else blocks):
        if w <= 0:
            continue
        out = torch.empty(w, hq, d, dtype=dt, device="cuda")
        pool.prefill_attend(sid, toks[pos:pos + w], q[pos:pos + w].cuda(), k[pos:pos + w].cuda(),
                            v[pos:pos + w].cuda(), out)
        outs.append((pos, out))
        pos += w
    torch.cuda.synchronize()
    assert pool.check_device() == 0
    for p, out in outs:
        w = out.shape[0]
        ref = A.prefill_attention(_f64(k[:p + w]), _f64(v[:p + w]), _f64(q[p:p + w]), p)
        _assert_close(_f64(out), ref, dtype, with_ulp=True, what=f"block at {p}")
