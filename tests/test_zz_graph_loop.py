"""Decode loop through the CUDA-graph entry point (pst_decode_attention_graph).

Per step every live sequence appends one token (pst_append_batch), then the
decode step runs from a captured CUDA graph.  Appends that land in a leaf
chunk change only device-side chunk lengths, so the graph is replayed as is;
a new chunk, a departure or other q / out buffers change the tables or the
pointers and make the library capture again.  Checked at every step against
the regular entry point (bit for bit) and at some steps
against the fp64 oracle (fp32 outputs of a twin pool within the parity bound,
the pool-dtype outputs their rounding); the number of captures must equal the
number of distinct (table version, q, out) triples the loop used.
"""
import pytest
import torch

from oracle import attention as A
from prefix_shared_kv_tree_gb300 import workloads as W
from tests import parity_util as PU

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pst():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from prefix_shared_kv_tree_gb300 import build
    build.build_library()
    from prefix_shared_kv_tree_gb300 import pst as mod
    return mod


_f64 = PU.f64


def _tree(seed, dtype, hkv, d, c, n_seqs):
    """A shared root of 3 full chunks + 10 tokens, then per sequence a private
    tail whose last chunk is partly filled (so appends first fill it, then
    start new chunks)."""
    g = torch.Generator().manual_seed(seed)
    dt = W.DTYPES[dtype]
    root_n = 3 * c + 10
    root_t = torch.randint(0, 50, (root_n,), generator=g, dtype=torch.int32)
    root_k = torch.randn(root_n, hkv, d, generator=g).to(dt)
    root_v = torch.randn(root_n, hkv, d, generator=g).to(dt)
    seqs = []
    for s in range(n_seqs):
        tail = c - 3 + s  # ends 3 + ... tokens short of a chunk boundary, sequence-dependent
        t = torch.randint(0, 50, (tail,), generator=g, dtype=torch.int32)
        t[0] = 1000 + s
        seqs.append((torch.cat([root_t, t]),
                     torch.cat([root_k, torch.randn(tail, hkv, d, generator=g).to(dt)]),
                     torch.cat([root_v, torch.randn(tail, hkv, d, generator=g).to(dt)])))
    return seqs


@pytest.mark.parametrize("dtype,hq,hkv", [("bf16", 8, 2), ("f16", 4, 4)])
def test_graph_decode_loop(pst, dtype, hq, hkv):
    d, c, n_seqs = 128, 64, 6
    dt = W.DTYPES[dtype]
    tw = PU.Twin(pst, hq, hkv, d, c, 256, dtype)
    pool = tw.native
    kv = {}
    for (t, k, v) in _tree(21, dtype, hkv, d, c, n_seqs):
        sid, _ = tw.insert(t, k.cuda(), v.cuda())
        kv[sid] = (k, v)
    g = torch.Generator().manual_seed(5)

    def buffers():
        b = len(tw.batch_order())
        q = torch.empty(b, hq, d, dtype=dt, device="cuda")
        return q, torch.empty_like(q), torch.empty(b, hq, d, dtype=torch.float32, device="cuda"), torch.empty_like(q)

    order = tw.batch_order()
    q, out, wide, ref = buffers()
    seen = set()
    for step in range(c + 12):
        ids = sorted(kv)
        k = torch.randn(len(ids), hkv, d, generator=g).to(dt)
        v = torch.randn(len(ids), hkv, d, generator=g).to(dt)
        tw.append_batch(ids, [9] * len(ids), k.cuda(), v.cuda())
        for i, sid in enumerate(ids):
            kv[sid] = (torch.cat([kv[sid][0], k[i:i + 1]]), torch.cat([kv[sid][1], v[i:i + 1]]))
        if step == 30:  # a departure: the batch shrinks, so new q / out buffers
            victim = ids[len(ids) // 2]
            tw.remove(victim)
            del kv[victim]
            order = tw.batch_order()
            q, out, wide, ref = buffers()
        q.copy_(torch.randn(q.shape, generator=g).to(dt))
        out.fill_(float("nan"))
        wide.fill_(float("nan"))
        pool.decode_attention_graph(q, out)
        tw.wide.decode_attention_graph(q, wide)
        seen.add((pool.stats()["table_version"], q.data_ptr(), out.data_ptr()))
        pool.decode_attention(q, ref)
        torch.cuda.synchronize()
        assert tw.check_device() == 0
        assert torch.isfinite(out.float()).all(), f"step {step}"
        # the same kernels on the same tables: the same bits as the regular entry point
        assert torch.equal(out, ref), f"step {step}"
        if step % 13 == 0 or step == c + 11:
            want = A.decode_attention([(_f64(kv[s][0]), _f64(kv[s][1])) for s in order], _f64(q))
            PU.check(out, wide, want, dtype, f"graph loop {dtype} step {step}")
    st = pool.stats()
    assert st["graph_captures"] == len(seen), (st["graph_captures"], len(seen))
    assert st["graph_captures"] < c  # most steps replayed a captured graph


def test_misaligned_q_or_out_is_refused(pst):
    """q and out must start on a 16-byte boundary (the kernels move 16-byte
    vectors); every decode entry point refuses otherwise with PST_ERR_INVALID
    and launches nothing."""
    hq, hkv, d, c = 4, 2, 128, 64
    seqs = _tree(8, "f16", hkv, d, c, 3)
    pool = pst.Pool(hq, hkv, d, c, 64, "f16", 0, 0, 0, device=0)
    for (t, k, v) in seqs:
        pool.insert(t, k.cuda(), v.cuda())
    B = len(pool.batch_order())
    flat = torch.zeros(B * hq * d + 8, dtype=torch.float16, device="cuda")
    good = flat[:B * hq * d].view(B, hq, d)
    bad = flat[1:1 + B * hq * d].view(B, hq, d)  # 2 bytes past a 16-byte boundary
    out = torch.empty(B, hq, d, dtype=torch.float16, device="cuda")
    pool.decode_attention(good, out)  # tables on the device
    torch.cuda.synchronize()
    for call in (pool.decode_attention, pool.decode_attention_graph, pool.decode_attention_noalloc):
        with pytest.raises(pst.PstError) as e:
            call(bad, out)
        assert e.value.status == pst.PST_ERR_INVALID
        with pytest.raises(pst.PstError) as e:
            call(good, bad)
        assert e.value.status == pst.PST_ERR_INVALID
    torch.cuda.synchronize()
    assert pool.check_device() == 0
