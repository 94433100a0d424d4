"""Multi-layer pools: the K/V of n_layers decoder layers under one prefix tree.

The tree and the chunk tables depend on token ids only, so every layer shares
them (ChunkAttention, Knowl 5: the context is built once per step, behind the
layers' earlier kernels); layer l's attention reads layer l's K/V.  Checked
against the fp64 oracle layer by layer: decode after an insert that writes all
layers at once; a decode loop whose appends add each token to the tree first
and then write its K/V layer by layer, each layer replaying its own captured
graph (checked against the regular entry point); a chunked prefill written and attended
layer by layer (Chunked Prefill, sections 1-2); byte-exact read-back of all
layers; and the refusals (rows in a shared chunk, a layer out of range).
"""
import pytest
import torch

from oracle import attention as A
from prefix_shared_kv_tree_gb300 import workloads as W
from tests import parity_util as PU

pytestmark = pytest.mark.gpu

N_LAYERS = 3


@pytest.fixture(scope="module")
def pst():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from prefix_shared_kv_tree_gb300 import build
    build.build_library()
    from prefix_shared_kv_tree_gb300 import pst as mod
    return mod


_f64 = PU.f64


# dtype, Hq, Hkv, c: tensor-core chunk-first at c = 64 and (two tiles per chunk)
# c = 128; fp32 on the CUDA-core kernel for both phases
CASES = [("bf16", 8, 2, 64), ("f16", 4, 4, 128), ("f32", 2, 1, 32)]


@pytest.mark.parametrize("dtype,hq,hkv,c", CASES)
def test_layers_decode_loop_and_prefill(pst, dtype, hq, hkv, c):
    L = N_LAYERS
    d = 64 if dtype == "f32" else 128
    dt = W.DTYPES[dtype]
    g = torch.Generator().manual_seed(40 + c)
    tw = PU.Twin(pst, hq, hkv, d, c, 512, dtype, n_layers=L)
    pool = tw.native

    # a shared root of 3 full chunks + 10 tokens, four sequences with private tails
    root_n = 3 * c + 10
    root_t = torch.randint(0, 50, (root_n,), generator=g, dtype=torch.int32)
    root_k = torch.randn(L, root_n, hkv, d, generator=g).to(dt)
    root_v = torch.randn(L, root_n, hkv, d, generator=g).to(dt)
    kv = {}  # sequence id -> its K, V on the CPU, [L][n][Hkv][d]
    for s in range(4):
        tail = c // 2 + 7 * s
        t = torch.randint(0, 50, (tail,), generator=g, dtype=torch.int32)
        t[0] = 1000 + s
        k = torch.cat([root_k, torch.randn(L, tail, hkv, d, generator=g).to(dt)], dim=1)
        v = torch.cat([root_v, torch.randn(L, tail, hkv, d, generator=g).to(dt)], dim=1)
        sid, m = tw.insert(torch.cat([root_t, t]), k.cuda(), v.cuda())
        assert m == (0 if s == 0 else 3 * c)
        kv[sid] = (k, v)

    def check_decode(what):
        order = tw.batch_order()
        for layer in range(L):
            q = torch.randn(len(order), hq, d, generator=g).to(dt).cuda()
            out, wide = tw.decode(q, "decode_attention_layer", layer)
            if layer == 0:  # the layer-free entry point reads layer 0
                out0 = torch.empty_like(out)
                pool.decode_attention(q, out0)
                torch.cuda.synchronize()
                assert torch.equal(out0, out), what
            want = A.decode_attention([(_f64(kv[s][0][layer]), _f64(kv[s][1][layer])) for s in order], _f64(q))
            PU.check(out, wide, want, dtype, f"layers {dtype} c{c}: {what}, layer {layer}")
        assert tw.check_device() == 0

    check_decode("after insert")

    # decode loop: each step adds the token to the tree (no K/V), then every
    # layer writes its row of the token and attends, from its own captured
    # graph with its own q / out buffers; every sequence crosses a chunk
    # boundary on the way
    def buffers():
        b = len(tw.batch_order())
        qs = [torch.empty(b, hq, d, dtype=dt, device="cuda") for _ in range(L)]
        return qs, [torch.empty_like(x) for x in qs], torch.empty_like(qs[0])

    qg, og, ref = buffers()
    seen = set()
    for step in range(c + 3):
        ids = sorted(kv)
        tw.append_batch(ids, [7] * len(ids))
        kn = torch.randn(L, len(ids), hkv, d, generator=g).to(dt)
        vn = torch.randn(L, len(ids), hkv, d, generator=g).to(dt)
        for layer in range(L):
            tw.write_kv_last(layer, ids, kn[layer].cuda(), vn[layer].cuda())
        for i, sid in enumerate(ids):
            kv[sid] = (torch.cat([kv[sid][0], kn[:, i:i + 1]], dim=1), torch.cat([kv[sid][1], vn[:, i:i + 1]], dim=1))
        if step == 9:  # a departure: the batch shrinks, so new q / out buffers
            victim = ids[1]
            tw.remove(victim)
            del kv[victim]
            qg, og, ref = buffers()
        for layer in range(L):
            qg[layer].copy_(torch.randn(qg[layer].shape, generator=g).to(dt))
            og[layer].fill_(float("nan"))
            pool.decode_attention_graph_layer(layer, qg[layer], og[layer])
            seen.add((pool.stats()["table_version"], layer, qg[layer].data_ptr(), og[layer].data_ptr()))
            pool.decode_attention_layer(layer, qg[layer], ref)
            torch.cuda.synchronize()
            assert torch.isfinite(og[layer].float()).all(), (step, layer)
            # the same kernels on the same tables: the same bits
            assert torch.equal(og[layer], ref), (step, layer)
        if step % 4 == 0 or step == c + 2:
            check_decode(f"decode step {step}")
    st = pool.stats()
    assert st["graph_captures"] == len(seen), (st["graph_captures"], len(seen))
    assert st["graph_captures"] < L * (c + 3) // 2  # most steps replayed their layer's graph

    # read-back of every layer, byte-exact
    sid0 = sorted(kv)[0]
    n0 = pool.seq_length(sid0)
    ko = torch.empty(L, n0, hkv, d, dtype=dt, device="cuda")
    vo = torch.empty_like(ko)
    pool.gather_kv(sid0, ko, vo)
    torch.cuda.synchronize()
    assert torch.equal(ko.cpu(), kv[sid0][0]) and torch.equal(vo.cpu(), kv[sid0][1])

    # chunked prefill layer by layer: a new sequence matches two root chunks
    # (no K/V to write), then each block joins the tree and, per layer, gets
    # its K/V written and its rows attended
    sid, m = tw.insert(root_t[:2 * c])
    assert m == 2 * c
    pk, pv = root_k[:, :2 * c], root_v[:, :2 * c]
    pos = 2 * c
    for w in (c + 5, 1, 2 * c - 3):
        toks = torch.randint(0, 50, (w,), generator=g, dtype=torch.int32)
        kb = torch.randn(L, w, hkv, d, generator=g).to(dt)
        vb = torch.randn(L, w, hkv, d, generator=g).to(dt)
        tw.extend(sid, toks)
        assert tw.seq_length(sid) == pos + w
        for layer in range(L):
            tw.write_kv(layer, sid, kb[layer].cuda(), vb[layer].cuda())
            q = torch.randn(w, hq, d, generator=g).to(dt)
            out, wide = tw.prefill_attend_layer(layer, sid, pos, q.cuda())
            torch.cuda.synchronize()
            want = A.prefill_attention(_f64(torch.cat([pk[layer], kb[layer]])), _f64(torch.cat([pv[layer], vb[layer]])),
                                       _f64(q), pos)
            PU.check(out, wide, want, dtype, f"layers {dtype} c{c}: prefill block at {pos}, layer {layer}")
        pk, pv = torch.cat([pk, kb], dim=1), torch.cat([pv, vb], dim=1)
        pos += w
    assert tw.check_device() == 0

    # refusals: rows of shared chunks, layers out of range
    n = pool.seq_length(sid)
    junk = torch.zeros(n, hkv, d, dtype=dt, device="cuda")
    with pytest.raises(pst.PstError) as e:
        pool.write_kv(0, sid, junk, junk)  # its first two chunks are the shared root's
    assert e.value.status == pst.PST_ERR_STATE
    q = torch.zeros(len(pool.batch_order()), hq, d, dtype=dt, device="cuda")
    for bad in (-1, L):
        with pytest.raises(pst.PstError) as e:
            pool.decode_attention_layer(bad, q, torch.empty_like(q))
        assert e.value.status == pst.PST_ERR_INVALID
        with pytest.raises(pst.PstError) as e:
            pool.write_kv_last(bad, [sid], junk[:1], junk[:1])
        assert e.value.status == pst.PST_ERR_INVALID
    with pytest.raises(pst.PstError) as e:  # one launch: two rows for one sequence would collide
        pool.write_kv_last(0, [sid, sid], junk[:2], junk[:2])
    assert e.value.status == pst.PST_ERR_INVALID
    torch.cuda.synchronize()
    assert pool.check_device() == 0
