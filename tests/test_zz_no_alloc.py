"""The allocation-free decode entry point (pst_decode_attention_noalloc).

Some callers cannot allocate device memory while they run -- a serving
runtime that gave all GPU memory to its own allocator up front, or a hot loop
where cudaMalloc / cudaFree would synchronise the device.  For them the
library offers a decode variant whose scratch (partial rows and the work
counter) lives in a fixed device area it defines itself.  This test calls it
through the C ABI twice in a row and checks both results against the regular
entry point: the same kernels run on the same tables and only the scratch
addresses differ, so the outputs must be the same bits.  It also checks that
the calls change neither the device's free memory nor the pool's buffers, and
the two refusals (stale tables, batch too large for the area).

Kept in a file of its own that sorts last, so a stop-at-first-failure run has
already run every other test when it gets here.
"""
import pytest
import torch

from prefix_shared_kv_tree_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pst():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from prefix_shared_kv_tree_gb300 import build
    build.build_library()
    from prefix_shared_kv_tree_gb300 import pst as mod
    return mod


def _pool(pst, spec, extra=64):
    chunks = 0
    mult = 1
    for n, fan in spec.levels:
        mult *= fan
        chunks += mult * -(-n // spec.chunk_size)
    return pst.Pool(spec.n_q_heads, spec.n_kv_heads, spec.head_dim, spec.chunk_size, chunks + extra, spec.dtype,
                    device=0)


@pytest.mark.parametrize("spec", [
    # GQA tree: both the tensor-core chunk-first kernel and the CUDA-core kernel run
    W.WorkloadSpec("noalloc_gqa", 8, 2, 128, 64, "bf16", ((256, 1), (128, 4), (64, 3)), 4343),
    # no sharing: the CUDA-core kernel alone
    W.WorkloadSpec("noalloc_plain", 4, 4, 64, 64, "f16", ((192, 6),), 4344),
])
def test_noalloc_matches_regular_entry_point_twice(pst, spec):
    wl = W.generate(spec)
    pool = _pool(pst, spec)
    W.insert_all(pool, wl)
    q = wl.q.cuda()
    ref = torch.empty_like(q)
    pool.decode_attention(q, ref)  # uploads the tables (may allocate)
    outs = [torch.full_like(q, float("nan")) for _ in range(3)]
    pool.decode_attention_noalloc(q, outs[2])  # warm-up: kernels loaded, launch attributes set
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    stats0 = pool.stats()
    for out in outs[:2]:
        pool.decode_attention_noalloc(q, out)
        torch.cuda.synchronize()
        assert pool.check_device() == 0
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert pool.stats() == stats0
    for out in outs:
        assert torch.isfinite(out.float()).all()
        assert torch.equal(out, ref)


def test_noalloc_refuses_stale_tables_and_oversize(pst):
    spec = W.WorkloadSpec("noalloc_refuse", 4, 4, 128, 64, "f16", ((128, 1), (64, 3)), 4345)
    wl = W.generate(spec)
    pool = _pool(pst, spec)
    W.insert_all(pool, wl)
    q = wl.q.cuda()
    out = torch.empty_like(q)
    with pytest.raises(pst.PstError) as e:  # tables never uploaded yet
        pool.decode_attention_noalloc(q, out)
    assert e.value.status == pst.PST_ERR_STATE
    pool.decode_attention(q, out)
    pool.decode_attention_noalloc(q, out)   # now fine

    # a batch whose partial rows exceed the fixed 32 MiB area is refused
    # (4000 sequences x 16 KV heads: about 128K partial rows of 520 bytes)
    big = W.WorkloadSpec("noalloc_big", 16, 16, 128, 64, "f16", ((64, 1), (64, 4000)), 4346)
    wl2 = W.generate(big, device="cuda")
    pool2 = _pool(pst, big)
    W.insert_all(pool2, wl2)
    q2 = wl2.q
    out2 = torch.empty_like(q2)
    pool2.decode_attention(q2, out2)
    assert pool2.stats()["partial_rows"] * (128 + 2) * 4 > 32 << 20
    with pytest.raises(pst.PstError) as e:
        pool2.decode_attention_noalloc(q2, out2)
    assert e.value.status == pst.PST_ERR_INVALID
    torch.cuda.synchronize()
    assert pool2.check_device() == 0
