"""Failure detection without a GPU fault: a bounded wait that runs out.

Every spin-wait in the attention kernels is bounded by the GPU's global timer.
Here one warp waits, through the kernels' own bounded mbarrier wait, on a
barrier that nothing arrives on (pst_selftest_bounded_wait): the wait must give
up after its limit, set the wait-timeout bit of the device error word and
return, and the context must stay usable -- a decode on the same device
afterwards still matches the fp64 oracle and leaves the error word clear.
"""
import time

import numpy as np
import pytest
import torch

from oracle import attention as A
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


def _f64(t):
    return t.detach().float().cpu().double().numpy()


def test_bounded_wait_gives_up_and_the_context_survives(pst):
    t0 = time.perf_counter()
    code, lanes = pst.selftest_bounded_wait(0)
    waited = time.perf_counter() - t0
    assert code == pst.PST_DEVICE_WAIT_TIMEOUT
    assert lanes == 32               # every lane's wait returned unfinished
    assert 1.9 < waited < 60         # the limit is 2 s of the GPU's global timer

    spec = W.SPECS["tiny"]
    wl = W.generate(spec)
    pool = pst.Pool(spec.n_q_heads, spec.n_kv_heads, spec.head_dim, spec.chunk_size, 64, spec.dtype, device=0)
    W.insert_all(pool, wl)
    q = wl.q.cuda()
    out = torch.empty_like(q)
    pool.decode_attention(q, out)
    torch.cuda.synchronize()
    assert pool.check_device() == 0
    ref = A.decode_attention([(_f64(wl.seq_k(s)), _f64(wl.seq_v(s))) for s in range(wl.n_sequences)], _f64(wl.q))
    assert float(np.abs(_f64(out) - ref).max()) <= 1e-5
