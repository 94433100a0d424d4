"""Shared parity checks of the CUDA path against the fp64 oracle.

The stated bound is max |gpu - oracle| <= 2e-3 for fp16/bf16 K/V and <= 1e-5
for fp32.  It is applied, without any widening, to the kernels' fp32 results:
every case runs on two pools built from the same calls, one writing its
outputs in the pool dtype and one with PST_FLAG_F32_OUT, which writes the fp32
value the kernels would otherwise round.  Then

  * |out_f32 - oracle| <= tolerance, element by element, and
  * out_native == round-to-nearest-even(out_f32), bit for bit,

so the product path's 16-bit outputs are the correctly rounded fp32 results
(ChunkAttention, Knowl 3 computes the result; the rounding to the output type
is the only step after it).  The same tables drive both pools, so their fp32
arithmetic is identical.

Every check also records max abs error and the normwise relative error
max|gpu - oracle| / max|oracle| (and the largest element-wise relative error
over elements with |oracle| >= 1e-2); with PST_PARITY_REPORT naming a file,
one JSON line per check is appended to it.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

from prefix_shared_kv_tree_gb300 import workloads as W

TOL = {"f16": 2e-3, "bf16": 2e-3, "f32": 1e-5}
F32_OUT = 4  # PST_FLAG_F32_OUT


def f64(t) -> np.ndarray:
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().float().cpu().double().numpy()


def errors(got, ref) -> dict:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    big = np.abs(ref) >= 1e-2
    return {"max_abs": float(err.max()) if err.size else 0.0,
            "rel_norm": float(err.max() / max(np.abs(ref).max(), 1e-300)) if err.size else 0.0,
            "max_rel_elem": float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0,
            "max_abs_ref": float(np.abs(ref).max()) if ref.size else 0.0,
            "n": int(err.size)}


def record(what: str, stats: dict, **extra) -> None:
    path = os.environ.get("PST_PARITY_REPORT")
    line = dict(case=what, **stats, **extra)
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(line) + "\n")


def assert_close(got, ref, dtype: str, what: str) -> dict:
    """|got - ref| <= TOL[dtype] everywhere (got: fp32 or fp64 values)."""
    got = f64(got)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    st = errors(got, ref)
    record(what, st, dtype=dtype, tol=TOL[dtype])
    err = np.abs(got - ref)
    bad = err > TOL[dtype]
    assert not bad.any(), f"{what}: max err {err.max():.3e} > {TOL[dtype]} at {np.argwhere(bad)[:3].tolist()}"
    return st


def assert_rounded(native: torch.Tensor, wide: torch.Tensor, what: str) -> None:
    """The pool-dtype output is the fp32 output rounded to nearest even, bit for bit."""
    assert wide.dtype == torch.float32, what
    want = wide.to(native.dtype)
    if not torch.equal(native.view(torch.int16) if native.element_size() == 2 else native,
                       want.view(torch.int16) if want.element_size() == 2 else want):
        diff = (native.float() - want.float()).abs()
        raise AssertionError(f"{what}: native output is not RNE(fp32 output): {int((diff > 0).sum())} elements differ")


def check(native: torch.Tensor, wide: torch.Tensor, ref, dtype: str, what: str) -> dict:
    """Both parity checks of one output (wide is native itself for fp32 pools)."""
    st = assert_close(wide, ref, dtype, what)
    if wide is not native:
        assert_rounded(native, wide, what)
    return st


class Twin:
    """The same pool twice -- outputs in the pool dtype, and fp32 outputs
    (PST_FLAG_F32_OUT) -- driven by the same calls.  For fp32 pools the two
    coincide and one pool serves both."""

    def __init__(self, pst, hq, hkv, d, c, max_chunks, dtype, min_share=0, max_seqs=0, flags=0, n_layers=0,
                 device=0):
        self.dtype = dtype
        self.dt = W.DTYPES[dtype]
        self.native = pst.Pool(hq, hkv, d, c, max_chunks, dtype, min_share, max_seqs, flags, device=device,
                               n_layers=n_layers)
        self.wide = (self.native if dtype == "f32" else
                     pst.Pool(hq, hkv, d, c, max_chunks, dtype, min_share, max_seqs, flags | F32_OUT,
                              device=device, n_layers=n_layers))
        self.pools = [self.native] if self.wide is self.native else [self.native, self.wide]

    # tree operations: same call on both pools, the first pool's result
    def _both(self, name, *a, **kw):
        res = [getattr(p, name)(*a, **kw) for p in self.pools]
        assert all(r == res[0] for r in res), (name, res)
        return res[0]

    def insert(self, *a, **kw):
        return self._both("insert", *a, **kw)

    def append_batch(self, *a, **kw):
        return self._both("append_batch", *a, **kw)

    def remove(self, *a, **kw):
        return self._both("remove", *a, **kw)

    def extend(self, *a, **kw):
        return self._both("extend", *a, **kw)

    def write_kv(self, *a, **kw):
        return self._both("write_kv", *a, **kw)

    def write_kv_last(self, *a, **kw):
        return self._both("write_kv_last", *a, **kw)

    def batch_order(self):
        return self._both("batch_order")

    def seq_length(self, sid):
        return self._both("seq_length", sid)

    def stats(self):
        return self.native.stats()

    def check_device(self) -> int:
        return max(p.check_device() for p in self.pools)

    # attention: (native output, fp32 output)
    def _outs(self, shape):
        n = torch.empty(shape, dtype=self.dt, device="cuda")
        w = n if self.wide is self.native else torch.empty(shape, dtype=torch.float32, device="cuda")
        return n, w

    def decode(self, q, method="decode_attention", *lead):
        n, w = self._outs(q.shape)
        n.fill_(float("nan"))
        if w is not n:
            w.fill_(float("nan"))
        getattr(self.native, method)(*lead, q, n)
        if w is not n:
            getattr(self.wide, method)(*lead, q, w)
        torch.cuda.synchronize()
        assert self.check_device() == 0
        return n, w

    def prefill_attend(self, sid, tokens, q, k, v):
        n, w = self._outs(q.shape)
        self.native.prefill_attend(sid, tokens, q, k, v, n)
        if w is not n:
            self.wide.prefill_attend(sid, tokens, q, k, v, w)
        return n, w

    def prefill_attend_layer(self, layer, sid, p0, q):
        n, w = self._outs(q.shape)
        self.native.prefill_attend_layer(layer, sid, p0, q, n)
        if w is not n:
            self.wide.prefill_attend_layer(layer, sid, p0, q, w)
        return n, w


def oracle_all_rows(A, wl, q=None) -> np.ndarray:
    """Every (sequence, head) row of a workload's decode step from the fp64
    oracle: each sequence's full K/V materialised (no sharing), one sequence
    at a time.  Segments are read back to the host once."""
    segs = [(s.k.float().cpu().numpy(), s.v.float().cpu().numpy()) for s in wl.segments]
    qn = f64(wl.q if q is None else q)
    out = np.empty(qn.shape, np.float64)
    for u, path in enumerate(wl.seq_paths):
        k = np.concatenate([segs[i][0] for i in path])
        v = np.concatenate([segs[i][1] for i in path])
        out[u] = A.decode_attention([(k, v)], qn[u:u + 1])[0]
    return out
