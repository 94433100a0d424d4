"""ctypes binding of libpst.so (include/pst.h) -- argument marshalling only.

Every function of the C ABI is exposed under its own name; ``Pool`` wraps a
pool handle with methods that take torch tensors (device buffers) and numpy /
torch CPU arrays (token ids, host buffers) and pass their pointers through.
All computation happens in the library's CUDA kernels and C++ tree manager.
Importing this module fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, Structure, byref, c_char_p, c_double, c_float, c_int, c_int32, c_int64, c_void_p

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("PST_LIBRARY") or os.path.join(_HERE, "libpst.so")

PST_OK, PST_ERR_INVALID, PST_ERR_OOM, PST_ERR_NOT_FOUND, PST_ERR_CUDA, PST_ERR_STATE, PST_ERR_DEVICE = range(7)
STATUS_NAMES = {0: "OK", 1: "INVALID", 2: "OOM", 3: "NOT_FOUND", 4: "CUDA", 5: "STATE", 6: "DEVICE"}
PST_F16, PST_BF16, PST_F32 = 0, 1, 2
DTYPE_CODES = {"f16": PST_F16, "bf16": PST_BF16, "f32": PST_F32}
PST_FLAG_NO_TENSOR_CORES = 1
PST_FLAG_CONCURRENT_PHASES = 2
PST_FLAG_F32_OUT = 4
MIN_SHARE_NEVER = 2**31 - 1


class pst_config(Structure):
    _fields_ = [("n_q_heads", c_int32), ("n_kv_heads", c_int32), ("head_dim", c_int32), ("chunk_size", c_int32),
                ("max_chunks", c_int64), ("dtype", c_int32), ("min_share", c_int32), ("max_seqs", c_int32),
                ("flags", c_int32), ("n_layers", c_int32)]


class pst_stats_t(Structure):
    _fields_ = [("live_seqs", c_int64), ("used_chunks", c_int64), ("free_chunks", c_int64), ("max_chunks", c_int64),
                ("shared_chunks", c_int64), ("unique_tokens", c_int64), ("logical_tokens", c_int64),
                ("table_version", c_int64), ("rebuild_count", c_int64), ("last_rebuild_us", c_double),
                ("phase1_items", c_int64), ("phase2_items", c_int64), ("partial_rows", c_int64),
                ("graph_captures", c_int64), ("phase1_ctas", c_int64), ("phase2_ctas", c_int64),
                ("simt_first", c_int64)]


class PstError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"pst status {STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_P = c_void_p
_I64P = POINTER(c_int64)
_I32P = POINTER(c_int32)

# name: (restype, argtypes)
SIGNATURES = {
    "pst_pool_create": (c_int, [POINTER(pst_config), c_int, POINTER(c_void_p)]),
    "pst_pool_free": (c_int, [_P]),
    "pst_match": (c_int, [_P, _P, c_int64, _I64P]),
    "pst_insert": (c_int, [_P, _P, c_int64, _P, _P, _P, _I64P, _I64P]),
    "pst_append": (c_int, [_P, c_int64, c_int32, _P, _P, _P]),
    "pst_append_batch": (c_int, [_P, c_int64, _P, _P, _P, _P, _P]),
    "pst_remove": (c_int, [_P, c_int64]),
    "pst_batch_order": (c_int, [_P, _P, c_int64, _I64P]),
    "pst_seq_length": (c_int, [_P, c_int64, _I64P]),
    "pst_decode_attention": (c_int, [_P, _P, _P, _P]),
    "pst_decode_attention_host": (c_int, [_P, _P, _P, _P]),
    "pst_decode_attention_noalloc": (c_int, [_P, _P, _P, _P]),
    "pst_decode_attention_graph": (c_int, [_P, _P, _P, _P]),
    "pst_prefill_attend": (c_int, [_P, c_int64, _P, c_int64, _P, _P, _P, _P, _P]),
    "pst_gather_kv": (c_int, [_P, c_int64, _P, _P, _P]),
    "pst_extend": (c_int, [_P, c_int64, _P, c_int64]),
    "pst_write_kv": (c_int, [_P, c_int32, c_int64, c_int64, _P, _P, _P]),
    "pst_write_kv_last": (c_int, [_P, c_int32, c_int64, _P, _P, _P, _P]),
    "pst_decode_attention_layer": (c_int, [_P, c_int32, _P, _P, _P]),
    "pst_decode_attention_graph_layer": (c_int, [_P, c_int32, _P, _P, _P]),
    "pst_prefill_attend_layer": (c_int, [_P, c_int32, c_int64, c_int64, c_int64, _P, _P, _P]),
    "pst_export_tables": (c_int, [_P, _P, c_int64, _I64P, _P, c_int64, _I64P, _P, c_int64, _I64P]),
    "pst_stats": (c_int, [_P, POINTER(pst_stats_t)]),
    "pst_set_profiling": (c_int, [_P, c_int]),
    "pst_phase_times": (c_int, [_P, POINTER(c_float)]),
    "pst_last_launch_count": (c_int, [_P, _I32P]),
    "pst_selftest_bounded_wait": (c_int, [c_int, _I32P, _I32P]),
    "pst_check_device": (c_int, [_P, _I32P]),
    "pst_last_error": (c_char_p, []),
    "pst_version": (c_char_p, []),
}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


PST_DEVICE_WAIT_TIMEOUT = 1
PST_DEVICE_BAD_INDEX = 2


def selftest_bounded_wait(device: int = 0):
    """pst_selftest_bounded_wait: (device error word, lanes whose wait gave up)."""
    code, lanes = c_int32(), c_int32()
    check(lib.pst_selftest_bounded_wait(device, byref(code), byref(lanes)))
    return code.value, lanes.value


def check(status: int) -> None:
    if status != PST_OK:
        raise PstError(status, lib.pst_last_error().decode())


def _ptr(x) -> int | None:
    """Device/host address of a torch tensor or numpy array (None passes NULL)."""
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        assert x.flags["C_CONTIGUOUS"]
        return x.ctypes.data
    assert x.is_contiguous(), "tensors must be contiguous"
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _tokens(tokens) -> np.ndarray:
    if hasattr(tokens, "numpy"):
        tokens = tokens.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))


class Pool:
    """A pst_pool handle.  device=-1 makes a host-only pool (tree and tables only)."""

    def __init__(self, n_q_heads: int, n_kv_heads: int, head_dim: int, chunk_size: int, max_chunks: int,
                 dtype: str = "f16", min_share: int = 0, max_seqs: int = 0, flags: int = 0, device: int = 0,
                 n_layers: int = 0):
        self.cfg = pst_config(n_q_heads, n_kv_heads, head_dim, chunk_size, max_chunks, DTYPE_CODES[dtype],
                              min_share, max_seqs, flags, n_layers)
        self.dtype = dtype
        self.device = device
        h = c_void_p()
        check(lib.pst_pool_create(byref(self.cfg), device, byref(h)))
        self.h = h

    def close(self) -> None:
        if self.h:
            check(lib.pst_pool_free(self.h))
            self.h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- tree operations
    def match(self, tokens) -> int:
        t = _tokens(tokens)
        n = c_int64()
        check(lib.pst_match(self.h, _ptr(t), len(t), byref(n)))
        return n.value

    def insert(self, tokens, k=None, v=None, stream=None):
        t = _tokens(tokens)
        sid, m = c_int64(), c_int64()
        check(lib.pst_insert(self.h, _ptr(t), len(t), _ptr(k), _ptr(v), _stream(stream) if k is not None else None,
                             byref(sid), byref(m)))
        return sid.value, m.value

    def append(self, seq_id: int, token: int, k=None, v=None, stream=None) -> None:
        check(lib.pst_append(self.h, seq_id, token, _ptr(k), _ptr(v), _stream(stream) if k is not None else None))

    def append_batch(self, seq_ids, tokens, k=None, v=None, stream=None) -> None:
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        t = _tokens(tokens)
        check(lib.pst_append_batch(self.h, len(ids), _ptr(ids), _ptr(t), _ptr(k), _ptr(v),
                                   _stream(stream) if k is not None else None))

    def remove(self, seq_id: int) -> None:
        check(lib.pst_remove(self.h, seq_id))

    def batch_order(self) -> list:
        b = c_int64()
        check(lib.pst_batch_order(self.h, None, 0, byref(b)))
        out = np.zeros(max(1, b.value), dtype=np.int64)
        check(lib.pst_batch_order(self.h, _ptr(out), len(out), byref(b)))
        return out[:b.value].tolist()

    def seq_length(self, seq_id: int) -> int:
        n = c_int64()
        check(lib.pst_seq_length(self.h, seq_id, byref(n)))
        return n.value

    # ---- attention
    def decode_attention(self, q, out, stream=None) -> None:
        check(lib.pst_decode_attention(self.h, _ptr(q), _ptr(out), _stream(stream)))

    def decode_attention_noalloc(self, q, out, stream=None) -> None:
        """pst_decode_attention_noalloc: same result, scratch in the library's fixed device area."""
        check(lib.pst_decode_attention_noalloc(self.h, _ptr(q), _ptr(out), _stream(stream)))

    def decode_attention_graph(self, q, out, stream=None) -> None:
        """pst_decode_attention_graph: same result, the step replayed from a CUDA graph."""
        check(lib.pst_decode_attention_graph(self.h, _ptr(q), _ptr(out), _stream(stream)))

    def decode_attention_host(self, q_host, out_host, stream=None) -> None:
        check(lib.pst_decode_attention_host(self.h, _ptr(q_host), _ptr(out_host), _stream(stream)))

    def prefill_attend(self, seq_id: int, tokens, q, k_new, v_new, out, stream=None) -> None:
        t = _tokens(tokens)
        check(lib.pst_prefill_attend(self.h, seq_id, _ptr(t), len(t), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out),
                                     _stream(stream)))

    def gather_kv(self, seq_id: int, k_out, v_out, stream=None) -> None:
        check(lib.pst_gather_kv(self.h, seq_id, _ptr(k_out), _ptr(v_out), _stream(stream)))

    # ---- one layer at a time (pools with n_layers > 1)
    def extend(self, seq_id: int, tokens) -> None:
        """pst_extend: append a block of tokens to the tree only."""
        t = _tokens(tokens)
        check(lib.pst_extend(self.h, seq_id, _ptr(t), len(t)))

    def write_kv(self, layer: int, seq_id: int, k, v, stream=None) -> None:
        """pst_write_kv: layer `layer`'s K/V of the sequence's last k.shape[0] tokens."""
        check(lib.pst_write_kv(self.h, layer, seq_id, k.shape[0], _ptr(k), _ptr(v), _stream(stream)))

    def write_kv_last(self, layer: int, seq_ids, k, v, stream=None) -> None:
        """pst_write_kv_last: layer `layer`'s K/V of each sequence's last token."""
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        check(lib.pst_write_kv_last(self.h, layer, len(ids), _ptr(ids), _ptr(k), _ptr(v), _stream(stream)))

    def decode_attention_layer(self, layer: int, q, out, stream=None) -> None:
        check(lib.pst_decode_attention_layer(self.h, layer, _ptr(q), _ptr(out), _stream(stream)))

    def decode_attention_graph_layer(self, layer: int, q, out, stream=None) -> None:
        """pst_decode_attention_graph_layer: one captured step per layer."""
        check(lib.pst_decode_attention_graph_layer(self.h, layer, _ptr(q), _ptr(out), _stream(stream)))

    def prefill_attend_layer(self, layer: int, seq_id: int, p0: int, q, out, stream=None) -> None:
        check(lib.pst_prefill_attend_layer(self.h, layer, seq_id, p0, q.shape[0], _ptr(q), _ptr(out),
                                           _stream(stream)))

    # ---- introspection
    def export_tables(self):
        ns, ne, b = c_int64(), c_int64(), c_int64()
        check(lib.pst_export_tables(self.h, None, 0, byref(ns), None, 0, byref(ne), None, 0, byref(b)))
        shared = np.zeros((max(1, ns.value), 4), dtype=np.int32)
        ent = np.zeros((max(1, ne.value), 2), dtype=np.int32)
        offs = np.zeros(b.value + 1, dtype=np.int64)
        check(lib.pst_export_tables(self.h, _ptr(shared), ns.value, byref(ns), _ptr(ent), ne.value, byref(ne),
                                    _ptr(offs), len(offs), byref(b)))
        shared = [tuple(int(x) for x in r) for r in shared[:ns.value]]
        per_seq = [[tuple(int(x) for x in r) for r in ent[offs[u]:offs[u + 1]]] for u in range(b.value)]
        return shared, per_seq

    def stats(self) -> dict:
        s = pst_stats_t()
        check(lib.pst_stats(self.h, byref(s)))
        return {name: getattr(s, name) for name, _ in pst_stats_t._fields_}

    def set_profiling(self, enable: bool) -> None:
        check(lib.pst_set_profiling(self.h, 1 if enable else 0))

    def phase_times(self):
        ms = (c_float * 3)()
        check(lib.pst_phase_times(self.h, ms))
        return list(ms)

    def last_launch_count(self) -> int:
        n = c_int32()
        check(lib.pst_last_launch_count(self.h, byref(n)))
        return n.value

    def check_device(self) -> int:
        code = c_int32()
        st = lib.pst_check_device(self.h, byref(code))
        if st not in (PST_OK, PST_ERR_DEVICE):
            check(st)
        return code.value


def version() -> str:
    return lib.pst_version().decode()
