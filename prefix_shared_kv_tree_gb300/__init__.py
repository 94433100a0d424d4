"""GB300-native prefix-shared KV-tree decode attention (ChunkAttention).

The compute path lives in the C-ABI library ``libpst.so`` (hand-written CUDA
for sm_103a plus a C++ prefix-tree manager).  ``prefix_shared_kv_tree_gb300.pst``
is the thin ctypes binding; importing it loads the library and fails loudly
when it has not been built.  ``workloads`` draws the seeded synthetic inputs.
"""
__all__ = ["pst", "workloads"]
