"""Block-sparse GQA decode attention with learned block selection, for GB300 (sm_103a).

The compute path is a C-ABI CUDA library (``libsparsepool.so``, declared in
``include/sparse_pool.h``); ``binding`` is its thin ctypes binding on torch tensors.
``workloads`` draws the seeded synthetic inputs.  Nothing here falls back to the CPU:
a call without the built library raises.
"""
