"""libpagedattn: paged KV-cache attention under continuous batching, for GB300 (sm_103a).

The compute path is the C-ABI library ``libpagedattn.so`` (hand-written CUDA
kernels, built in-tree by ``build.py``); ``binding`` is a thin ctypes layer
that passes torch tensors' device pointers and the current stream to it.
"""
