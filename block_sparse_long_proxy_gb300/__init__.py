"""libmsa: MiniMax Sparse Attention hot path on GB300 (sm_103a).

The compute lives in the CUDA library libmsa.so (built by
__graft_entry__.build()); `block_sparse_long_proxy_gb300.msa` is its thin
ctypes binding.  `synth` draws seeded synthetic inputs.
"""
