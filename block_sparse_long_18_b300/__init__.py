"""Sparse GQA full-attention layer (block indexer -> top-k block selection -> gated
sparse attention) on NVIDIA B300 (sm_103a).

The compute path is the CUDA library ``csrc/`` builds into ``libsgqa.so`` behind a C ABI
(``include/sgqa.h``); ``block_sparse_long_18_b300.sgqa`` is its thin Python binding.
``block_sparse_long_18_b300.inputs`` draws the seeded synthetic workloads.
"""
__version__ = "0.1.0"
