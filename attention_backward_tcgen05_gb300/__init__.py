"""fab: fused attention backward (ggml_flash_attn_back semantics) for GB300.

The compute path is a C-ABI CUDA library (``libfab.so``, built for sm_103a)
declared in ``include/fab.h``; ``binding`` marshals torch tensors into it.
``inputs`` draws the seeded synthetic workloads.
"""
