"""tiled_mma_atom_gb300 — tiled GEMM D = A·Bᵀ (fp32 accumulate) for GB300.

The compute path is a C-ABI shared library of hand-written sm_103a CUDA
(``csrc/``, built into ``libtmg.so``); this package only marshals torch
tensors into that library's calls.  Importing the package does not load the
library; the first call does, and fails loudly if it is missing.
"""
