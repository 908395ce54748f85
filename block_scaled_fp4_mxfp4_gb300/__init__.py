"""Block-scaled FP4 (MXFP4 / NVFP4) quantization and GEMM for GB300 (sm_103a).

The compute path is the C-ABI library ``libmxfp4.so`` built from ``csrc/``
(declared in ``include/mxfp4.h``); ``block_scaled_fp4_mxfp4_gb300.mxfp4`` is its
thin Python binding. Importing this package does not load the library, so the
seeded input generators in ``workloads`` stay usable without a GPU.
"""
__version__ = "0.1.0"
