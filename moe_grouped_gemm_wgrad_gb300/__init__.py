"""Grouped MoE backward GEMMs for GB300 (sm_103a): MXFP8 quantize, MXFP8 grouped
wgrad and fp32 grouped dgrad, as a C-ABI CUDA library (``libmgw.so``) with a thin
ctypes binding (:mod:`moe_grouped_gemm_wgrad_gb300.mgw`).

Importing this package loads nothing; the library is loaded on first use and a
missing or unbuilt library raises instead of falling back to anything else.
"""
