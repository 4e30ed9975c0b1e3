"""Routed Mixture-of-Experts expert execution on one GB300 (sm_103a).

The compute lives in ``libmoe.so`` (C ABI: ``include/moe.h``; CUDA sources in
``csrc/``): local dispatch, tcgen05 grouped GEMMs with a fused SiLU(gate)*up
epilogue, and the weighted top-k combine. ``binding`` wraps it with ctypes
for PyTorch device buffers; ``build`` compiles it in-tree with nvcc.
"""
