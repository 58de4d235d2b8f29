"""Ulysses sequence-parallel attention on one GB300: P virtual ranks in one HBM.

The compute path is the C-ABI library ``libulysses.so`` (hand-written sm_103a
CUDA kernels); this package is the thin ctypes binding over it.
"""
