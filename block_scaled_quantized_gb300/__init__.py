"""GB300-native residue-compensated block-scaled FP4 linear layers.

The compute path is librs (C ABI, hand-written sm_103a CUDA): a fused
activation + residue quantizer and a tcgen05 block-scaled GEMM with on-chip
Fold.  ``rs`` is the ctypes binding; ``workloads`` draws seeded synthetic
inputs; ``build`` compiles librs in-tree.
"""
