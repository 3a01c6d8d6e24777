"""Routed int4 MoE layer for NVIDIA B300 (sm_103a).

The compute path is the C-ABI library ``libmoe_int4.so`` (hand-written CUDA
kernels) loaded by :mod:`int4_routed_expert_06_b300.binding`; this package
adds the ctypes binding and seeded synthetic inputs (:mod:`.synth`).
"""
__all__ = ["binding", "synth"]
