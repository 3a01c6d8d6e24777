"""CPU oracle of the routed int4 MoE layer: test infrastructure only.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline and
reference legs import this package; the CUDA package never does.
"""
