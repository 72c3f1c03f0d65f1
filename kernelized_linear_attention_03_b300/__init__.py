"""KATA causal normalised linear-attention forward on B300 (sm_103a).

The compute lives in ``libkata.so`` (hand-written CUDA behind a C ABI declared
in ``include/kata.h``); ``binding`` marshals torch tensors into those calls.
``inputs`` holds the seeded synthetic workloads.
"""
