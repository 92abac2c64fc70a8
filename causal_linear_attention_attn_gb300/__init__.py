"""GB300 (sm_103a) normalized linear attention with the ELU(x)+1 feature map.

The compute path is the C-ABI library ``liblinattn.so`` (hand-written CUDA,
see ``csrc/``); :mod:`.linattn` is its thin ctypes binding and
:mod:`.inputs` the seeded synthetic workloads.  Importing this package does
not load the library; importing :mod:`.linattn` does, and fails loudly if it
has not been built.
"""
__all__ = ["inputs", "linattn"]
