"""GB300-native masked time-RoPE attention for request-centric ranking sequences.

The compute path is the CUDA library ``librec_attn.so`` (sources in ``csrc/``,
C-ABI declared in ``include/rec_attn.h``); ``binding`` marshals torch tensors
into that C-ABI.  Nothing here computes attention on the CPU: if the library is
missing, calls raise.

Submodules are imported lazily so that ``workloads`` (seeded input generators)
can be used without loading CUDA.
"""
__all__ = ["binding", "workloads", "build", "sharding"]
