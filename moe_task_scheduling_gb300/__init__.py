"""Event-Tensor MoE megakernel for GB300 (sm_103a).

The compute path is the C-ABI library libetmoe.so (hand-written CUDA);
`etmoe` is its thin ctypes binding and `workloads` draws seeded synthetic
inputs.  Importing the package loads nothing; `etmoe.load()` opens the
library and raises if it is missing.
"""
__all__ = ["etmoe", "workloads"]
