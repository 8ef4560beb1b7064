"""GB300-native routed-MoE FFN decode step on Q8_0 experts (libluce_moe).

The compute path is the CUDA library ``lib/libluce_moe.so`` (C ABI in
``include/luce_moe.h``), reached through :mod:`.binding`.  Importing this
package loads nothing; the library is loaded on the first call and a
missing build raises instead of falling back to anything.

Submodules: ``build`` (nvcc build), ``binding`` (ctypes, same names as the
C ABI), ``layer`` (torch-owned buffers for one step), ``workloads`` (seeded
synthetic inputs).
"""

__all__ = ["build", "binding", "layer", "workloads"]
