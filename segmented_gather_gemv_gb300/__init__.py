"""GB300-native multi-LoRA delta path (Punica-style segmented gather GEMV).

``y += scale_a * (x . A_a^T) . B_a^T`` for a batch in which every token row
routes to its own adapter ``a`` in a contiguous adapter pool, computed by
hand-written sm_103a CUDA kernels behind a C ABI (``include/lora_sgmv.h``).

Submodules:
  ``binding``    thin ctypes binding of the C ABI (same call names);
  ``build``      compiles the CUDA library in-tree for sm_103a;
  ``workloads``  seeded synthetic inputs (no method arithmetic).

Importing the package does not load the CUDA library; the first call into
``binding`` does, and raises if the library has not been built.
"""
import importlib

__all__ = ["binding", "build", "workloads"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module("." + name, __name__)
    raise AttributeError(name)
