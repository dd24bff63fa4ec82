"""GB300 (sm_103a) MXFP4 grouped MoE library: route sort, W4A16 grouped GEMM,
SwiGLU and deterministic combine behind a C ABI (``include/moe_mxfp4.h``).

Submodules:
  binding    ctypes binding of the C ABI (torch tensors in, CUDA kernels run)
  build_lib  in-tree nvcc build of ``_build/libmoe_mxfp4.so``
  inputs     seeded synthetic workloads (random numbers and byte layouts only)

The binding is imported lazily so that ``inputs`` can be used without torch or
a GPU.
"""

__all__ = ["binding", "build_lib", "inputs"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
