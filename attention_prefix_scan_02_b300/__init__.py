"""B300-native softmax-attention prefix scan (Aaren many-to-many output).

The compute path is the CUDA library libaaren.so (built for sm_103a, C ABI in
include/aaren.h).  The Python binding in `binding` only marshals torch tensors
into that ABI; importing this package does not load the library, the first
call does, and it raises if the library is missing (there is no CPU fallback).
"""

__all__ = ["binding", "inputs"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
