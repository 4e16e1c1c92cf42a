"""GB300-native grouped-query attention: prefill and split-KV decode.

The compute path is the CUDA library ``libgqa_attn.so`` (sources under
``csrc/``, C ABI in ``include/gqa_attn.h``). The Python side is argument
marshalling only: ``ops`` binds the C ABI through ctypes, ``inputs`` draws
seeded synthetic tensors, ``build`` compiles the library with nvcc.

Nothing here falls back to a CPU or PyTorch computation: if the library is
missing, the ops raise.
"""

__all__ = ["ops", "inputs", "build"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
