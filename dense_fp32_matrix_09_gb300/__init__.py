"""GB300-native single-precision GEMM: C = alpha*A*B + beta*C (row-major).

The computation lives in the CUDA library ``libsgemm.so`` (sources under
``csrc/``), reached through its C ABI (``include/sgemm.h``).  ``sgemm`` is the
ctypes binding with the same entry-point names; ``inputs`` draws seeded
synthetic problems.  The binding is loaded on first use so that modules which
only need the input generators import without the compiled library.
"""
__all__ = ["sgemm", "inputs"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
