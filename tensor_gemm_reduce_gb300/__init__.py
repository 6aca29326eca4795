"""Fused GEMM + reduce-scatter (row-parallel linear, 8 virtual ranks) for GB300.

The compute path is the CUDA library built from csrc/ (see build.py); the
binding in gemm_rs.py is imported lazily so that the workload generator can be
used without the library.
"""
__all__ = ["workloads", "gemm_rs", "metrics", "build"]


def __getattr__(name):
    import importlib
    if name in __all__:
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
