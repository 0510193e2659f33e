"""Purlin collectives on one GB300: R logical ranks in one GPU's memory.

The library is libpurlin1 (C ABI in include/purlin.h, CUDA kernels for
sm_103a); ``copy_reduce_datapath_gb300.purlin`` is its Python binding.  The
binding is loaded lazily so that ``import copy_reduce_datapath_gb300`` works
before the library is built; touching ``purlin`` without the built library
raises ImportError.
"""
import importlib

__all__ = ["purlin", "build"]


def __getattr__(name):
    if name in ("purlin", "build"):
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
