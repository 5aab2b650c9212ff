"""Paged KV-cache decode for GB300 (sm_103a).

The product is the C-ABI library ``_lib/libpagedkv.so`` (sources in ``csrc/``,
declarations in ``include/pa.h``).  ``_native`` binds it with ctypes under the
same function names; ``pool.KVPool`` passes PyTorch device memory and streams to
it.  ``workloads`` draws the seeded synthetic inputs used by tests and the
benchmark.
"""
import importlib

from . import _native, workloads  # noqa: F401
from ._native import PAError  # noqa: F401

__all__ = ["_native", "PAError", "KVPool", "workloads"]


def __getattr__(name):
    if name == "KVPool":
        return importlib.import_module(".pool", __name__).KVPool
    raise AttributeError(name)
