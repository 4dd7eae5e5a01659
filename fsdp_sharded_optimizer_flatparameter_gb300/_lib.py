"""Locates and loads ``libzs.so``; fails loudly when it is missing."""

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libzs.so")


def load_library():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            "libzs.so is not built (%s). Build it with "
            "`python fsdp_sharded_optimizer_flatparameter_gb300/_build.py` "
            "or `python -c 'import __graft_entry__ as g; g.build()'`; there is no fallback." % LIB_PATH)
    # torch first, so the CUDA runtime it ships is the one the library binds to
    try:
        import torch  # noqa: F401
    except ImportError:
        pass
    return ctypes.CDLL(LIB_PATH, mode=ctypes.RTLD_GLOBAL)
