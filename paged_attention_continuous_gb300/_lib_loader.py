"""Locate and load the in-tree ``_lib/libcb.so``; fail loudly if it is absent."""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libcb.so")


def load_library() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build the CUDA library first with "
            "`python paged_attention_continuous_gb300/build.py` (there is no CPU fallback)")
    return ctypes.CDLL(LIB_PATH, mode=ctypes.RTLD_GLOBAL)
