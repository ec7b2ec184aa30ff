"""GB300-native DSA indexer: paged index-key store and streaming score + top-k.

The compute path is libdsaidx.so (CUDA, sm_103a), reached through the C ABI
in include/dsaidx.h; `dsaidx` is the Python binding over it.
"""
from .dsaidx import (FMT_BF16, FMT_FP4, FMT_FP8, HEADS, HEAD_DIM, PAGE_SIZE, Context, DsaError, lib,
                     page_bytes, status_str)

__all__ = ["FMT_BF16", "FMT_FP8", "FMT_FP4", "HEADS", "HEAD_DIM", "PAGE_SIZE", "Context", "DsaError",
           "lib", "page_bytes", "status_str"]
