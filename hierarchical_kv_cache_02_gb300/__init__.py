"""GB300-native decode hot path of HiSparse (hierarchical KV cache for sparse-attention decoding).

The compute lives in libhisparse.so (hand-written sm_103a CUDA behind the C ABI of
include/hisparse.h); this package is its thin Python binding plus the seeded input
generators used by tests and benchmarks.
"""
from ._lib import (DEVERR_APPEND, DEVERR_CLOCK, DEVERR_DUP, DEVERR_LOC, DEVERR_PAGE, DEVERR_RANGE, DEVERR_SLOTS,
                   DEVERR_TIMEOUT, LAYOUT_GQA, LAYOUT_MLA, POLICY_FIFO, POLICY_LRU, POLICY_RANDOM, POLICY_SWAP_VANILLA)
from .pool import HsConfig, HsError, HsPool

__all__ = ["HsConfig", "HsPool", "HsError", "LAYOUT_MLA", "LAYOUT_GQA", "POLICY_LRU", "POLICY_FIFO",
           "POLICY_RANDOM", "POLICY_SWAP_VANILLA", "DEVERR_RANGE", "DEVERR_DUP", "DEVERR_CLOCK",
           "DEVERR_APPEND", "DEVERR_LOC", "DEVERR_TIMEOUT", "DEVERR_PAGE",
           "DEVERR_SLOTS"]
