"""CPU oracle for the HiSparse decode hot path -- TEST INFRASTRUCTURE ONLY.

Only `tests/`, the package smoke check and the benchmark's CPU-baseline leg may
import this module.  The product (the CUDA library and its Python binding)
never imports or calls it, and the two share no code: the oracle is plain C
(hs_oracle.c, single-threaded, fp64 attention) compiled here with gcc.

What it follows (blog summary of "HiSparse: Scaling Sparse-Attention Decoding
with Hierarchical KV Cache Management"):
  * `Cache.resolve`   -- §3 (resolve the top-k against a B-slot buffer, keep hits,
                         swap in misses, evict) and §5 (hits to MRU, misses after
                         the hits, in-place LRU; never rebuild from the top-k);
  * policies          -- §4 (LRU, FIFO, random, swap-vanilla; Belady offline);
  * `Cache.append`    -- §3 step (5) (write-through of the new token's KV);
  * `attention`       -- §3 "exact": attention over exactly the selected positions.
Pins: tests/test_oracle_*.py check every function against brute force, closed
forms and invariants.  Parity unpinned: the absolute miss rates of the pages'
replayed traces (the traces are not available); only the policies' order is
compared.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hs_oracle.c")
_SO = os.path.join(_HERE, "_hs_oracle.so")
_lock = threading.Lock()
_lib = None

LRU, FIFO, RANDOM, SWAP = 0, 1, 2, 3
POLICY = {"lru": LRU, "fifo": FIFO, "random": RANDOM, "swap": SWAP}
ERR_RANGE, ERR_DUP, ERR_CLOCK, ERR_APPEND, ERR_SLOTS = 1, 2, 4, 8, 128


def build() -> str:
    """Compile the oracle with gcc (plain C11, -O2, no fast-math)."""
    if not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I, I64, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64
            lib.orc_cache_new.restype = P
            lib.orc_cache_new.argtypes = [I, I, I, U64, I, I, I, I, I64]
            lib.orc_set_cap.restype = I
            lib.orc_set_cap.argtypes = [P, I]
            lib.orc_cache_free.restype = None
            lib.orc_cache_free.argtypes = [P]
            lib.orc_resolve.restype = I
            lib.orc_resolve.argtypes = [P, P, P]
            lib.orc_append.restype = I
            lib.orc_append.argtypes = [P, I64]
            lib.orc_get_slots.restype = None
            lib.orc_get_slots.argtypes = [P, P, P]
            lib.orc_get_counters.restype = None
            lib.orc_get_counters.argtypes = [P, P]
            lib.orc_validate.restype = ctypes.c_uint32
            lib.orc_validate.argtypes = [P, I, I64, P]
            lib.orc_belady.restype = I64
            lib.orc_belady.argtypes = [I, I, I, I64, P, P]
            lib.orc_attention.restype = None
            lib.orc_attention.argtypes = [I, I, I, I, P, P, I64, I64, P, I, ctypes.c_double, P]
            _lib = lib
    return _lib


class Cache:
    """The B-slot hot buffer of one (request r, layer l) in a pool of R x L."""

    def __init__(self, B, k, policy="lru", seed=0, R=1, L=1, r=0, l=0, C=1 << 20):
        self.lib = _load()
        pol = POLICY[policy] if isinstance(policy, str) else int(policy)
        self.B, self.k = int(B), int(k)
        self._h = self.lib.orc_cache_new(self.B, self.k, pol, ctypes.c_uint64(seed & (2**64 - 1)),
                                         R, L, r, l, int(C))
        if not self._h:
            raise ValueError("bad oracle cache parameters")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self.lib.orc_cache_free(h)
            self._h = None

    def resolve(self, S):
        S = np.ascontiguousarray(S, dtype=np.int32)
        assert S.shape == (self.k,)
        locs = np.empty(self.k, dtype=np.int32)
        m = self.lib.orc_resolve(self._h, S.ctypes.data, locs.ctypes.data)
        return m, locs

    def append(self, p):
        return self.lib.orc_append(self._h, int(p))

    def set_cap(self, cap):
        """The buffer now holds slots [0, cap) only (a buffer grown on demand)."""
        if self.lib.orc_set_cap(self._h, int(cap)) != 0:
            raise ValueError("cap outside [0, B]")

    def slots(self):
        tag = np.empty(self.B, dtype=np.int32)
        stamp = np.empty(self.B, dtype=np.uint32)
        self.lib.orc_get_slots(self._h, tag.ctypes.data, stamp.ctypes.data)
        return tag, stamp

    def counters(self):
        out = np.empty(6, dtype=np.uint64)
        self.lib.orc_get_counters(self._h, out.ctypes.data)
        keys = ("clock", "nres", "err", "hits", "misses", "appends")
        return {k_: int(v) for k_, v in zip(keys, out)}


def validate(S, C):
    lib = _load()
    S = np.ascontiguousarray(S, dtype=np.int32)
    valid = np.empty(S.shape[0], dtype=np.uint8)
    err = lib.orc_validate(S.ctypes.data, S.shape[0], int(C), valid.ctypes.data)
    return valid.astype(bool), int(err)


def belady(B, trace, C):
    """Offline-optimal miss counts per step for a no-append trace [T][k]."""
    lib = _load()
    trace = np.ascontiguousarray(trace, dtype=np.int32)
    T, k = trace.shape
    misses = np.empty(T, dtype=np.int32)
    lib.orc_belady(int(B), int(k), int(T), int(C), trace.ctypes.data, misses.ctypes.data)
    return misses


def attention(q_bits, hist_bits, S, scale, kv_heads, Dqk, Dv):
    """fp64 attention of q [Hq][Dqk] over history rows S of hist [C][rec_elems] (bf16 bit patterns
    as uint16).  kv_heads = 0 selects the shared-latent (MLA) record layout."""
    lib = _load()
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    hist_bits = np.ascontiguousarray(hist_bits, dtype=np.uint16)
    S = np.ascontiguousarray(S, dtype=np.int32)
    Hq = q_bits.shape[0]
    assert q_bits.shape[1] == Dqk
    C, rec_elems = hist_bits.shape
    out = np.empty((Hq, Dv), dtype=np.float64)
    lib.orc_attention(Hq, int(kv_heads), int(Dqk), int(Dv), q_bits.ctypes.data, hist_bits.ctypes.data,
                      int(rec_elems), int(C), S.ctypes.data, int(S.shape[0]), float(scale), out.ctypes.data)
    return out
