"""Seeded synthetic inputs shared by the CPU oracle and the CUDA path.

Nothing here computes any part of the cache method: this module only produces
the data a decode step consumes --
  * top-k selection traces that stand in for the sparse-attention indexer
    (HiSparse blog summary, §3 "indexer-agnostic" and §4 "selection has
    locality"): `drift_traces`;
  * bf16 query vectors and KV records drawn from N(0, 1): `normal_bf16`.
The trace generator is plain C (tracegen.c) compiled with gcc on first use.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tracegen.c")
_SO = os.path.join(_HERE, "_tracegen.so")
_lock = threading.Lock()
_lib = None


def build() -> str:
    """Compile tracegen.c into a shared object next to it (rebuilt when the source is newer)."""
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
            lib.tg_drift_traces.restype = ctypes.c_int
            lib.tg_drift_traces.argtypes = [
                ctypes.c_uint64, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                ctypes.c_int, ctypes.c_double, ctypes.c_int64, ctypes.c_void_p]
            for name in ("tg_xoshiro_stream", "tg_splitmix_stream"):
                fn = getattr(lib, name)
                fn.restype = None
                fn.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p]
            _lib = lib
    return _lib


@dataclass(frozen=True)
class TraceSpec:
    """Shape of a drifting top-k trace.

    ctx0: positions that exist before step 0.  appends: the context grows by one
    token per step (the token appended at step t is position ctx0 + t and is
    always selected).  Without appends the newest position is ctx0 - 1.
    """
    ctx0: int
    k: int
    steps: int
    keep: float = 0.9
    recency_mean: float = 512.0
    recency_share: float = 0.7
    appends: bool = False
    burst_every: int = 0
    burst_frac: float = 0.4
    far_gap: int = 0


def drift_traces(spec: TraceSpec, num_requests: int, num_layers: int, seed: int) -> np.ndarray:
    """int32 array [steps][num_layers][num_requests][k] of distinct positions per row."""
    lib = _load()
    out = np.empty((spec.steps, num_layers, num_requests, spec.k), dtype=np.int32)
    rc = lib.tg_drift_traces(
        ctypes.c_uint64(seed & 0xFFFFFFFFFFFFFFFF), num_requests, num_layers, spec.ctx0,
        int(spec.appends), spec.k, spec.steps, spec.keep, spec.recency_mean, spec.recency_share,
        spec.burst_every, spec.burst_frac, spec.far_gap, out.ctypes.data)
    if rc != 0:
        raise ValueError(f"trace generator rejected {spec}")
    return out


def xoshiro256ss_stream(seed: int, n: int) -> np.ndarray:
    lib = _load()
    out = np.empty(n, dtype=np.uint64)
    lib.tg_xoshiro_stream(ctypes.c_uint64(seed), n, out.ctypes.data)
    return out


def splitmix64_stream(seed: int, n: int) -> np.ndarray:
    lib = _load()
    out = np.empty(n, dtype=np.uint64)
    lib.tg_splitmix_stream(ctypes.c_uint64(seed), n, out.ctypes.data)
    return out


def normal_bf16(shape, seed: int, device="cpu"):
    """bf16 tensor of N(0, 1) draws from torch's generator seeded with `seed`.

    CPU and CUDA generators give different streams; a test uses one of them and
    hands the same tensor to both sides.
    """
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
