"""Python binding of the HiSparse hot-path library: a thin wrapper over the C ABI.

Every method only checks and marshals its arguments (PyTorch tensors -> raw pointers plus
the current CUDA stream) and calls the matching hs_* entry point; all work runs in the
library's CUDA kernels.
"""
from __future__ import annotations

import ctypes
import math
from dataclasses import dataclass, fields

import numpy as np

from . import _lib


class HsError(RuntimeError):
    def __init__(self, call: str, status: int):
        super().__init__(f"{call} returned {_lib.STATUS_NAMES.get(status, status)}")
        self.status = status


def _check(call, status):
    if status != _lib.HS_OK:
        raise HsError(call, status)


@dataclass
class HsConfig:
    num_requests: int
    num_layers: int
    capacity: int
    layout: int = _lib.LAYOUT_GQA
    num_q_heads: int = 32
    num_kv_heads: int = 8
    head_dim_qk: int = 128
    head_dim_v: int = 128
    top_k: int = 2048
    buffer_slots: int = 4096
    policy: int = _lib.POLICY_LRU
    seed: int = 0
    io_chunk_bytes: int = 64
    log_steps: int = 0
    shared_prefix: int = 0
    fetch_in_attention: int = 0
    host_page_tokens: int = 0
    host_on_demand: int = 0
    buffer_page_slots: int = 0
    device_pool_slots: int = 0
    host_to_device_ratio: float = 0.0
    early_fetch: int = 0

    @property
    def record_bytes(self) -> int:
        if self.layout == _lib.LAYOUT_MLA:
            return 2 * self.head_dim_qk
        return 2 * self.num_kv_heads * (self.head_dim_qk + self.head_dim_v)

    @property
    def record_elems(self) -> int:
        return self.record_bytes // 2

    @property
    def default_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim_qk)

    def to_c(self) -> _lib.hs_config:
        c = _lib.hs_config()
        for f in fields(self):
            v = getattr(self, f.name)
            setattr(c, f.name, float(v) if f.name == "host_to_device_ratio" else int(v))
        return c


def _stream_ptr(stream, device):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _dev_tensor(t, dtype, shape, name, device):
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda" or t.device.index != device:
        raise ValueError(f"{name} must live on cuda:{device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


class HsPool:
    """One pool: host history, hot buffers and metadata for R requests x L layers."""

    def __init__(self, cfg: HsConfig, device: int = 0):
        self.lib = _lib.load()
        self.cfg = cfg
        self.device = int(device)
        self._c = cfg.to_c()
        h = ctypes.c_void_p()
        _check("hs_pool_create", self.lib.hs_pool_create(ctypes.byref(self._c), self.device, ctypes.byref(h)))
        self._h = h

    # -- lifecycle -------------------------------------------------------------
    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            self.lib.hs_pool_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def reset(self, stream=None):
        _check("hs_pool_reset", self.lib.hs_pool_reset(self._h, _stream_ptr(stream, self.device)))

    # -- setup -----------------------------------------------------------------
    def prefill(self, req: int, layer: int, pos0: int, records, stream=None):
        """records: bf16 [n][record_elems] on the host or on this device (contiguous)."""
        import torch

        if records.dtype != torch.bfloat16 or records.dim() != 2 or records.shape[1] != self.cfg.record_elems:
            raise ValueError("records must be bf16 [n][record_elems]")
        if not records.is_contiguous():
            raise ValueError("records must be contiguous")
        if records.device.type == "cuda" and records.device.index != self.device:
            raise ValueError("device records must be on the pool's device")
        st = _stream_ptr(stream, self.device)
        _check("hs_prefill_write", self.lib.hs_prefill_write(self._h, int(req), int(layer), int(pos0),
                                                             int(records.shape[0]), ctypes.c_void_p(records.data_ptr()), st))
        torch.cuda.current_stream(self.device).synchronize() if stream is None else stream.synchronize()

    # -- the capturable hot path --------------------------------------------------
    def append(self, layer: int, pos, rec, stream=None):
        import torch

        R = self.cfg.num_requests
        p = _dev_tensor(pos, torch.int64, (R,), "pos", self.device)
        r = _dev_tensor(rec, torch.bfloat16, (R, self.cfg.record_elems), "rec", self.device)
        _check("hs_append_writethrough", self.lib.hs_append_writethrough(self._h, int(layer), p, r,
                                                                         _stream_ptr(stream, self.device)))

    def resolve(self, layer: int, topk, locs=None, stream=None):
        import torch

        R, k = self.cfg.num_requests, self.cfg.top_k
        t = _dev_tensor(topk, torch.int32, (R, k), "topk", self.device)
        if locs is None:
            locs = torch.empty((R, k), dtype=torch.int32, device=f"cuda:{self.device}")
        lo = _dev_tensor(locs, torch.int32, (R, k), "locs", self.device)
        _check("hs_resolve", self.lib.hs_resolve(self._h, int(layer), t, lo, _stream_ptr(stream, self.device)))
        return locs

    def append_resolve(self, layer: int, pos, rec, topk, locs=None, stream=None):
        """append(layer, pos, rec) then resolve(layer, topk, locs), fused into one kernel."""
        import torch

        c = self.cfg
        R, k = c.num_requests, c.top_k
        p = _dev_tensor(pos, torch.int64, (R,), "pos", self.device)
        rr = _dev_tensor(rec, torch.bfloat16, (R, c.record_elems), "rec", self.device)
        t = _dev_tensor(topk, torch.int32, (R, k), "topk", self.device)
        if locs is None:
            locs = torch.empty((R, k), dtype=torch.int32, device=f"cuda:{self.device}")
        lo = _dev_tensor(locs, torch.int32, (R, k), "locs", self.device)
        _check("hs_append_resolve", self.lib.hs_append_resolve(self._h, int(layer), p, rr, t, lo,
                                                               _stream_ptr(stream, self.device)))
        return locs

    def resolve_range(self, layer: int, r0: int, topk, locs=None, pos=None, rec=None, stream=None):
        """Resolve (after the fused append when pos and rec are given) requests [r0, r0 + n), n =
        topk.shape[0]; all tensors hold rows for those requests only."""
        import torch

        c = self.cfg
        n, k = int(topk.shape[0]), c.top_k
        t = _dev_tensor(topk, torch.int32, (n, k), "topk", self.device)
        if locs is None:
            locs = torch.empty((n, k), dtype=torch.int32, device=f"cuda:{self.device}")
        lo = _dev_tensor(locs, torch.int32, (n, k), "locs", self.device)
        p = rr = ctypes.c_void_p()
        if (pos is None) != (rec is None):
            raise ValueError("pos and rec go together")
        if pos is not None:
            p = _dev_tensor(pos, torch.int64, (n,), "pos", self.device)
            rr = _dev_tensor(rec, torch.bfloat16, (n, c.record_elems), "rec", self.device)
        _check("hs_resolve_range", self.lib.hs_resolve_range(self._h, int(layer), int(r0), n, p, rr, t, lo,
                                                             _stream_ptr(stream, self.device)))
        return locs

    def sparse_attn_range(self, layer: int, r0: int, q, locs, out=None, scale=None, stream=None):
        import torch

        c = self.cfg
        n = int(q.shape[0])
        qp = _dev_tensor(q, torch.bfloat16, (n, c.num_q_heads, c.head_dim_qk), "q", self.device)
        lp = _dev_tensor(locs, torch.int32, (n, c.top_k), "locs", self.device)
        if out is None:
            out = torch.empty((n, c.num_q_heads, c.head_dim_v), dtype=torch.float32, device=f"cuda:{self.device}")
        op = _dev_tensor(out, torch.float32, (n, c.num_q_heads, c.head_dim_v), "out", self.device)
        s = c.default_scale if scale is None else float(scale)
        _check("hs_sparse_attn_range", self.lib.hs_sparse_attn_range(self._h, int(layer), int(r0), n, qp, lp,
                                                                     ctypes.c_float(s), op,
                                                                     _stream_ptr(stream, self.device)))
        return out

    def sparse_attn(self, layer: int, q, locs, out=None, scale=None, kv=None, stream=None):
        """q bf16 [R][Hq][Dqk]; locs int32 [R][k]; out fp32 [R][Hq][Dv].  kv: optional resident
        bf16 [R][rows][record_elems] (then locs index its rows instead of the hot buffer)."""
        import torch

        c = self.cfg
        R = c.num_requests
        qp = _dev_tensor(q, torch.bfloat16, (R, c.num_q_heads, c.head_dim_qk), "q", self.device)
        lp = _dev_tensor(locs, torch.int32, (R, c.top_k), "locs", self.device)
        if out is None:
            out = torch.empty((R, c.num_q_heads, c.head_dim_v), dtype=torch.float32, device=f"cuda:{self.device}")
        op = _dev_tensor(out, torch.float32, (R, c.num_q_heads, c.head_dim_v), "out", self.device)
        kvp, rows = ctypes.c_void_p(), 0
        if kv is not None:
            if kv.dim() != 3:
                raise ValueError("kv must be [R][rows][record_elems]")
            rows = kv.shape[1]
            kvp = _dev_tensor(kv, torch.bfloat16, (R, rows, c.record_elems), "kv", self.device)
        s = c.default_scale if scale is None else float(scale)
        _check("hs_sparse_attn", self.lib.hs_sparse_attn(self._h, int(layer), qp, lp, kvp, int(rows),
                                                         ctypes.c_float(s), op, _stream_ptr(stream, self.device)))
        return out

    # -- counters and inspection (synchronous) --------------------------------------
    def stats(self, reset: bool = False, raise_on_error: bool = False):
        c = self.cfg
        R, L = c.num_requests, c.num_layers
        tot = _lib.hs_totals()
        cnt = np.zeros((R, L, 4), dtype=np.uint64)
        err = np.zeros((R, L), dtype=np.uint32)
        log = np.zeros((max(c.log_steps, 0), R, L), dtype=np.uint32)
        st = self.lib.hs_stats(self._h, ctypes.byref(tot), cnt.ctypes.data, err.ctypes.data,
                               log.ctypes.data if c.log_steps > 0 else None, int(bool(reset)))
        if st not in (_lib.HS_OK, _lib.HS_ERR_DEVICE_FLAG) or (raise_on_error and st != _lib.HS_OK):
            raise HsError("hs_stats", st)
        return {"hits": tot.hits, "misses": tot.misses, "appends": tot.appends, "host_bytes": tot.host_bytes,
                "error_bits": tot.error_bits, "resolves": tot.resolves, "status": st,
                "per_rl": cnt, "errors": err, "step_log": log}

    def read_state(self, layer: int):
        c = self.cfg
        tag = np.empty((c.num_requests, c.buffer_slots), dtype=np.int32)
        stamp = np.empty((c.num_requests, c.buffer_slots), dtype=np.uint32)
        clock = np.empty((c.num_requests,), dtype=np.uint32)
        _check("hs_read_state", self.lib.hs_read_state(self._h, int(layer), tag.ctypes.data, stamp.ctypes.data,
                                                       clock.ctypes.data))
        return tag, stamp, clock

    def read_buffer(self, req: int, layer: int):
        c = self.cfg
        out = np.empty((c.buffer_slots, c.record_elems), dtype=np.uint16)
        _check("hs_read_buffer", self.lib.hs_read_buffer(self._h, int(req), int(layer), out.ctypes.data))
        return out

    # -- memory layer: paged host pool ------------------------------------------------
    def reserve(self, req: int, end: int, layer: int = -1):
        """Reserve the host pages of (req, layer) covering positions [0, end) and, with a device cache
        pool, grow its buffer to min(B, max(end, k)) slots; layer -1: all layers.  All or nothing."""
        _check("hs_reserve", self.lib.hs_reserve(self._h, int(req), int(layer), int(end)))

    def release(self, req: int):
        """End request `req`: its private host pages (and device buffer pages, with a device cache
        pool) return to the free lists and its buffers are emptied; its counters stay."""
        _check("hs_release", self.lib.hs_release(self._h, int(req)))

    def debug_stall_next(self, kernels: int):
        """Test hook: the next launch of each kernel in `kernels` (STALL_ATTN, STALL_RESOLVE) leaves
        one barrier arrival out, so its bounded wait gives up and reports DEVERR_TIMEOUT.
        STALL_FETCH: one record a fetch CTA claimed is never marked as landed; the deciding CTA that
        needs it gives up waiting, reports DEVERR_TIMEOUT and fetches it from the host itself."""
        _check("hs_debug_stall_next", self.lib.hs_debug_stall_next(self._h, int(kernels)))

    def device_usage(self) -> dict:
        used, free, page = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check("hs_device_usage", self.lib.hs_device_usage(self._h, ctypes.byref(used), ctypes.byref(free),
                                                           ctypes.byref(page)))
        return {"pages_in_use": used.value, "pages_free": free.value, "page_slots": page.value}

    def host_usage(self) -> dict:
        used, free, pinned = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check("hs_host_usage", self.lib.hs_host_usage(self._h, ctypes.byref(used), ctypes.byref(free),
                                                       ctypes.byref(pinned)))
        return {"pages_in_use": used.value, "pages_free": free.value, "bytes_pinned": pinned.value}

    def read_history(self, req: int, layer: int, pos0: int, n: int):
        out = np.empty((n, self.cfg.record_elems), dtype=np.uint16)
        _check("hs_read_history", self.lib.hs_read_history(self._h, int(req), int(layer), int(pos0), int(n),
                                                           out.ctypes.data))
        return out
