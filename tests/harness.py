"""Shared test harness: one seeded decode scenario run through the CUDA library and the oracle.

A scenario is R requests x L layers with a history of `ctx0` prefilled records per
(request, layer), then `steps` decode steps.  Each step, for every layer: optionally append the
new token (position ctx0 + t), resolve the layer's top-k trace, run sparse attention.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

import oracle
from hierarchical_kv_cache_02_gb300 import HsConfig, inputs

POLICY_NAMES = {0: "lru", 1: "fifo", 2: "random", 3: "swap"}

# attention tolerance: the stated bar (bf16 inputs, fp32 accumulation vs fp64), and for the GQA kernel,
# whose probabilities enter the MMA as bf16 high part + remainder (~16 mantissa bits), a tighter bound
# derived from fp32 rounding of <=576-term dot products and base-2 exponentials.  The shared-latent
# kernel feeds bf16 probabilities (relative error <= 2^-9 per weight, normaliser summed over the same
# rounded weights), which only the stated bar covers.
ATOL_MAX, ATOL_MEAN = 2e-2, 2e-3
ATOL_FP32 = 1e-4


@dataclass
class Scenario:
    cfg: HsConfig
    ctx0: int
    steps: int
    appends: bool
    keep: float = 0.9
    recency_mean: float = 512.0
    burst_every: int = 0
    seed: int = 1
    trace: np.ndarray = field(init=False)      # [steps][L][R][k] int32
    hist: dict = field(init=False)             # (r, l) -> uint16 [C][rec_elems]
    q: np.ndarray = field(init=False)          # [steps][L][R][Hq][Dqk] uint16

    def __post_init__(self):
        c = self.cfg
        R, L = c.num_requests, c.num_layers
        spec = inputs.TraceSpec(ctx0=self.ctx0, k=c.top_k, steps=self.steps, keep=self.keep,
                                recency_mean=self.recency_mean, appends=self.appends,
                                burst_every=self.burst_every, far_gap=int(8 * self.recency_mean))
        self.trace = inputs.drift_traces(spec, R, L, seed=self.seed)
        C, P0, E = c.capacity, c.shared_prefix, c.record_elems
        self.hist = {}
        for l in range(L):
            shared = inputs.normal_bf16((P0, E), seed=self.seed * 7919 + 17 * l).view(dtype=_torch().int16).numpy()
            for r in range(R):
                own = inputs.normal_bf16((C - P0, E), seed=self.seed * 7919 + 1000003 * (r + 1) + 17 * l)
                own = own.view(dtype=_torch().int16).numpy()
                self.hist[(r, l)] = np.ascontiguousarray(np.concatenate([shared, own]).view(np.uint16))
        qs = inputs.normal_bf16((self.steps, L, R, c.num_q_heads, c.head_dim_qk), seed=self.seed * 31 + 5)
        self.q = qs.view(dtype=_torch().int16).numpy().view(np.uint16)

    @property
    def scale(self):
        return float(np.float32(1.0 / math.sqrt(self.cfg.head_dim_qk)))


def _torch():
    import torch

    return torch


def bf16_tensor(bits_u16, device=None):
    torch = _torch()
    t = torch.from_numpy(np.ascontiguousarray(bits_u16).view(np.int16)).view(torch.bfloat16)
    return t.to(device) if device is not None else t


def prefill(pool, sc: Scenario):
    c = sc.cfg
    for l in range(c.num_layers):
        for r in range(c.num_requests):
            lo = c.shared_prefix if r > 0 else 0
            if sc.ctx0 > lo:
                pool.prefill(r, l, lo, bf16_tensor(sc.hist[(r, l)][lo:sc.ctx0]))


def gpu_step(pool, sc: Scenario, t: int, device="cuda:0", attn=True, fused=False):
    """One decode step on the GPU; returns per-layer (locs, out) as CPU arrays.  fused: the append
    and the resolve of a layer go through the single fused call."""
    torch = _torch()
    c = sc.cfg
    R = c.num_requests
    res = []
    for l in range(c.num_layers):
        topk = torch.from_numpy(sc.trace[t, l]).to(device)
        if sc.appends:
            pos = torch.full((R,), sc.ctx0 + t, dtype=torch.int64, device=device)
            rec = bf16_tensor(np.stack([sc.hist[(r, l)][sc.ctx0 + t] for r in range(R)]), device)
            if fused:
                locs = pool.append_resolve(l, pos, rec, topk)
            else:
                pool.append(l, pos, rec)
                locs = pool.resolve(l, topk)
        else:
            locs = pool.resolve(l, topk)
        out = None
        if attn:
            q = bf16_tensor(sc.q[t, l], device)
            out = pool.sparse_attn(l, q, locs, scale=sc.scale).cpu().numpy()
        res.append((locs.cpu().numpy(), out))
    return res


class OracleRun:
    """Oracle caches for every (r, l) of a scenario, stepped in lock-step with the GPU."""

    def __init__(self, sc: Scenario, pairs=None):
        c = sc.cfg
        self.sc = sc
        self.pairs = pairs or [(r, l) for r in range(c.num_requests) for l in range(c.num_layers)]
        self.caches = {(r, l): oracle.Cache(c.buffer_slots, c.top_k, POLICY_NAMES[c.policy], seed=c.seed,
                                            R=c.num_requests, L=c.num_layers, r=r, l=l, C=c.capacity)
                       for (r, l) in self.pairs}

    def step(self, t):
        out = {}
        for (r, l), cache in self.caches.items():
            if self.sc.appends:
                cache.append(self.sc.ctx0 + t)
            m, locs = cache.resolve(self.sc.trace[t, l, r])
            out[(r, l)] = (m, locs)
        return out

    def attention(self, t, r, l):
        c = self.sc.cfg
        kvh = 0 if c.layout == 0 else c.num_kv_heads
        return oracle.attention(self.sc.q[t, l, r], self.sc.hist[(r, l)], self.sc.trace[t, l, r], self.sc.scale,
                                kvh, c.head_dim_qk, c.head_dim_v)


def assert_attn_close(got, ref, what="", tight=True):
    err = np.abs(got.astype(np.float64) - ref)
    assert err.max() <= ATOL_MAX and err.mean() <= ATOL_MEAN, (what, float(err.max()), float(err.mean()))
    if tight:
        assert err.max() <= ATOL_FP32, (what, "above the fp32 bound", float(err.max()))
    return float(err.max())


def assert_layer_matches_oracle(sc: Scenario, orc: OracleRun, ref_step, t, l, locs, out=None, what=""):
    """Slots of every request of layer l at step t equal the oracle's (ref_step = orc.step(t)), and
    the attention output (if given) is within the tolerance of fp64 over the selected positions."""
    c = sc.cfg
    for r in range(c.num_requests):
        assert np.array_equal(locs[r], ref_step[(r, l)][1]), (what, t, r, l)
        if out is not None:
            assert_attn_close(out[r], orc.attention(t, r, l), (what, t, r, l), tight=c.layout == 1)


def assert_pool_matches_oracle(pool, orc: OracleRun, what=""):
    """Tags, stamps and clocks of every layer, and the per-(request, layer) counters, equal the
    oracle's; no error bit is set."""
    c = orc.sc.cfg
    for l in range(c.num_layers):
        tag, stamp, clock = pool.read_state(l)
        for r in range(c.num_requests):
            otag, ostamp = orc.caches[(r, l)].slots()
            assert np.array_equal(tag[r], otag) and np.array_equal(stamp[r], ostamp), (what, r, l)
            assert clock[r] == orc.caches[(r, l)].counters()["clock"], (what, r, l)
    st = pool.stats()
    for (r, l), cache in orc.caches.items():
        cnt = cache.counters()
        assert list(st["per_rl"][r, l, :3]) == [cnt["hits"], cnt["misses"], cnt["appends"]], (what, r, l)
        assert st["per_rl"][r, l, 3] == cnt["misses"] * c.record_bytes, (what, r, l)
    assert st["error_bits"] == 0, what
