"""Parity at the full sizes of the benchmark workloads, in the launch configuration bench.py times.

The oracle cannot simulate every (request, layer) of these workloads in seconds, so each test
checks sampled outputs that the oracle computes one by one:
  * for sampled (request, layer) pairs, the oracle replays the whole trace (append, resolve) and
    every step's slots must match bit for bit (plus tags and stamps at sampled steps, and the
    final counters of those pairs);
  * attention of sampled (request, layer, step) against fp64 over the selected positions;
  * properties that hold at any size for all pairs: hits + misses = k per resolve, no error bits.
"""
import math

import numpy as np
import pytest

import oracle
from harness import ATOL_MAX, ATOL_MEAN

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from hierarchical_kv_cache_02_gb300 import LAYOUT_GQA, LAYOUT_MLA, HsConfig, HsPool, inputs


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def run_full(cfg, ctx0, steps, spec, pairs, attn_samples, seed, state_every=8, shared=False, appends=True,
             fused=False):
    """fused: each layer's append and resolve go through the single fused call (hs_append_resolve),
    the form bench.py times; else through the two separate calls."""
    R, L, k, E = cfg.num_requests, cfg.num_layers, cfg.top_k, cfg.record_elems
    trace = inputs.drift_traces(spec, R, L, seed=seed)                          # [S][L][R][k]
    pool = HsPool(cfg)
    hist_cpu = {}
    for l in range(L):
        for r in range(1 if shared else R):
            h = inputs.normal_bf16((ctx0, E), seed=seed * 1000 + 97 * l + 7919 * r, device="cuda")
            pool.prefill(r, l, 0, h)
            for (pr, pl) in pairs:
                if pl == l and (shared or pr == r):
                    hist_cpu[(pr, pl)] = _bits(h)
            del h
    q = inputs.normal_bf16((steps, L, R, cfg.num_q_heads, cfg.head_dim_qk), seed=seed + 1, device="cuda")
    app = inputs.normal_bf16((steps, L, R, E), seed=seed + 2, device="cuda")
    app_cpu = {pair: _bits(app[:, pair[1], pair[0]]) for pair in pairs}
    topk = torch.from_numpy(trace).cuda()
    scale = float(np.float32(1.0 / math.sqrt(cfg.head_dim_qk)))
    kvh = 0 if cfg.layout == LAYOUT_MLA else cfg.num_kv_heads
    caches = {(r, l): oracle.Cache(cfg.buffer_slots, k, "lru", seed=cfg.seed, R=R, L=L, r=r, l=l, C=cfg.capacity)
              for (r, l) in pairs}
    locs = [torch.empty((R, k), dtype=torch.int32, device="cuda") for _ in range(L)]
    out = torch.empty((R, cfg.num_q_heads, cfg.head_dim_v), dtype=torch.float32, device="cuda")
    sampled_layers = sorted({l for _, l in pairs})
    worst = 0.0
    for t in range(steps):
        for l in range(L):
            if appends:
                pos = torch.full((R,), ctx0 + t, dtype=torch.int64, device="cuda")
                if fused:
                    pool.append_resolve(l, pos, app[t, l], topk[t, l], locs[l])
                else:
                    pool.append(l, pos, app[t, l])
                    pool.resolve(l, topk[t, l], locs[l])
            else:
                pool.resolve(l, topk[t, l], locs[l])
            pool.sparse_attn(l, q[t, l], locs[l], out, scale=scale)
            if l in sampled_layers:
                got_locs = locs[l].cpu().numpy()
                for (r, pl) in pairs:
                    if pl != l:
                        continue
                    if appends:
                        caches[(r, l)].append(ctx0 + t)
                    _, rl = caches[(r, l)].resolve(trace[t, l, r])
                    assert np.array_equal(got_locs[r], rl), (t, r, l)
                    if (t, r, l) in attn_samples:
                        hist = hist_cpu[(r, l)]
                        if appends:
                            hist = np.concatenate([hist, app_cpu[(r, l)][:t + 1]])
                        ref = oracle.attention(_bits(q[t, l, r]), hist, trace[t, l, r], scale, kvh, cfg.head_dim_qk,
                                               cfg.head_dim_v)
                        err = np.abs(out[r].cpu().numpy().astype(np.float64) - ref)
                        assert err.max() <= ATOL_MAX and err.mean() <= ATOL_MEAN, (t, r, l, float(err.max()))
                        worst = max(worst, float(err.max()))
                if t % state_every == state_every - 1 or t == steps - 1:
                    tag, stamp, clock = pool.read_state(l)
                    for (r, pl) in pairs:
                        if pl == l:
                            otag, ostamp = caches[(r, l)].slots()
                            assert np.array_equal(tag[r], otag) and np.array_equal(stamp[r], ostamp), (t, r, l)
                            assert clock[r] == caches[(r, l)].counters()["clock"]
    st = pool.stats()
    assert st["error_bits"] == 0
    hm = st["per_rl"][:, :, 0] + st["per_rl"][:, :, 1]
    assert (hm == steps * k).all()  # every resolve: hits + misses = k
    for (r, l), c in caches.items():
        cnt = c.counters()
        assert list(st["per_rl"][r, l, :3]) == [cnt["hits"], cnt["misses"], cnt["appends"]], (r, l)
    pool.close()
    return worst


@pytest.mark.parametrize("fused", [False, True])
def test_full_mla_batch8(fused):
    """Batch 8, 1 layer, context 32768, 576-dim latent, 64 heads, k=2048, B=4096, LRU, 128 steps,
    drift keep 88% / recency mean 2048, write-through append every step (fused = True: fused into
    the resolve, the call bench.py times)."""
    ctx0, steps = 32768, 128
    cfg = HsConfig(num_requests=8, num_layers=1, capacity=ctx0 + steps, layout=LAYOUT_MLA, num_q_heads=64,
                   num_kv_heads=1, head_dim_qk=576, head_dim_v=512, top_k=2048, buffer_slots=4096, seed=3)
    spec = inputs.TraceSpec(ctx0=ctx0, k=2048, steps=steps, keep=0.88, recency_mean=2048, appends=True)
    pairs = [(0, 0), (5, 0)]
    samples = {(0, 0, 0), (127, 0, 0), (64, 5, 0)}
    run_full(cfg, ctx0, steps, spec, pairs, samples, seed=11, fused=fused)


@pytest.mark.parametrize("fetch,fused", [(0, False), (0, True), (1, False), (1, True), (2, True)])
def test_full_gqa_batch16_32_layers(fetch, fused):
    """Batch 16, 32 layers, 8 KV heads x (128 K + 128 V), 32 q heads, context 131072 shared by the
    requests (17 GB pinned), k=2048, B=4096, drift keep 88%, write-through append, 64 steps
    (16 with the misses fetched inside the attention, 32 with fetch CTAs).  fused = True runs
    hs_append_resolve (16 resolve clusters with the early miss copies staged in shared memory), the
    call the headline bench times; fetch = 1 with fused = True is the bench's two-micro-batch pass
    at full batch; fetch = 2 adds the fetch CTAs that copy misses while the decision runs."""
    ctx0 = 131072
    steps = {0: 64, 1: 16, 2: 32}[fetch]
    cfg = HsConfig(num_requests=16, num_layers=32, capacity=ctx0 + steps, layout=LAYOUT_GQA, num_q_heads=32,
                   num_kv_heads=8, head_dim_qk=128, head_dim_v=128, top_k=2048, buffer_slots=4096, seed=5,
                   shared_prefix=ctx0, fetch_in_attention=int(fetch == 1), early_fetch=int(fetch == 2))
    spec = inputs.TraceSpec(ctx0=ctx0, k=2048, steps=steps, keep=0.88, recency_mean=2048, appends=True)
    pairs = [(3, 7), (15, 31)]
    samples = {(steps - 1, 3, 7), (steps // 2, 15, 31), (0, 15, 31)}
    run_full(cfg, ctx0, steps, spec, pairs, samples, seed=13, shared=True, fused=fused)


@pytest.mark.parametrize("early", [0, 1])
def test_full_stress_bursts(early):
    """Batch 16, 4 layers, context 262144, 576-dim latent, 64 heads, k=2048, B=8192, LRU, bursts
    (every 32 steps 40% of the top-k jumps to a far region), 128 steps with write-through append
    fused into the resolve (the call bench.py times); early = 1 with fetch CTAs."""
    ctx0, steps = 262144, 128
    cfg = HsConfig(num_requests=16, num_layers=4, capacity=ctx0 + steps, layout=LAYOUT_MLA, num_q_heads=64,
                   num_kv_heads=1, head_dim_qk=576, head_dim_v=512, top_k=2048, buffer_slots=8192, seed=7,
                   early_fetch=early)
    spec = inputs.TraceSpec(ctx0=ctx0, k=2048, steps=steps, keep=0.88, recency_mean=2048, appends=True,
                            burst_every=32, burst_frac=0.4, far_gap=8 * 2048)
    pairs = [(2, 1), (11, 3)]
    samples = {(32, 2, 1), (96, 11, 3)}
    run_full(cfg, ctx0, steps, spec, pairs, samples, seed=17, state_every=16, fused=True)


def test_full_csa_batch8():
    """Compressed entries (one record per 4 tokens): batch 8, 1 layer, 8192 entries (a 32768-token
    context), 576-dim latent, 64 heads, top-512 entries, B=1024, LRU, 96 steps, no appends (an entry
    is complete only after 4 tokens)."""
    ctx0, steps = 8192, 96
    cfg = HsConfig(num_requests=8, num_layers=1, capacity=ctx0, layout=LAYOUT_MLA, num_q_heads=64,
                   num_kv_heads=1, head_dim_qk=576, head_dim_v=512, top_k=512, buffer_slots=1024, seed=19)
    spec = inputs.TraceSpec(ctx0=ctx0, k=512, steps=steps, keep=0.88, recency_mean=512, appends=False)
    pairs = [(1, 0), (6, 0)]
    samples = {(0, 1, 0), (95, 6, 0), (48, 1, 0)}
    run_full(cfg, ctx0, steps, spec, pairs, samples, seed=23, appends=False)


def test_policy_sweep_miss_curves():
    """One request, context 131072, k=2048, 256 steps, keep 85%: swap-vanilla B=2048, LRU / FIFO /
    random B=4096, LRU B=8192.  Per-step miss curves of the GPU equal the oracle's bit for bit, and
    the oracle's Belady curve lower-bounds every online policy."""
    ctx0, steps, k = 131072, 256, 2048
    spec = inputs.TraceSpec(ctx0=ctx0, k=k, steps=steps, keep=0.85, recency_mean=2048, appends=False)
    trace = inputs.drift_traces(spec, 1, 1, seed=23)
    hist = inputs.normal_bf16((ctx0, 576), seed=29, device="cuda")
    curves = {}
    for name, pol, B in (("swap", 3, 2048), ("lru", 0, 4096), ("fifo", 1, 4096), ("random", 2, 4096),
                         ("lru", 0, 8192)):
        cfg = HsConfig(num_requests=1, num_layers=1, capacity=ctx0, layout=LAYOUT_MLA, num_q_heads=16,
                       num_kv_heads=1, head_dim_qk=576, head_dim_v=512, top_k=k, buffer_slots=B, policy=pol, seed=41,
                       log_steps=steps)
        pool = HsPool(cfg)
        pool.prefill(0, 0, 0, hist)
        topk = torch.from_numpy(trace).cuda()
        locs = torch.empty((1, k), dtype=torch.int32, device="cuda")
        for t in range(steps):
            pool.resolve(0, topk[t, 0], locs)
        gpu_curve = pool.stats()["step_log"][:, 0, 0].astype(np.int64)
        cache = oracle.Cache(B, k, name, seed=41, R=1, L=1, r=0, l=0, C=ctx0)
        ref = np.array([cache.resolve(trace[t, 0, 0])[0] for t in range(steps)])
        assert np.array_equal(gpu_curve, ref), (name, B)
        tag, stamp, _ = pool.read_state(0)
        otag, ostamp = cache.slots()
        assert np.array_equal(tag[0], otag) and np.array_equal(stamp[0], ostamp), (name, B)
        curves[(name, B)] = ref
        pool.close()
    bel = oracle.belady(4096, trace[:, 0, 0], ctx0)
    for key in (("lru", 4096), ("fifo", 4096), ("random", 4096)):
        assert curves[key].sum() >= bel.sum(), key
    assert curves[("lru", 8192)].sum() <= curves[("lru", 4096)].sum()
