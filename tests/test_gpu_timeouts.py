"""Bounded waits inside the kernels, exercised without any GPU fault.

Every mbarrier wait in the kernels gives up after about a second, records DEVERR_TIMEOUT and lets
the kernel return.  A test hook (hs_debug_stall_next) makes the next launch of a kernel leave one
barrier arrival out, so that the wait for it runs out: the test checks that the call took the
wait's limit, that hs_stats reports the timeout, and that the context and the pool stay usable --
after a cold start the same pool runs the scenario again in agreement with the oracle.
"""
import time

import pytest

from harness import OracleRun, Scenario, assert_layer_matches_oracle, assert_pool_matches_oracle, gpu_step, prefill

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from hierarchical_kv_cache_02_gb300 import DEVERR_TIMEOUT, LAYOUT_GQA, LAYOUT_MLA, HsConfig, HsPool
from hierarchical_kv_cache_02_gb300._lib import STALL_ATTN, STALL_FETCH, STALL_RESOLVE


def _scenario():
    cfg = HsConfig(num_requests=2, num_layers=1, capacity=3000 + 4, layout=LAYOUT_MLA, num_q_heads=64, num_kv_heads=1,
                   head_dim_qk=576, head_dim_v=512, top_k=512, buffer_slots=1024, seed=11)
    return Scenario(cfg, ctx0=3000, steps=3, appends=True, keep=0.85, recency_mean=300, seed=41)


@pytest.mark.parametrize("kernel", ["attention", "resolve"])
def test_wait_gives_up_reports_and_leaves_the_pool_usable(kernel):
    sc = _scenario()
    pool = HsPool(sc.cfg)
    prefill(pool, sc)
    gpu_step(pool, sc, 0, fused=True)
    torch.cuda.synchronize()
    assert pool.stats(reset=True)["error_bits"] == 0
    # the next launch of the kernel leaves one arrival out: its wait runs to the limit and gives up
    pool.debug_stall_next(STALL_ATTN if kernel == "attention" else STALL_RESOLVE)
    t0 = time.perf_counter()
    gpu_step(pool, sc, 1, fused=True)  # outputs of this step are undefined
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    st = pool.stats(reset=True)
    assert st["error_bits"] & DEVERR_TIMEOUT, st["error_bits"]
    assert elapsed >= 0.9, elapsed  # the wait ran for its limit (about one second)
    # the hook was consumed: a cold start replays the scenario in agreement with the oracle
    pool.reset()
    orc = OracleRun(sc)
    for t in range(sc.steps):
        res = gpu_step(pool, sc, t, fused=True)
        ref = orc.step(t)
        locs, out = res[0]
        assert_layer_matches_oracle(sc, orc, ref, t, 0, locs, out, what=(kernel, t))
    assert_pool_matches_oracle(pool, orc, what=kernel)
    assert pool.stats()["error_bits"] == 0
    pool.close()


@pytest.mark.parametrize("layout", [LAYOUT_GQA, LAYOUT_MLA])
def test_fetch_wait_gives_up_and_leaves_the_pool_usable(layout):
    """Early fetch: the deciding CTAs of one request never signal the fetch CTAs, whose wait runs to
    its limit and gives up; the call reports DEVERR_TIMEOUT, and after a cold start the same pool
    replays the scenario in agreement with the oracle."""
    if layout == LAYOUT_GQA:
        cfg = HsConfig(num_requests=3, num_layers=2, capacity=4000 + 4, layout=LAYOUT_GQA, num_q_heads=32,
                       num_kv_heads=8, head_dim_qk=128, head_dim_v=128, top_k=512, buffer_slots=1024, seed=5,
                       early_fetch=1)
    else:
        cfg = HsConfig(num_requests=2, num_layers=1, capacity=3000 + 4, layout=LAYOUT_MLA, num_q_heads=64,
                       num_kv_heads=1, head_dim_qk=576, head_dim_v=512, top_k=512, buffer_slots=1024, seed=11,
                       early_fetch=1)
    sc = Scenario(cfg, ctx0=cfg.capacity - 4, steps=3, appends=True, keep=0.85, recency_mean=300, seed=43)
    pool = HsPool(cfg)
    prefill(pool, sc)
    gpu_step(pool, sc, 0, fused=True)
    torch.cuda.synchronize()
    assert pool.stats(reset=True)["error_bits"] == 0
    pool.debug_stall_next(STALL_FETCH)
    t0 = time.perf_counter()
    gpu_step(pool, sc, 1, fused=True)  # outputs of this step are undefined
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    st = pool.stats(reset=True)
    assert st["error_bits"] & DEVERR_TIMEOUT, st["error_bits"]
    assert elapsed >= 0.9, elapsed  # the wait ran for its limit (about one second)
    pool.reset()
    orc = OracleRun(sc)
    for t in range(sc.steps):
        res = gpu_step(pool, sc, t, fused=True)
        ref = orc.step(t)
        for l in range(cfg.num_layers):
            locs, out = res[l]
            assert_layer_matches_oracle(sc, orc, ref, t, l, locs, out, what=("fetch stall", t))
    assert_pool_matches_oracle(pool, orc, what="fetch stall")
    assert pool.stats()["error_bits"] == 0
    pool.close()
