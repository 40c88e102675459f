"""The device cache pool (HiSparse summary §8: the coordinator allocates and grows each request's
per-layer device cache on demand; the host pool's size is tied to it by host_to_device_ratio).

A buffer grown ahead of the positions its request uses must give results identical to the full
buffer, bit for bit.  A buffer held below that evicts among its own slots exactly as the oracle's
capped buffer does.  Fewer than k slots refuse the step."""
import numpy as np
import pytest

from harness import OracleRun, Scenario, assert_attn_close, bf16_tensor, gpu_step, prefill

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from hierarchical_kv_cache_02_gb300 import (DEVERR_APPEND, DEVERR_SLOTS, LAYOUT_GQA, LAYOUT_MLA, HsConfig, HsError,
                                            HsPool)
from hierarchical_kv_cache_02_gb300 import _lib

SHAPES = {  # layout, Hq, Hkv, Dqk, Dv: the three attention kernels
    "gqa": (LAYOUT_GQA, 32, 8, 128, 128),
    "mla64": (LAYOUT_MLA, 64, 1, 576, 512),
    "mla8": (LAYOUT_MLA, 8, 1, 576, 512),
}


def _cfg(shape="gqa", fetch=0, pool_slots=0, B=512, k=64, C=340, R=3, L=2, policy=0, P0=0, host_on_demand=0,
         host_page=0, ratio=0.0):
    lay, Hq, Hkv, Dqk, Dv = SHAPES[shape]
    return HsConfig(num_requests=R, num_layers=L, capacity=C, layout=lay, num_q_heads=Hq, num_kv_heads=Hkv,
                    head_dim_qk=Dqk, head_dim_v=Dv, top_k=k, buffer_slots=B, policy=policy, seed=11,
                    shared_prefix=P0, fetch_in_attention=int(fetch == 1), early_fetch=int(fetch == 2),
                    device_pool_slots=pool_slots, buffer_page_slots=16,
                    host_on_demand=host_on_demand, host_page_tokens=host_page, host_to_device_ratio=ratio)


@pytest.mark.parametrize("shape,fetch,P0", [("gqa", 0, 0), ("gqa", 1, 256), ("gqa", 2, 0), ("mla64", 0, 0),
                                            ("mla64", 2, 256), ("mla8", 0, 256)])
def test_buffers_grown_ahead_of_the_context_match_full_buffers(shape, fetch, P0):
    """Each step the coordinator grows every buffer to cover the token it appends: caps 304 -> 336
    of B = 512, so the buffers never hold all B slots, yet everything equals the full pool's."""
    ctx0, T = 300, 24
    full_cfg = _cfg(shape, fetch, P0=P0)
    grown_cfg = _cfg(shape, fetch, pool_slots=3 * 2 * 512, P0=P0)
    sc = Scenario(full_cfg, ctx0=ctx0, steps=T, appends=True, recency_mean=64.0, seed=41)
    full, grown = HsPool(full_cfg), HsPool(grown_cfg)
    prefill(full, sc)
    prefill(grown, sc)
    R, L = full_cfg.num_requests, full_cfg.num_layers
    assert grown.device_usage()["pages_in_use"] == 0  # prefill writes the host pool only
    for t in range(T):
        for r in range(R):
            grown.reserve(r, ctx0 + t + 1)
        a, b = gpu_step(full, sc, t, fused=True), gpu_step(grown, sc, t, fused=True)
        for l in range(L):
            assert np.array_equal(a[l][0], b[l][0]), (t, l)
            assert np.array_equal(a[l][1], b[l][1]), (t, l)
    cap = -(-(ctx0 + T) // 16) * 16
    assert grown.device_usage() == {"pages_in_use": R * L * cap // 16, "pages_free": (R * L * 512 - R * L * cap) // 16,
                                    "page_slots": 16}
    for l in range(L):
        x, y = full.read_state(l), grown.read_state(l)
        assert all(np.array_equal(u, v) for u, v in zip(x, y))
        assert (x[0][:, cap:] == -1).all()  # the full buffers never used a slot the grown ones lack
        for r in range(R):
            assert np.array_equal(full.read_buffer(r, l)[:cap], grown.read_buffer(r, l)[:cap])
            assert (grown.read_buffer(r, l)[cap:] == 0).all()
    assert np.array_equal(full.stats()["per_rl"], grown.stats()["per_rl"])
    full.close()
    grown.close()


@pytest.mark.parametrize("fetch", [0, 2])
@pytest.mark.parametrize("policy", [0, 2, 3])
def test_buffer_held_below_its_context_evicts_like_the_capped_oracle(policy, fetch):
    """Buffers reserved to 100 positions hold 112 slots while the traces range over 300+: the
    kernels evict among those slots exactly as the oracle's capped buffer does (fetch = 2: with the
    resolve's fetch CTAs, whose residency hint must ignore slots past the buffer's count)."""
    cfg = _cfg("gqa", fetch=fetch, pool_slots=3 * 2 * 512, policy=policy)
    sc = Scenario(cfg, ctx0=300, steps=16, appends=True, recency_mean=96.0, seed=43)
    pool = HsPool(cfg)
    prefill(pool, sc)
    for r in range(cfg.num_requests):
        pool.reserve(r, 100)
    orc = OracleRun(sc)
    for cache in orc.caches.values():
        cache.set_cap(112)
    for t in range(sc.steps):
        got = gpu_step(pool, sc, t, fused=True)
        ref = orc.step(t)
        for (r, l), (m, locs) in ref.items():
            assert np.array_equal(got[l][0][r], locs), (t, r, l)
            assert_attn_close(got[l][1][r], orc.attention(t, r, l), (t, r, l))
    for l in range(cfg.num_layers):
        tag, stamp, clock = pool.read_state(l)
        for r in range(cfg.num_requests):
            otag, ostamp = orc.caches[(r, l)].slots()
            assert np.array_equal(tag[r], otag) and np.array_equal(stamp[r], ostamp)
            assert clock[r] == orc.caches[(r, l)].counters()["clock"]
    assert pool.stats()["error_bits"] == 0
    pool.close()


@pytest.mark.parametrize("fetch", [0, 2])
def test_fewer_than_k_slots_refuse_the_step(fetch):
    """Request 1 never gets device pages: its resolves change nothing and flag HS_DEVERR_SLOTS; the
    other requests' results are those of a full pool."""
    full_cfg, cfg = _cfg("gqa"), _cfg("gqa", fetch=fetch, pool_slots=3 * 2 * 512)
    sc = Scenario(full_cfg, ctx0=300, steps=3, appends=True, seed=45)
    full, pool = HsPool(full_cfg), HsPool(cfg)
    prefill(full, sc)
    prefill(pool, sc)
    pool.reserve(0, 340)
    pool.reserve(2, 340)
    for t in range(sc.steps):
        a, b = gpu_step(full, sc, t, fused=True), gpu_step(pool, sc, t, fused=True)
        for l in range(cfg.num_layers):
            for r in (0, 2):
                assert np.array_equal(a[l][0][r], b[l][0][r]) and np.array_equal(a[l][1][r], b[l][1][r])
            assert (b[l][0][1] == -1).all()
            assert (b[l][1][1] == 0).all()  # no valid entry: zeros
    st = pool.stats()
    assert (st["errors"][1] == DEVERR_SLOTS).all() and (st["errors"][[0, 2]] == 0).all()
    assert (st["per_rl"][1] == 0).all()
    for l in range(cfg.num_layers):
        tag, stamp, clock = pool.read_state(l)
        assert (tag[1] == -1).all() and (stamp[1] == 0).all() and clock[1] == 1
    # the stand-alone append refuses too; a position outside the pool adds HS_DEVERR_APPEND
    pos = torch.tensor([300, 300, 300], dtype=torch.int64, device="cuda")
    rec = bf16_tensor(np.zeros((3, cfg.record_elems), dtype=np.uint16), "cuda")
    pool.stats(reset=True)
    pool.append(0, pos, rec)
    assert pool.stats()["errors"][1, 0] == DEVERR_SLOTS
    pos[1] = 10_000
    topk = torch.from_numpy(sc.trace[0, 0]).cuda()
    pool.append_resolve(0, pos, rec, topk)
    assert pool.stats()["errors"][1, 0] == DEVERR_SLOTS | DEVERR_APPEND
    full.close()
    pool.close()


@pytest.mark.parametrize("policy", [0, 2])
def test_release_starts_the_request_cold(policy):
    """After hs_release a request index serves a new request from an empty buffer: its results
    equal a fresh pool's; its device pages went back to the free list and came out again."""
    cfg = _cfg("gqa", pool_slots=3 * 2 * 512, policy=policy, host_on_demand=1, host_page=64)
    sc = Scenario(cfg, ctx0=300, steps=6, appends=True, seed=47)
    pool, fresh = HsPool(cfg), HsPool(cfg)
    for p in (pool, fresh):
        prefill(p, sc)
        for r in range(cfg.num_requests):
            p.reserve(r, 340)
    for t in range(sc.steps):
        gpu_step(pool, sc, t, fused=True)
    used = pool.device_usage()["pages_in_use"]
    pool.release(1)
    assert pool.device_usage()["pages_in_use"] == used - cfg.num_layers * -(-340 // 16)
    for l in range(cfg.num_layers):
        tag, stamp, clock = pool.read_state(l)
        assert (tag[1] == -1).all() and (stamp[1] == 0).all() and clock[1] == 1
        assert (pool.read_history(1, l, 0, 10) == 0).all()
    for l in range(cfg.num_layers):  # the new request's prompt, then its reservation
        pool.prefill(1, l, 0, bf16_tensor(sc.hist[(1, l)][:300]))
    pool.reserve(1, 340)
    assert pool.device_usage()["pages_in_use"] == used
    for t in range(sc.steps):
        a, b = gpu_step(fresh, sc, t, fused=True), gpu_step(pool, sc, t, fused=True)
        for l in range(cfg.num_layers):
            assert np.array_equal(a[l][0][1], b[l][0][1]), (t, l)
            assert np.array_equal(a[l][1][1], b[l][1][1]), (t, l)
    pool.close()
    fresh.close()


def test_device_pool_exhaustion_reserves_nothing():
    cfg = _cfg("gqa", pool_slots=2 * 512 + 100, R=3, L=2, C=512)  # 71 pages of 16 slots
    pool = HsPool(cfg)
    pool.reserve(0, 400)  # 2 layers x 25 pages
    before = (pool.device_usage(), pool.host_usage())
    with pytest.raises(HsError) as e:
        pool.reserve(1, 400)  # needs 50 more, 21 are left
    assert e.value.status == _lib.HS_ERR_ALLOC_DEV
    assert (pool.device_usage(), pool.host_usage()) == before
    pool.reserve(1, 100, layer=0)  # 7 pages fit
    assert pool.device_usage()["pages_in_use"] == 57
    pool.close()


def test_host_to_device_ratio_bounds_the_host_pool():
    """Device pool 3 x 2 x 512 slots of 4 KB = 12 MiB; ratio 1.5 lets the host pool pin 18 MiB, i.e.
    72 host pages of 64 records (256 KB)."""
    cfg = _cfg("gqa", pool_slots=3 * 2 * 512, host_on_demand=1, host_page=64, ratio=1.5, C=4096)
    pool = HsPool(cfg)
    limit = int(1.5 * 3 * 2 * 512 * 4096)
    pool.reserve(0, 2048)  # 2 layers x 32 pages
    u = pool.host_usage()
    assert u["pages_in_use"] == 64 and u["bytes_pinned"] == limit  # the slab stops at the bound
    before = (pool.device_usage(), pool.host_usage())
    with pytest.raises(HsError) as e:
        pool.reserve(1, 2048)  # 64 more pages, 8 are left
    assert e.value.status == _lib.HS_ERR_ALLOC_HOST
    assert (pool.device_usage(), pool.host_usage()) == before
    pool.reserve(1, 256)  # 2 x 4 pages: the rest of the bound
    assert pool.host_usage() == {"pages_in_use": 72, "pages_free": 0, "bytes_pinned": limit}
    pool.close()
    # a full host reservation (3 x 2 x 64 pages = 96 MiB) over the bound fails at creation
    with pytest.raises(HsError) as e:
        HsPool(_cfg("gqa", pool_slots=3 * 2 * 512, host_page=64, ratio=1.5, C=4096))
    assert e.value.status == _lib.HS_ERR_ALLOC_HOST
