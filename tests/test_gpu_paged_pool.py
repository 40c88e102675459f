"""The memory layer's paged host pool (HiSparse summary §8: host pool allocated in pages, grown on
demand).  Paging changes where the history lives, never what the kernels compute: every result
must equal the fully reserved pool's, bit for bit."""
import numpy as np
import pytest

from harness import Scenario, bf16_tensor, gpu_step, prefill

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from hierarchical_kv_cache_02_gb300 import DEVERR_APPEND, DEVERR_PAGE, LAYOUT_GQA, HsConfig, HsPool


def _cfg(on_demand, page=0, fetch=0, P0=0, C=3000 + 8):
    return HsConfig(num_requests=3, num_layers=2, capacity=C, layout=LAYOUT_GQA, num_q_heads=32, num_kv_heads=8,
                    head_dim_qk=128, head_dim_v=128, top_k=200, buffer_slots=400, seed=5, shared_prefix=P0,
                    fetch_in_attention=int(fetch == 1), early_fetch=int(fetch == 2), host_page_tokens=page,
                    host_on_demand=on_demand)


@pytest.mark.parametrize("fetch", [0, 1, 2])
@pytest.mark.parametrize("P0", [0, 2048])
def test_on_demand_pages_match_full_reservation(fetch, P0):
    """Small pages reserved on demand (prefill, then hs_reserve ahead of the appends) against the
    pool that reserves every page at creation: slots, outputs, state, counters and the history."""
    full_cfg, lazy_cfg = _cfg(0, fetch=fetch, P0=P0), _cfg(1, page=64, fetch=fetch, P0=P0)
    sc = Scenario(full_cfg, ctx0=3000, steps=8, appends=True, seed=31)
    full, lazy = HsPool(full_cfg), HsPool(lazy_cfg)
    prefill(full, sc)
    prefill(lazy, sc)
    R, L = full_cfg.num_requests, full_cfg.num_layers
    # the full reservation pins exactly its pages (1024 tokens of 4096 bytes each), all in use
    full_pages = L * (P0 // 1024) + R * L * (-(-(3000 + 8) // 1024) - P0 // 1024)
    assert full.host_usage() == {"pages_in_use": full_pages, "pages_free": 0, "bytes_pinned": full_pages * 1024 * 4096}
    used_after_prefill = lazy.host_usage()["pages_in_use"]
    shared_pages = P0 // 64
    private_pages = -(-(3000 - P0) // 64) if P0 == 0 else -(-3000 // 64) - shared_pages
    assert used_after_prefill == L * shared_pages + R * L * private_pages
    for r in range(R):
        lazy.reserve(r, 3000 + sc.steps)
    assert lazy.host_usage()["pages_in_use"] == L * shared_pages + R * L * (-(-(3000 + sc.steps) // 64) - shared_pages)
    for t in range(sc.steps):
        a, b = gpu_step(full, sc, t, fused=True), gpu_step(lazy, sc, t, fused=True)
        for l in range(L):
            assert np.array_equal(a[l][0], b[l][0]), (t, l)
            assert np.array_equal(a[l][1], b[l][1]), (t, l)
    for l in range(L):
        x, y = full.read_state(l), lazy.read_state(l)
        assert all(np.array_equal(u, v) for u, v in zip(x, y))
        for r in range(R):
            assert np.array_equal(full.read_history(r, l, 0, 3000 + sc.steps), lazy.read_history(r, l, 0, 3000 + sc.steps))
    assert np.array_equal(full.stats()["per_rl"], lazy.stats()["per_rl"])
    full.close()
    lazy.close()


def test_append_on_unreserved_page_is_flagged_and_skipped():
    cfg = _cfg(1, page=64, C=3200)
    sc = Scenario(cfg, ctx0=3000, steps=2, appends=True, seed=33)
    pool = HsPool(cfg)
    prefill(pool, sc)  # reserves pages 0-46, i.e. positions [0, 3008)
    pool.reserve(0, 3001)  # nothing new
    R = cfg.num_requests
    pos = torch.full((R,), 3100, dtype=torch.int64, device="cuda")  # on page 48: reserved for nobody
    rec = bf16_tensor(np.stack([sc.hist[(r, 0)][3000] for r in range(R)]), "cuda")
    tag_before = pool.read_state(0)[0].copy()
    pool.append(0, pos, rec)
    st = pool.stats()
    assert st["error_bits"] & DEVERR_APPEND
    assert np.array_equal(pool.read_state(0)[0], tag_before)  # nothing was installed
    assert st["appends"] == 0
    pool.close()


@pytest.mark.parametrize("fetch", [0, 2])
def test_miss_on_unreserved_page_is_flagged(fetch):
    cfg = _cfg(1, page=64, fetch=fetch)
    pool = HsPool(cfg)
    R, k = cfg.num_requests, cfg.top_k
    recs = bf16_tensor(np.zeros((1000, cfg.record_elems), dtype=np.uint16), "cuda")
    for r in range(R):
        for l in range(cfg.num_layers):
            pool.prefill(r, l, 0, recs)  # positions [0, 1000) only
    topk = torch.arange(2000, 2000 + k, dtype=torch.int32, device="cuda").repeat(R, 1)  # pages never reserved
    pool.resolve(0, topk)
    assert pool.stats()["error_bits"] & DEVERR_PAGE
    pool.close()


def test_release_returns_pages_for_reuse():
    cfg = _cfg(1, page=64)
    pool = HsPool(cfg)
    pool.reserve(0, 3008)
    u = pool.host_usage()
    per_request = cfg.num_layers * -(-3008 // 64)
    assert u["pages_in_use"] == per_request
    pinned = u["bytes_pinned"]
    pool.release(0)
    u = pool.host_usage()
    assert u["pages_in_use"] == 0 and u["pages_free"] >= per_request
    assert np.all(pool.read_history(0, 0, 0, 10) == 0)  # released history reads as zeros
    pool.reserve(1, 3008)  # served from the free list: no new pinned memory
    u = pool.host_usage()
    assert u["pages_in_use"] == per_request and u["bytes_pinned"] == pinned
    pool.close()
