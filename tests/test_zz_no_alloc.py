"""The allocation-free attention entry point against the pool-based one and against the oracle.

hs_sparse_attn_noalloc exists for callers that may not call cudaMalloc at all (an engine whose
allocator owns all device memory, a process with a fixed footprint).  It keeps its split
partials in a fixed device array instead of a pool, but runs the same kernels with the same split
plan as hs_sparse_attn over caller-resident KV, so the two must agree bit for bit; both must also
meet the attention tolerance against the fp64 oracle.  Each case makes two calls in a row through
the C ABI, the second with a different shape, so the second call runs on the first one's leftovers
in the shared scratch.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import oracle
from harness import assert_attn_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from hierarchical_kv_cache_02_gb300 import LAYOUT_GQA, LAYOUT_MLA, HsConfig, HsPool, _lib, inputs


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _inputs(cfg, rows, seed):
    R, k = cfg.num_requests, cfg.top_k
    q = inputs.normal_bf16((R, cfg.num_q_heads, cfg.head_dim_qk), seed=seed).cuda()
    kv = inputs.normal_bf16((R, rows, cfg.record_elems), seed=seed + 1).cuda()
    rng = np.random.default_rng(seed)
    locs = np.stack([rng.choice(rows, size=k, replace=False) for _ in range(R)]).astype(np.int32)
    locs[0, ::7] = -1  # padding entries are skipped
    return q, kv, torch.from_numpy(locs).cuda()


def _noalloc(lib, cfg, q, locs, kv, scale, out):
    c = cfg.to_c()
    return lib.hs_sparse_attn_noalloc(ctypes.byref(c), ctypes.c_void_p(q.data_ptr()),
                                      ctypes.c_void_p(locs.data_ptr()), ctypes.c_void_p(kv.data_ptr()),
                                      int(kv.shape[1]), ctypes.c_float(scale), ctypes.c_void_p(out.data_ptr()),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _gqa(R, k):
    return HsConfig(num_requests=R, num_layers=1, capacity=3000, layout=LAYOUT_GQA, num_q_heads=32,
                    num_kv_heads=8, head_dim_qk=128, head_dim_v=128, top_k=k, buffer_slots=max(512, k))


def _mla(R, k, Hq):
    return HsConfig(num_requests=R, num_layers=1, capacity=3000, layout=LAYOUT_MLA, num_q_heads=Hq,
                    num_kv_heads=1, head_dim_qk=576, head_dim_v=512, top_k=k, buffer_slots=max(512, k))


# two calls in a row per case; the second changes the batch and the selection length
CASES = {
    "gqa": (_gqa(4, 500), _gqa(3, 700)),                        # per-KV-head mma.sync kernel
    "mla64": (_mla(2, 300, 64), _mla(3, 640, 64)),              # 64-head tcgen05 kernel + split combine
    "mla16": (_mla(2, 256, 16), _mla(1, 520, 16)),              # CUDA-core shared-latent kernel
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_noalloc_matches_pool_attention_and_oracle_twice(case):
    lib = _lib.load()
    rows = 3000
    for call, (cfg, seed) in enumerate(zip(CASES[case], (101, 202))):
        pool = HsPool(cfg)
        scale = cfg.default_scale
        q, kv, locs = _inputs(cfg, rows, seed)
        ref = pool.sparse_attn(0, q, locs, scale=scale, kv=kv)
        torch.cuda.synchronize()
        out = torch.full_like(ref, 7.0)
        assert _noalloc(lib, cfg, q, locs, kv, scale, out) == _lib.HS_OK, call
        torch.cuda.synchronize()
        # the same kernels with the same split plan: bit-identical to the pool's call
        assert torch.equal(out, ref), (case, call)
        # and within the attention tolerance of fp64 over exactly the selected rows
        qb, kvb, lc = _bits(q), _bits(kv), locs.cpu().numpy()
        kvh = 0 if cfg.layout == LAYOUT_MLA else cfg.num_kv_heads
        got = out.cpu().numpy()
        for r in range(cfg.num_requests):
            exp = oracle.attention(qb[r], kvb[r], lc[r], scale, kvh, cfg.head_dim_qk, cfg.head_dim_v)
            assert_attn_close(got[r], exp, (case, call, r), tight=cfg.layout == LAYOUT_GQA)
        pool.close()


def test_noalloc_ignores_pool_settings():
    """Only the documented fields decide the kernel: a config that also asks for the misses to be
    fetched inside the attention (a pool setting) gives the same result as one that does not."""
    lib = _lib.load()
    cfg = _gqa(2, 300)
    q, kv, locs = _inputs(cfg, 3000, 7)
    a = torch.empty((2, 32, 128), dtype=torch.float32, device="cuda")
    b = torch.empty_like(a)
    assert _noalloc(lib, cfg, q, locs, kv, cfg.default_scale, a) == _lib.HS_OK
    cfg.fetch_in_attention = 1
    assert _noalloc(lib, cfg, q, locs, kv, cfg.default_scale, b) == _lib.HS_OK
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = _lib.load()
    cfg = HsConfig(num_requests=4096, num_layers=1, capacity=3000, layout=LAYOUT_GQA, num_q_heads=32,
                   num_kv_heads=8, head_dim_qk=128, head_dim_v=128, top_k=64, buffer_slots=64)
    q = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    locs = torch.zeros(16, dtype=torch.int32, device="cuda")
    out = torch.zeros(16, dtype=torch.float32, device="cuda")
    # 4096 requests x 32 heads x 130 floats of partials exceed the fixed scratch: rejected before any launch
    c = cfg.to_c()
    rc = lib.hs_sparse_attn_noalloc(ctypes.byref(c), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(locs.data_ptr()),
                                    ctypes.c_void_p(kv.data_ptr()), 3000, ctypes.c_float(0.1),
                                    ctypes.c_void_p(out.data_ptr()), None)
    assert rc == _lib.HS_ERR_SCRATCH
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0  # nothing was enqueued
