"""The allocation-free attention entry point against the pool-based one.

hs_sparse_attn_noalloc exists for callers that may not call cudaMalloc at all (an engine whose
allocator owns all device memory, a process with a fixed footprint).  It keeps its split
partials in a fixed device array instead of a pool.  Here it is called twice in a row through
the C ABI, each time on fresh inputs, and must agree with hs_sparse_attn (resident-KV form)
within the attention tolerance the other tests use.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

from harness import ATOL_MAX, ATOL_MEAN

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from hierarchical_kv_cache_02_gb300 import LAYOUT_GQA, LAYOUT_MLA, HsConfig, HsPool, _lib, inputs


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


@pytest.mark.parametrize("layout", ["gqa", "mla"])
def test_noalloc_matches_pool_attention_twice(layout):
    if layout == "gqa":
        cfg = HsConfig(num_requests=4, num_layers=1, capacity=3000, layout=LAYOUT_GQA, num_q_heads=32,
                       num_kv_heads=8, head_dim_qk=128, head_dim_v=128, top_k=500, buffer_slots=512)
    else:
        cfg = HsConfig(num_requests=2, num_layers=1, capacity=3000, layout=LAYOUT_MLA, num_q_heads=64,
                       num_kv_heads=1, head_dim_qk=576, head_dim_v=512, top_k=300, buffer_slots=512)
    lib = _lib.load()
    pool = HsPool(cfg)
    scale = cfg.default_scale
    for call, seed in enumerate((101, 202)):
        q, kv, locs = _inputs(cfg, 3000, seed)
        ref = pool.sparse_attn(0, q, locs, scale=scale, kv=kv)
        out = torch.full_like(ref, float("nan"))
        assert _noalloc(lib, cfg, q, locs, kv, scale, out) == _lib.HS_OK, call
        torch.cuda.synchronize()
        err = (out.double() - ref.double()).abs()
        assert torch.isfinite(out).all(), call
        assert err.max().item() <= ATOL_MAX and err.mean().item() <= ATOL_MEAN, (call, err.max().item())
    pool.close()


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
