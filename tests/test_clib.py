"""The C ABI library loads without a GPU, exports every entry point include/hisparse.h
declares, and rejects bad configurations on the host before touching the device."""
import ctypes
import os
import re

import pytest

from hierarchical_kv_cache_02_gb300 import _lib, build
from hierarchical_kv_cache_02_gb300.pool import HsConfig

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return _lib.load()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(hs_\w+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(lib):
    declared = _declared()
    assert declared, "no declarations found"
    for name in declared:
        assert hasattr(lib, name), name
    assert declared == set(_lib.EXPORTS)


def test_record_bytes(lib):
    gqa = HsConfig(num_requests=1, num_layers=1, capacity=10)
    mla = HsConfig(num_requests=1, num_layers=1, capacity=10, layout=0, num_q_heads=64, num_kv_heads=1,
                   head_dim_qk=576, head_dim_v=512)
    assert lib.hs_record_bytes(ctypes.byref(gqa.to_c())) == 4096
    assert lib.hs_record_bytes(ctypes.byref(mla.to_c())) == 1152


@pytest.mark.parametrize("change", [
    dict(top_k=5000, buffer_slots=4096),          # k > B
    dict(top_k=4097, buffer_slots=8192),          # k above the resolve's limit of 4096
    dict(buffer_slots=20000, top_k=10),           # B too large
    dict(io_chunk_bytes=48),                      # not a power of two
    dict(io_chunk_bytes=256),                     # above the limit
    dict(num_q_heads=30),                         # Hq not a multiple of the KV heads
    dict(head_dim_qk=96),                         # unsupported head size
    dict(policy=7),
    dict(shared_prefix=11),                       # beyond capacity
    dict(num_requests=0),
    dict(early_fetch=2),                          # not 0 or 1
    dict(early_fetch=1, fetch_in_attention=1),    # the fetch CTAs and the attention's fetch exclude each other
])
def test_bad_config_rejected_on_host(lib, change):
    base = dict(num_requests=2, num_layers=1, capacity=10, top_k=8, buffer_slots=16)
    base.update(change)
    cfg = HsConfig(**base).to_c()
    h = ctypes.c_void_p()
    assert lib.hs_pool_create(ctypes.byref(cfg), 0, ctypes.byref(h)) == _lib.HS_ERR_CONFIG
    assert not h.value


def test_null_arguments(lib):
    assert lib.hs_pool_create(None, 0, None) == _lib.HS_ERR_ARG
    assert lib.hs_resolve(None, 0, None, None, None) == _lib.HS_ERR_ARG
    assert lib.hs_sparse_attn(None, 0, None, None, None, 0, ctypes.c_float(1.0), None, None) == _lib.HS_ERR_ARG
    assert lib.hs_pool_destroy(None) == _lib.HS_OK


@pytest.mark.parametrize("which", ["q", "out", "locs"])
def test_misaligned_attention_arguments_rejected_on_host(lib, which):
    """The attention kernels move queries and outputs in 16-byte vectors and slot lists in 4-byte
    words: a misaligned pointer is refused before anything touches the device (the addresses here
    are never dereferenced)."""
    cfg = HsConfig(num_requests=1, num_layers=1, capacity=64, top_k=8, buffer_slots=16).to_c()
    ptrs = {"q": 0x10000, "locs": 0x20000, "kv": 0x30000, "out": 0x40000}
    ptrs[which] += 8 if which != "locs" else 2
    rc = lib.hs_sparse_attn_noalloc(ctypes.byref(cfg), ctypes.c_void_p(ptrs["q"]), ctypes.c_void_p(ptrs["locs"]),
                                    ctypes.c_void_p(ptrs["kv"]), ctypes.c_int64(16), ctypes.c_float(1.0),
                                    ctypes.c_void_p(ptrs["out"]), None)
    assert rc == _lib.HS_ERR_ARG
