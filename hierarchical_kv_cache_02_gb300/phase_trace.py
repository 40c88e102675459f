"""Phase tables of the fused resolve and the shared-latent tensor-core attention.

Builds a variant of the library with -DHS_PHASE_TRACE (in _build/phase/, leaving the normal build
alone), in which thread 0 of each CTA records %globaltimer at the boundaries of the kernels' phases.
For each named workload of bench.py it runs the decode steps to a steady state, records one launch
of the resolve (layer 0) and, for the shared-latent workloads, one launch of the attention, and
prints the median over the CTAs of each stamp, in microseconds from the first CTA's start.

    python -m hierarchical_kv_cache_02_gb300.phase_trace gqa_b16_l32 mla_b8 stress_b16_l4 mla_b8:early gqa_b16_l32@32

Needs a GPU.  The workloads are those of bench.py (GQA with 4 of its 32 layers unless NAME@L names
the layer count: one layer's steady state is the same, but its host history spans an eighth of the
bytes).  NAME:early runs the resolve with its fetch CTAs (early_fetch = 1).  With HS_PHASE_DUMP set
to a folder, the raw stamps of every CTA ([256][64] nanoseconds, 0 = not stamped) are also saved
there as NAME_resolve.npy and NAME_attn.npy.
"""
from __future__ import annotations

import ctypes
import os
import sys

import numpy as np

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))
TRACE_LIB = os.path.join(_build.BUILD, "phase", "libhisparse_phase.so")

RESOLVE = dict(enumerate(["start", "append slot", "hash", "probe", "rank", "early copies issued", "select",
                          "compaction + cluster sync", "writes", "host fetch"]))
RESOLVE.update({10: "  thread 0: hash inserts done", 11: "  thread 0: append search reduced",
                12: "  hash: first barrier passed", 13: "  thread 0: probes done",
                14: "  select pass 0: histogram (or the bitmap)", 15: "  select pass 0: bin (or threshold) found",
                16: "  select pass 1: histogram", 17: "  select pass 1: bin found",
                18: "  compaction: counts scanned", 19: "  thread 0: victims placed",
                20: "  compaction: barrier passed", 21: "fetch CTAs: misses found", 22: "fetch CTAs: done",
                23: "fetch CTAs: victims known"})
ATTN = {0: "start", 1: "setup", 38: "scores of tile 0 issued", 39: "scores of tile 1 issued",
        40: "value product of tile 0 issued", 41: "value product of tile 1 issued",
        43: "softmax: scores of tile 0 seen", 44: "softmax: scores of tile 1 seen",
        46: "softmax: weights of tile 0 written", 47: "softmax: weights of tile 1 written",
        49: "softmax: waiting for the last value product", 50: "partial written",
        51: "value product of tile 0: weights seen", 53: "value rows 0-255 of tile 0 issued",
        55: "value rows 256-511 of tile 0 issued", 56: "softmax: value rows 0-127 of the last tile complete",
        57: "combine: CTA resident", 58: "combine: attention grid complete", 59: "combine: rows written"}
for _u in range(18):
    ATTN[2 + _u] = f"load {_u} issued"
    ATTN[20 + _u] = f"load {_u} landed (score products issued)"


def _table(tr, names):
    used = tr[:, 0] > 0
    if not used.any():
        return []
    t0 = int(tr[used, 0].min())
    rows = []
    for ev in sorted(names):
        col = tr[:, ev].astype(np.int64)  # every CTA that stamped it (a later kernel may have more)
        col = col[col > 0]
        if len(col):
            rel = (col - t0) / 1e3
            rows.append((names[ev], len(col), float(np.median(rel)), float(rel.min()), float(rel.max())))
    rows.sort(key=lambda row: row[2])  # in time order (median)
    return rows, int(used.sum())


def main(argv):
    root = os.path.dirname(_HERE)
    if root not in sys.path:
        sys.path.insert(0, root)
    _build.build_library(force=True, extra_flags=("-DHS_PHASE_TRACE",), lib=TRACE_LIB,
                         build_dir=os.path.join(_build.BUILD, "phase"))
    _build.LIB = TRACE_LIB  # this process loads the traced variant
    import torch

    import bench
    from . import HsPool, _lib

    lib = _lib.load()
    for fn in ("hs_phase_resolve_read", "hs_phase_attn_read"):
        getattr(lib, fn).argtypes = [ctypes.c_void_p]
    for fn in ("hs_phase_resolve_clear", "hs_phase_attn_clear"):
        getattr(lib, fn).argtypes = []
    for name in argv or ["gqa_b16_l32", "mla_b8", "stress_b16_l4"]:
        # NAME:early runs the resolve with fetch CTAs (early_fetch = 1); NAME@L sets the layer count
        # (GQA: 4 of its 32 layers by default; its host history then spans an eighth of the bytes)
        name, _, nl = name.partition("@")
        name, _, mode = name.partition(":")
        w = dict(bench.WORKLOADS[name])
        if nl:
            w["L"] = int(nl)
        elif name == "gqa_b16_l32":
            w["L"] = 4
        W = 24
        wl = bench.Workload(w, W + 1, "cuda", seed=bench.replica_seed(0), fetch=mode or "resolve")
        pool = HsPool(wl.cfg)
        wl.prefill(pool)
        R, L, k = w["R"], w["L"], w["k"]
        locs = [torch.empty((R, k), dtype=torch.int32, device="cuda") for _ in range(L)]
        outs = [torch.empty((R, w["Hq"], w["Dv"]), dtype=torch.float32, device="cuda") for _ in range(L)]
        appends = w.get("appends", True)
        res_tr = np.zeros((256, 64), dtype=np.uint64)
        att_tr = np.zeros((256, 64), dtype=np.uint64)
        for t in range(W + 1):
            for l in range(L):
                traced = t == W and l == 0
                if traced:
                    torch.cuda.synchronize()
                    lib.hs_phase_resolve_clear()
                    lib.hs_phase_attn_clear()
                    torch.cuda.synchronize()

                def layer():
                    if appends:
                        pool.append_resolve(l, wl.pos[t], wl.app[t, l], wl.topk[t, l], locs[l])
                    else:
                        pool.resolve(l, wl.topk[t, l], locs[l])
                    pool.sparse_attn(l, wl.q[t, l], locs[l], outs[l], scale=wl.cfg.default_scale)

                # every layer runs as a captured graph replayed once, as in the bench, so the traced
                # layer's timeline shows the kernels' launch overlap without host launch costs
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph):
                    layer()
                graph.replay()
                if traced:
                    torch.cuda.synchronize()
                    lib.hs_phase_resolve_read(res_tr.ctypes.data)
                    lib.hs_phase_attn_read(att_tr.ctypes.data)
        st = pool.stats()
        pool.close()
        print(f"{name}{':' + mode if mode else ''}: misses per (request, layer, step) "
              f"{st['misses'] / (R * L * (W + 1)):.0f} of k = {k}")
        dump = os.environ.get("HS_PHASE_DUMP")  # a folder: the raw stamps of each workload, as .npy
        if dump:
            os.makedirs(dump, exist_ok=True)
            np.save(os.path.join(dump, f"{name}{'_' + mode if mode else ''}_resolve.npy"), res_tr)
            np.save(os.path.join(dump, f"{name}{'_' + mode if mode else ''}_attn.npy"), att_tr)
        rows, n = _table(res_tr, RESOLVE)
        print(f"  k_resolve, {n} CTAs (median / min / max over the CTAs, us from the first CTA's start)")
        for nm, cnt, med, lo, hi in rows:
            print(f"    {nm:44s} {med:7.2f} {lo:7.2f} {hi:7.2f}")
        tab = _table(att_tr, ATTN)
        # one timeline over both tables (the same %globaltimer), from the resolve's first CTA start
        r0 = int(res_tr[res_tr[:, 0] > 0, 0].min())

        def _span(tr, ev, fn):
            col = tr[:, ev].astype(np.int64)
            col = col[col > 0]
            return (fn(col) - r0) / 1e3 if len(col) else float("nan")

        line = (f"  timeline (us from the resolve's first CTA start): resolve done {_span(res_tr, 9, np.max):.2f}")
        if tab:
            line += (f", attention first CTA {_span(att_tr, 0, np.min):.2f}, last partial "
                     f"{_span(att_tr, 50, np.max):.2f}")
            if (att_tr[:, 59] > 0).any():
                line += f", combine done {_span(att_tr, 59, np.max):.2f}"
        print(line)
        if tab:
            rows, n = tab
            print(f"  k_attn_mla_pipe, {n} CTAs")
            for nm, cnt, med, lo, hi in rows:
                print(f"    {nm:44s} {med:7.2f} {lo:7.2f} {hi:7.2f}   ({cnt} CTAs)")


if __name__ == "__main__":
    main(sys.argv[1:])
