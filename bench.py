"""Benchmark of the HiSparse decode hot path on one GB300 (or N independent replicas).

One step = one decode step over every layer of the workload: per layer, write-through append
of the new token, fused resolve of the layer's top-k, sparse attention over the resolved slots.
Default workload (GQA, 32 layers): batch 16, 8 KV heads x (128 K + 128 V) bf16 per token,
32 query heads, context 131072, k = 2048, B = 4096 slots per (request, layer), LRU, drift
traces keeping 88% per step (recency mean 2048).  The 16 requests share one prefilled
131072-token history per layer (17 GB of pinned host memory); appended tokens are private.

Printed: one JSON line (rank 0).  `value` = decode layer-steps/s (one layer for the whole
batch) with every input resident in HBM; `e2e` = the same with per-step inputs copied from
pinned host memory and outputs copied back inside the timed region.  `roofline` rates the
attention against HBM from its launches timed back to back; `host_link` rates the resolve's miss
copies against a pinned copy measured in the same run.  The GQA workload also reports two other
schedules of the same steps: two micro-batches with the misses copied inside the attention, and
(a different selection pattern) layer groups sharing one top-k.
`--impl reference` times the CPU oracle (test infrastructure, single-threaded) on a bounded
sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "resolve+sparse-attn µs/layer and decode layer-steps/s; HBM & host-link GB/s"

WORKLOADS = {
    # batch 16, 32 layers, GQA 8 x (128 | 128), 32 q heads, ctx 131072, k 2048, B 4096, keep 88%
    "gqa_b16_l32": dict(R=16, L=32, ctx0=131072, layout=1, Hq=32, Hkv=8, Dqk=128, Dv=128, k=2048, B=4096,
                        keep=0.88, mu=2048.0, burst=0, shared=True, steps=64),
    # batch 8, 1 layer, MLA 576-dim latent, 64 heads, ctx 32768, k 2048, B 4096, keep 88%
    "mla_b8": dict(R=8, L=1, ctx0=32768, layout=0, Hq=64, Hkv=1, Dqk=576, Dv=512, k=2048, B=4096,
                   keep=0.88, mu=2048.0, burst=0, shared=False, steps=128),
    # stress: batch 16, 4 layers, MLA, ctx 262144, k 2048, B 8192, bursts every 32 steps
    "stress_b16_l4": dict(R=16, L=4, ctx0=262144, layout=0, Hq=64, Hkv=1, Dqk=576, Dv=512, k=2048, B=8192,
                          keep=0.88, mu=2048.0, burst=32, shared=False, steps=128),
    # compressed entries (one record per 4 tokens): batch 8, 1 layer, 32768-token context = 8192
    # entries, top-512 entries (2048 tokens), B 1024, MLA latent, 64 heads; an entry is complete only
    # after 4 tokens, so the decode steps append nothing
    "csa_b8": dict(R=8, L=1, ctx0=8192, layout=0, Hq=64, Hkv=1, Dqk=576, Dv=512, k=512, B=1024,
                   keep=0.88, mu=512.0, burst=0, shared=False, steps=128, appends=False),
    # tiny: 1 request, 1 layer, MLA 16 heads, ctx 4096, k 256, B 512, keep 90%, recency 512
    "tiny": dict(R=1, L=1, ctx0=4096, layout=0, Hq=16, Hkv=1, Dqk=576, Dv=512, k=256, B=512,
                 keep=0.9, mu=512.0, burst=0, shared=False, steps=64),
}


DEFAULT_WORKLOAD = "gqa_b16_l32"

# dram__bytes_read.sum + dram__bytes_write.sum of one attention launch from an ncu capture of the
# same kernel and per-launch size (profiles/; ncu replays with cold caches, so this is the DRAM
# traffic of a launch whose rows are not in L2); None where no capture of the current kernel exists
ATTN_TRAFFIC = {("gqa_b16_l32", "resolve"): 138.54e6, ("mla_b8", "resolve"): 19.60e6}
L2_BYTES = 129e6  # GB300 L2


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def record_bytes(w):
    return 2 * w["Dqk"] if w["layout"] == 0 else 2 * w["Hkv"] * (w["Dqk"] + w["Dv"])


def launches_per_layer(w, separate_append=False):
    """This library's kernels launched per layer of a step: the resolve (the append fused in, or its
    own launch), then the attention; the 64-head shared-latent attention adds its split combine."""
    attn = 2 if w["layout"] == 0 and w["Hq"] == 64 else 1
    return 1 + (1 if separate_append else 0) + attn


def steps_exceed_l2(w):
    """True when one step's attention launches together gather well over L2's size, so that timing
    them back to back (and step after step) never finds a launch's rows left in L2 by the last."""
    return w["L"] * attn_bytes_per_launch(w) >= 2 * L2_BYTES


def attn_bytes_per_launch(w):
    """Algorithmic bytes of one attention launch (one layer, all requests): the k gathered
    records, q, the fp32 output and the slot list."""
    return w["R"] * (w["k"] * record_bytes(w) + w["Hq"] * w["Dqk"] * 2 + w["Hq"] * w["Dv"] * 4 + w["k"] * 4)


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.device_index = device_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "samples": len(sm), "reasons": sorted(reasons)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def reduce_max(value, world):
    """Max over ranks (gloo or NCCL); the identity for one process."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# --------------------------------------------------------------------------------------------
class Workload:
    """Seeded synthetic inputs of one replica, resident on the GPU."""

    def __init__(self, w, steps, device, seed, fetch="resolve", index_share=1):
        import torch

        from hierarchical_kv_cache_02_gb300 import HsConfig, inputs

        self.w, self.steps, self.device = w, steps, device
        R, L, k = w["R"], w["L"], w["k"]
        self.cfg = HsConfig(num_requests=R, num_layers=L, capacity=w["ctx0"] + steps, layout=w["layout"],
                            num_q_heads=w["Hq"], num_kv_heads=w["Hkv"], head_dim_qk=w["Dqk"], head_dim_v=w["Dv"],
                            top_k=k, buffer_slots=w["B"], policy=0, seed=seed, io_chunk_bytes=64,
                            shared_prefix=w["ctx0"] if w["shared"] else 0,
                            fetch_in_attention=1 if fetch == "attention" else 0,
                            early_fetch=1 if fetch == "early" else 0)
        self.appends = w.get("appends", True)
        spec = inputs.TraceSpec(ctx0=w["ctx0"], k=k, steps=steps, keep=w["keep"], recency_mean=w["mu"],
                                appends=self.appends, burst_every=w["burst"], far_gap=int(8 * w["mu"]))
        t0 = time.time()
        self.trace_host = inputs.drift_traces(spec, R, L, seed=seed)            # [S][L][R][k]
        if index_share > 1:
            # layer groups share one selection (the group's first layer's), as with a shared indexer
            for l in range(L):
                self.trace_host[:, l] = self.trace_host[:, index_share * (l // index_share)]
        self.trace_secs = time.time() - t0
        self.topk = torch.from_numpy(self.trace_host).to(device)
        E = self.cfg.record_elems
        self.q = inputs.normal_bf16((steps, L, R, w["Hq"], w["Dqk"]), seed=seed + 1, device=device)
        self.app = inputs.normal_bf16((steps, L, R, E), seed=seed + 2, device=device)
        self.pos = (torch.arange(steps, dtype=torch.int64, device=device) + w["ctx0"]).view(steps, 1).expand(
            steps, R).contiguous()
        self.hist_seed = seed + 3

    def history_layer(self, l, r=0):
        """The prefilled records of (r, l): regenerated from its seed (no copy kept)."""
        from hierarchical_kv_cache_02_gb300 import inputs

        w = self.w
        s = self.hist_seed + 7919 * l + (0 if w["shared"] else 104729 * (r + 1))
        return inputs.normal_bf16((w["ctx0"], self.cfg.record_elems), seed=s, device=self.device)

    def prefill(self, pool):
        w = self.w
        for l in range(w["L"]):
            for r in range(1 if w["shared"] else w["R"]):
                pool.prefill(r, l, 0, self.history_layer(l, r))


def replica_seed(rank):
    """Seed of the synthetic inputs of replica `rank`: every rank serves its own batch of requests
    (its own traces, queries and histories), as independent replicas sharded by request would."""
    return 1000 + 17 * rank


def run_ours(args, w, world, rank, local):
    import torch

    from hierarchical_kv_cache_02_gb300 import HsPool, _lib

    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    _lib.load()
    W, K = args.warmup, args.steps
    S = W + K
    t_setup = time.time()
    fetch = args.fetch
    if fetch == "auto":
        fetch = "resolve"  # each kernel against its own roofline; "attention" overlaps the link with HBM
    G = max(1, args.index_share)
    wl = Workload(w, S, device, seed=replica_seed(rank), fetch=fetch, index_share=G)
    pool = HsPool(wl.cfg, device=local)
    wl.prefill(pool)
    torch.cuda.synchronize()
    setup_secs = time.time() - t_setup
    R, L, k = w["R"], w["L"], w["k"]
    scale = wl.cfg.default_scale
    locs = [torch.empty((R, k), dtype=torch.int32, device=device) for _ in range(L)]
    outs = [torch.empty((R, w["Hq"], w["Dv"]), dtype=torch.float32, device=device) for _ in range(L)]
    stream = torch.cuda.current_stream()

    def step(t, ev=None):
        for l in range(L):
            if ev is not None:
                ev[l][0].record(stream)
            if args.separate_append and wl.appends:
                pool.append(l, wl.pos[t], wl.app[t, l])
            if ev is not None:
                ev[l][1].record(stream)
            if args.separate_append or not wl.appends:
                pool.resolve(l, wl.topk[t, l], locs[l])
            else:
                pool.append_resolve(l, wl.pos[t], wl.app[t, l], wl.topk[t, l], locs[l])
            if ev is not None:
                ev[l][2].record(stream)
            pool.sparse_attn(l, wl.q[t, l], locs[l], outs[l], scale=scale)
            if ev is not None:
                ev[l][3].record(stream)

    # group mode: attentions on their own stream, resolves of the group each on a side stream (equal
    # priorities: giving the attentions priority measured slower, the resolves' fetches then lack SMs)
    astream = torch.cuda.Stream() if G > 1 else stream
    side = [torch.cuda.Stream() for _ in range(G)] if G > 1 else []

    def step_group(t, ev=None):
        # layer-group prefetch: a group's selection is known once the layer before the group has
        # finished its attention, so all resolves of the group (with their host fetches) start then,
        # each on its own stream; the attentions follow in layer order as their resolves complete
        for l0 in range(0, L, G):
            known = torch.cuda.Event()
            known.record(astream)
            done = []
            for j, l in enumerate(range(l0, min(L, l0 + G))):
                st = side[j]
                st.wait_event(known)
                with torch.cuda.stream(st):
                    if ev is not None:
                        ev[l][1].record(st)
                    if wl.appends:
                        pool.append_resolve(l, wl.pos[t], wl.app[t, l], wl.topk[t, l], locs[l], stream=st)
                    else:
                        pool.resolve(l, wl.topk[t, l], locs[l], stream=st)
                    if ev is not None:
                        ev[l][2].record(st)
                e = torch.cuda.Event()
                e.record(st)
                done.append(e)
            for j, l in enumerate(range(l0, min(L, l0 + G))):
                astream.wait_event(done[j])
                with torch.cuda.stream(astream):
                    if ev is not None:
                        ev[l][0].record(astream)
                    pool.sparse_attn(l, wl.q[t, l], locs[l], outs[l], scale=scale, stream=astream)
                    if ev is not None:
                        ev[l][3].record(astream)

    M = max(1, args.microbatches)
    groups = [(R * g // M, R * (g + 1) // M - R * g // M) for g in range(M)]
    streams = [torch.cuda.Stream() for _ in range(M)] if M > 1 else [stream]
    gevs = [[[[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(L)] for _ in range(M)]
            for _ in range(K)] if M > 1 else None

    def step_mb(t, i=None):
        # micro-batches: each group of requests runs its layers in order on its own stream.  The
        # groups' resolves form one chain (group g's resolve of layer l after group g-1's), and so do
        # their attentions, so one group's resolve runs while the group before it is in its attention
        # and the attentions (which copy the misses when fetch_in_attention is set) follow one another
        # on the host link instead of sharing it
        last_res, last_att = None, None
        for l in range(L):
            for g, (r0, n) in enumerate(groups):
                st = streams[g]
                with torch.cuda.stream(st):
                    if last_res is not None:
                        st.wait_event(last_res)
                    if i is not None:
                        gevs[i][g][l][0].record(st)
                    pool.resolve_range(l, r0, wl.topk[t, l, r0:r0 + n], locs[l][r0:r0 + n],
                                       pos=wl.pos[t, r0:r0 + n], rec=wl.app[t, l, r0:r0 + n], stream=st)
                    last_res = torch.cuda.Event()
                    last_res.record(st)
                    if i is not None:
                        gevs[i][g][l][1].record(st)
                    if last_att is not None:
                        st.wait_event(last_att)
                    if i is not None:
                        gevs[i][g][l][2].record(st)
                    pool.sparse_attn_range(l, r0, wl.q[t, l, r0:r0 + n], locs[l][r0:r0 + n],
                                           outs[l][r0:r0 + n], scale=scale, stream=st)
                    last_att = torch.cuda.Event()
                    last_att.record(st)
                    if i is not None:
                        gevs[i][g][l][3].record(st)

    def fork():
        cur = torch.cuda.current_stream()
        ev = torch.cuda.Event()
        ev.record(cur)
        for st in streams:
            st.wait_event(ev)

    def join():
        cur = torch.cuda.current_stream()
        for st in streams:
            ev = torch.cuda.Event()
            ev.record(st)
            cur.wait_event(ev)

    # the headline pass replays the K timed steps as one captured CUDA graph
    use_graph = not args.no_graph and G == 1

    def warm_up():
        """Cold start, then the W untimed warm-up steps."""
        pool.reset()
        for t in range(W):
            if M > 1:
                fork()
                step_mb(t)
                join()
            elif G > 1:
                astream.wait_stream(stream)
                step_group(t)
                stream.wait_stream(astream)
            else:
                step(t)
        torch.cuda.synchronize()
        pool.stats(reset=True)

    def run_steps(timed_events):
        """Cold start, W untimed warm-up steps, then K timed steps; returns seconds and pool stats."""
        graph = None
        if use_graph and not timed_events:
            # capture the timed steps after the warm-up and replay them once untimed (a graph's first
            # launch also uploads it); the timed replay then starts over from the same state
            warm_up()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                if M > 1:
                    fork()
                    for i in range(K):
                        step_mb(W + i)
                    join()
                else:
                    for i in range(K):
                        step(W + i)
            graph.replay()
            torch.cuda.synchronize()
        warm_up()
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        start.record(stream)
        if graph is not None:
            graph.replay()
        elif M > 1:
            fork()
            for i in range(K):
                step_mb(W + i, i if timed_events else None)
            join()
        elif G > 1:
            astream.wait_stream(stream)
            for i in range(K):
                step_group(W + i, evs[i] if timed_events else None)
            stream.wait_stream(astream)
        else:
            for i in range(K):
                step(W + i, evs[i] if timed_events else None)
        stop.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return start.elapsed_time(stop) / 1e3, pool.stats()

    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(L)] for _ in range(K)]
    # pass 1 (the headline): kernels back to back, no events between them (an event between two
    # kernels also blocks programmatic dependent launch)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    elapsed, st = run_steps(False)
    clk = clocks.stop()
    # pass 2: the same steps from the same cold start, with CUDA events around every kernel
    elapsed_ev, st_ev = run_steps(True)
    if M > 1:
        res_ms = np.array([[[e[g][l][0].elapsed_time(e[g][l][1]) for l in range(L)] for g in range(M)] for e in gevs])
        att_ms = np.array([[[e[g][l][2].elapsed_time(e[g][l][3]) for l in range(L)] for g in range(M)] for e in gevs])
        app_ms = np.zeros(1)
    elif G > 1:
        # resolves on their own streams, attentions on the main stream after their resolve
        app_ms = np.zeros(1)
        res_ms = np.array([[e[l][1].elapsed_time(e[l][2]) for l in range(L)] for e in evs])
        att_ms = np.array([[e[l][0].elapsed_time(e[l][3]) for l in range(L)] for e in evs])
    else:
        app_ms = np.array([[e[l][0].elapsed_time(e[l][1]) for l in range(L)] for e in evs])
        res_ms = np.array([[e[l][1].elapsed_time(e[l][2]) for l in range(L)] for e in evs])
        att_ms = np.array([[e[l][2].elapsed_time(e[l][3]) for l in range(L)] for e in evs])
    # pass 3: the attention alone, its L launches of the last step back to back; only where the L
    # launches together gather well over L2's size, so that no replay finds the last one's rows cached
    big = steps_exceed_l2(w)
    # a step that gathers at least half of L2 is timed as replays with L2 flushed in between; a smaller
    # one stays in L2 from one decode step to the next, as the hot buffers of such a workload would
    flushed = not big and w["L"] * attn_bytes_per_launch(w) * 2 >= L2_BYTES
    attn_b2b_us = None
    if M == 1 and G == 1 and big:
        attn_b2b_us = time_attention_back_to_back(pool, wl, locs, outs, scale, W + K - 1)
    elif M == 1 and G == 1 and flushed:
        attn_b2b_us = time_attention_flushed(pool, wl, locs, outs, scale, W + K - 1)
    max_elapsed = reduce_max(elapsed, world)
    units = world * K * L
    value = units / max_elapsed

    # ---- end to end through the public API: inputs from pinned host memory, outputs back -----
    e2e = None
    if not args.no_e2e and G == 1:
        e2e = run_e2e(pool, wl, W, K, world, locs, outs, scale, use_graph)

    # ---- host-link peak on this machine: pinned H2D copy, best of 5 ----
    h2d = measure_h2d(device)
    floor_us = measure_launch_floor()
    peaks = load_peaks()
    attn_us = float(att_ms.mean() * 1e3)
    # the roofline takes the back-to-back launch time where there is one (the event pair around a
    # single launch also holds the launch latency that the event between two kernels exposes)
    roof_us = attn_b2b_us if attn_b2b_us is not None else attn_us
    achieved = attn_bytes_per_launch(w) / M / (roof_us * 1e-6) / 1e9  # a launch covers R / M requests
    achieved_ev = attn_bytes_per_launch(w) / M / (attn_us * 1e-6) / 1e9
    rec = record_bytes(w)
    miss_bytes = float(st["host_bytes"])
    res_total_s = float(res_ms.sum() / 1e3)  # micro-batches' resolves (and attentions) run one after another
    link_kernel = "sparse_attn" if fetch == "attention" else "resolve"
    link_s = float(att_ms.sum() / 1e3) if fetch == "attention" else res_total_s
    if G > 1:
        # the group's resolves overlap one another and the attentions: link rate over the wall time
        link_kernel, link_s = "resolve (overlapped; whole-step wall time)", max_elapsed
    elif M > 1 and fetch == "attention":
        # the micro-batches' attentions move the misses one after another while the other group's
        # resolve decides: the link's average rate over the wall time of the steps
        link_kernel, link_s = "sparse_attn (micro-batches overlapped; whole-step wall time)", max_elapsed
    out = {
        "metric": METRIC, "value": value, "unit": "layer-steps/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": max_elapsed / K * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "requests": R, "layers": L, "context": w["ctx0"], "top_k": k,
                   "buffer_slots": w["B"], "layout": "gqa" if w["layout"] == 1 else "mla", "q_heads": w["Hq"],
                   "kv_heads": w["Hkv"], "record_bytes": rec, "policy": "lru", "keep": w["keep"],
                   "recency_mean": w["mu"], "burst_every": w["burst"], "shared_history": w["shared"],
                   "append": True, "miss_fetch": fetch, "microbatches": M,
                   "index_share": G, "parallelism": f"replicas{world}",
                   "launch": "one captured CUDA graph of the timed steps" if use_graph else "stream launches",
                   "l2": (f"inputs larger than L2 (each attention launch gathers "
                          f"{attn_bytes_per_launch(w) / 1e6:.0f} MB; a step touches {L} layers)") if big else
                         (f"a step's {L} attention launches gather {L * attn_bytes_per_launch(w) / 1e6:.0f} MB, "
                          "more than L2, and the steps run without a flush; the attention roofline is timed "
                          "with L2 flushed before each replay") if flushed else
                         (f"inputs smaller than L2, no flush: a step's {L} attention launch(es) gather "
                          f"{L * attn_bytes_per_launch(w) / 1e6:.0f} MB, so the hot buffers stay in L2 "
                          "from one decode step to the next, as they would in this workload's steady state")},
        "kernel_timing": "second timed pass over the same steps from the same cold start, CUDA events "
                         f"around every kernel ({elapsed_ev / (K * L) * 1e6:.1f} us/layer with the events)",
        "us_per_layer": {"total": max_elapsed / (K * L) * 1e6,
                         "resolve": float(res_ms.mean() * 1e3),  # includes the append when fused
                         "sparse_attn": attn_us, "append": float(app_ms.mean() * 1e3),
                         "resolve_plus_attn": float((res_ms + att_ms).mean() * 1e3)},
        "miss_rate": float(st["misses"]) / max(1.0, float(st["hits"] + st["misses"])),
        "roofline": {"kernel": "sparse_attn", "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": args.traffic if args.traffic is not None else ATTN_TRAFFIC.get((args.workload, "resolve" if fetch == "early" else fetch)),
                     "peak_source": peaks["source"],
                     "bytes_per_launch": attn_bytes_per_launch(w) // M,
                     "launch_us": roof_us,
                     "timing": ("CUDA events around 3 replays of a captured graph of the last timed step's "
                                f"{L} attention launches back to back (inputs of each launch larger than L2)")
                     if attn_b2b_us is not None and big else
                     (f"CUDA events around each of 5 replays of a captured graph of the last timed step's {L} "
                      "attention launches, L2 flushed before each replay (median)")
                     if attn_b2b_us is not None else "CUDA events around each launch",
                     # the same from the event pairs around each launch of the breakdown pass
                     "per_launch_events_us": attn_us,
                     "frac_per_launch_events": achieved_ev / peaks["hbm_gbs"],
                     "launch_floor_us": floor_us,
                     "share_of_layer": float(att_ms.mean() / (res_ms.mean() + att_ms.mean()))},
        # the kernel that moves the misses over the host link: the resolve, or the attention when the
        # copies were left to it
        # the resolve takes most of a layer's time and is bound by the host link, a resource with no
        # peak in MEASURED_PEAKS.json: its roofline is this object, against a pinned copy timed in
        # this run
        "host_link": {"kernel": link_kernel, "bound": "host link (NVLink-C2C)",
                      "miss_bytes_per_layer": miss_bytes / (K * L),
                      "achieved_gbs": miss_bytes / link_s / 1e9 if link_s > 0 else None,
                      "h2d_copy_peak_gbs": h2d,
                      "frac": (miss_bytes / link_s / 1e9) / h2d if link_s > 0 and h2d else None,
                      "share_of_layer": float(res_ms.mean() / (res_ms.mean() + att_ms.mean()))},
        "gpu_launches": K * L * launches_per_layer(w, args.separate_append),
        "clocks": clk,
        "setup_s": setup_secs,
        "errors": int(st["error_bits"]),
    }
    if e2e is not None:
        out["e2e"] = e2e
    pool.close()
    return out


def run_e2e(pool, wl, W, K, world, locs, outs, scale, use_graph=False):
    """Same steps after a cold reset, with every step's top-k, queries and new records copied from
    pinned host memory and all its attention outputs copied back, inside the timed region.  As a
    serving loop would, a copy stream moves step t+1's inputs in and step t's outputs out while
    step t computes (inputs and outputs double-buffered)."""
    import torch

    w = wl.w
    R, L, k = w["R"], w["L"], w["k"]
    S = W + K
    h_topk = torch.from_numpy(wl.trace_host).pin_memory()
    h_q = wl.q.cpu().pin_memory()
    h_app = wl.app.cpu().pin_memory()
    h_pos = wl.pos.cpu().pin_memory()
    h_out = torch.empty((S, L, R, w["Hq"], w["Dv"]), dtype=torch.float32).pin_memory()
    dev = wl.device
    d_topk = [torch.empty((L, R, k), dtype=torch.int32, device=dev) for _ in range(2)]
    d_q = [torch.empty((L, R, w["Hq"], w["Dqk"]), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    d_app = [torch.empty((L, R, wl.cfg.record_elems), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    d_pos = [torch.empty((R,), dtype=torch.int64, device=dev) for _ in range(2)]
    d_out = [torch.empty((L, R, w["Hq"], w["Dv"]), dtype=torch.float32, device=dev) for _ in range(2)]
    stream = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of the buffer's step have landed
    ev_done = [torch.cuda.Event() for _ in range(2)]  # the buffer's step has computed
    ev_out = [torch.cuda.Event() for _ in range(2)]   # its outputs are back on the host

    def copy_in(t):
        b = t % 2
        copy.wait_event(ev_done[b])  # the step that used these buffers two steps ago is done
        with torch.cuda.stream(copy):
            d_topk[b].copy_(h_topk[t], non_blocking=True)
            d_q[b].copy_(h_q[t], non_blocking=True)
            d_app[b].copy_(h_app[t], non_blocking=True)
            d_pos[b].copy_(h_pos[t], non_blocking=True)
            ev_in[b].record(copy)

    def compute_and_copy_out(t):
        b = t % 2
        cur = torch.cuda.current_stream()
        cur.wait_event(ev_in[b])
        cur.wait_event(ev_out[b])  # outputs of two steps ago have left these buffers
        for l in range(L):
            if wl.appends:
                pool.append_resolve(l, d_pos[b], d_app[b][l], d_topk[b][l], locs[l])
            else:
                pool.resolve(l, d_topk[b][l], locs[l])
            pool.sparse_attn(l, d_q[b][l], locs[l], d_out[b][l], scale=scale)
        ev_done[b].record(cur)
        copy.wait_event(ev_done[b])
        with torch.cuda.stream(copy):
            h_out[t].copy_(d_out[b], non_blocking=True)
            ev_out[b].record(copy)

    def run(t0, t1):
        cur = torch.cuda.current_stream()
        for e in ev_done + ev_out:  # no step is using either buffer yet
            e.record(cur)
        copy.wait_stream(cur)
        copy_in(t0)
        for t in range(t0, t1):
            if t + 1 < t1:
                copy_in(t + 1)
            compute_and_copy_out(t)
        cur.wait_stream(copy)

    graph = None
    if use_graph:
        # the timed steps, copies included, as one captured graph, replayed once untimed first
        pool.reset()
        run(0, W)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            run(W, S)
        graph.replay()
        torch.cuda.synchronize()
    pool.reset()
    run(0, W)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    start.record(stream)
    if graph is not None:
        graph.replay()
    else:
        run(W, S)
    stop.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    el = reduce_max(start.elapsed_time(stop) / 1e3, world)
    h2d_bytes = (h_topk[0].numel() * 4 + h_q[0].numel() * 2 + h_app[0].numel() * 2 + h_pos[0].numel() * 8)
    d2h_bytes = L * R * w["Hq"] * w["Dv"] * 4
    return {"value": world * K * L / el, "unit": "layer-steps/s", "h2d_bytes_per_step": int(h2d_bytes),
            "d2h_bytes_per_step": int(d2h_bytes), "ms_per_step": el / K * 1e3}


def time_attention_back_to_back(pool, wl, locs, outs, scale, t, reps=3):
    """Mean device time of one attention launch: the L layers' launches of step t, captured as one
    graph (programmatic dependent launch between them, no events in between), replayed once untimed,
    then `reps` times between two CUDA events.  Every launch gathers its own layer's hot buffers, more
    than L2 holds, so no launch finds its rows cached by the one before."""
    import torch

    L = wl.w["L"]

    def launches():
        for l in range(L):
            pool.sparse_attn(l, wl.q[t, l], locs[l], outs[l], scale=scale)

    launches()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        launches()
    graph.replay()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(reps):
        graph.replay()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) * 1e3 / (reps * L)


def time_attention_flushed(pool, wl, locs, outs, scale, t, reps=5):
    """Mean device time of one attention launch for workloads whose step gathers less than twice L2:
    the L layers' launches of step t, captured as one graph, replayed `reps` times; before each
    replay a write of twice L2's size evicts what the last replay left there, and CUDA events on the
    launching stream bracket the replay alone (the event pair's own latency is spread over L launches)."""
    import torch

    L = wl.w["L"]

    def launches():
        for l in range(L):
            pool.sparse_attn(l, wl.q[t, l], locs[l], outs[l], scale=scale)

    launches()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        launches()
    graph.replay()
    flush = torch.empty(int(2 * L2_BYTES) // 4, dtype=torch.float32, device=wl.device)
    torch.cuda.synchronize()
    times = []
    for i in range(reps):
        flush.fill_(float(i))
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        graph.replay()
        e.record()
        torch.cuda.synchronize()
        times.append(s.elapsed_time(e) * 1e3 / L)
    del flush
    return float(np.median(times))


def measure_h2d(device):
    import torch

    n = 1 << 30
    h = torch.empty(n, dtype=torch.uint8).pin_memory()
    d = torch.empty(n, dtype=torch.uint8, device=device)
    best = float("inf")
    for _ in range(5):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        d.copy_(h, non_blocking=True)
        e.record()
        torch.cuda.synchronize()
        best = min(best, s.elapsed_time(e) / 1e3)
    del h, d
    return n / best / 1e9


def measure_launch_floor():
    """CUDA-event time of a kernel that does nothing (median of 30 enqueued back to back, so the device
    never waits for the host): the per-launch floor that the event pairs around every kernel of the
    breakdown pass include."""
    import torch

    torch.cuda._sleep(1000000)  # keep the device busy while the pairs are enqueued
    pairs = []
    for _ in range(30):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        torch.cuda._sleep(1)
        e.record()
        pairs.append((s, e))
    torch.cuda.synchronize()
    return float(np.median([s.elapsed_time(e) * 1e3 for s, e in pairs]))


# --------------------------------------------------------------------------------------------
def oracle_sample(w, steps, seed, budget_s, pairs_max=64):
    """Time the CPU oracle on (request, layer) pairs of the workload: each pair replays its own
    top-k trace from step 0 (append, resolve) with fp64 attention every step, until the time
    budget is spent.  Returns seconds per (request, layer)-step and a description."""
    import torch

    import oracle
    from hierarchical_kv_cache_02_gb300 import inputs

    R, L, k = w["R"], w["L"], w["k"]
    appends = w.get("appends", True)
    spec = inputs.TraceSpec(ctx0=w["ctx0"], k=k, steps=steps, keep=w["keep"], recency_mean=w["mu"], appends=appends,
                            burst_every=w["burst"], far_gap=int(8 * w["mu"]))
    E = record_bytes(w) // 2
    kvh = 0 if w["layout"] == 0 else w["Hkv"]
    scale = float(np.float32(1.0 / math.sqrt(w["Dqk"])))
    # one history stands in for every sampled pair: the oracle's cost does not depend on the values
    hist = inputs.normal_bf16((w["ctx0"] + steps, E), seed=seed).view(torch.int16).numpy().view(np.uint16)
    total_t, n_rl_steps, pairs = 0.0, 0, 0
    cache_t = 0.0  # of which the cache simulation (append, resolve); the rest is the fp64 attention
    for p in range(pairs_max):
        r, l = p % R, (p * 7) % L
        # the trace of (r, l) in a batch seeded `seed` is the single trace seeded seed + r*65536 + l
        tr = inputs.drift_traces(spec, 1, 1, seed=seed + r * 65536 + l)[:, 0, 0]
        q = inputs.normal_bf16((steps, w["Hq"], w["Dqk"]), seed=seed + 1 + p).view(torch.int16).numpy().view(np.uint16)
        cache = oracle.Cache(w["B"], k, "lru", R=R, L=L, r=r, l=l, C=w["ctx0"] + steps)
        t0 = time.perf_counter()
        for t in range(steps):
            c0 = time.perf_counter()
            if appends:
                cache.append(w["ctx0"] + t)
            cache.resolve(tr[t])
            cache_t += time.perf_counter() - c0
            oracle.attention(q[t], hist, tr[t], scale, kvh, w["Dqk"], w["Dv"])
            n_rl_steps += 1
            if total_t + time.perf_counter() - t0 > budget_s:
                break
        total_t += time.perf_counter() - t0
        pairs += 1
        if total_t > budget_s:
            break
    per = total_t / max(1, n_rl_steps)
    desc = (f"{n_rl_steps} (request, layer)-steps of {pairs} pairs, each replayed from step 0 (append, resolve, "
            f"fp64 attention), {total_t:.1f} s on 1 core ({cache_t:.1f} s of it the cache simulation); "
            f"layer-steps/s = 1 / ({R} x s per (request, layer)-step)")
    split = {"cache_us_per_layer": R * cache_t / max(1, n_rl_steps) * 1e6,
             "attention_us_per_layer": R * (total_t - cache_t) / max(1, n_rl_steps) * 1e6}
    return per, desc, n_rl_steps, split


def cpu_info():
    """CPU model and the number of online cores of this host (for the CPU baselines)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith(("model name", "cpu model")):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return {"cpu_model": model or "unknown", "nproc": os.cpu_count()}


def run_reference(args, w, world, rank):
    """The CPU oracle on the host cores (rank 0 only).  Each of the W + K steps advances the same
    sample of (request, layer) pairs by one decode step -- append, resolve, fp64 attention -- which
    is a bounded part of the workload's R x L pairs; the K timed steps give the rate per (request,
    layer)-step, and `value` extrapolates it to whole layers (R pairs each) of the workload."""
    if rank != 0:
        return None
    import torch

    import oracle
    from hierarchical_kv_cache_02_gb300 import inputs

    K, W = args.steps, args.warmup
    budget = float(os.environ.get("HS_REF_STEP_SECONDS", "1.0"))  # seconds of oracle work per step
    R, L, k = w["R"], w["L"], w["k"]
    steps = W + K
    appends = w.get("appends", True)
    spec = inputs.TraceSpec(ctx0=w["ctx0"], k=k, steps=steps, keep=w["keep"], recency_mean=w["mu"], appends=appends,
                            burst_every=w["burst"], far_gap=int(8 * w["mu"]))
    E = record_bytes(w) // 2
    kvh = 0 if w["layout"] == 0 else w["Hkv"]
    scale = float(np.float32(1.0 / math.sqrt(w["Dqk"])))
    # one history stands in for every sampled pair: the oracle's cost does not depend on the values
    hist = inputs.normal_bf16((w["ctx0"] + steps, E), seed=99).view(torch.int16).numpy().view(np.uint16)
    pairs = []

    def add_pair(p):
        r, l = p % R, (p * 7) % L
        tr = inputs.drift_traces(spec, 1, 1, seed=99 + r * 65536 + l)[:, 0, 0]  # the trace of (r, l)
        q = inputs.normal_bf16((steps, w["Hq"], w["Dqk"]), seed=100 + p).view(torch.int16).numpy().view(np.uint16)
        pairs.append((oracle.Cache(w["B"], k, "lru", R=R, L=L, r=r, l=l, C=w["ctx0"] + steps), tr, q))

    cache_s = [0.0]  # time of the cache simulation (append, resolve) in the timed steps

    def advance(i, t, timed=False):
        cache, tr, q = pairs[i]
        c0 = time.perf_counter()
        if appends:
            cache.append(w["ctx0"] + t)
        cache.resolve(tr[t])
        if timed:
            cache_s[0] += time.perf_counter() - c0
        oracle.attention(q[t], hist, tr[t], scale, kvh, w["Dqk"], w["Dv"])

    # size the sample on the first warm-up step: pairs are added until the step has used its budget
    t0 = time.perf_counter()
    while len(pairs) < R * L and (not pairs or time.perf_counter() - t0 < budget):
        add_pair(len(pairs))
        advance(len(pairs) - 1, 0)
    P = len(pairs)
    for t in range(1, W):
        for i in range(P):
            advance(i, t)
    t_start = time.perf_counter()
    for t in range(W, steps):
        for i in range(P):
            advance(i, t, timed=True)
    elapsed = time.perf_counter() - t_start
    per = elapsed / (P * K)  # seconds per (request, layer)-step
    value = 1.0 / (R * per)
    desc = (f"each of the {K} timed steps (after {W} warm-up steps) advanced the same {P} of the workload's "
            f"{R * L} (request, layer) pairs by one decode step (append, resolve, fp64 attention): {P * K} "
            f"(request, layer)-steps in {elapsed:.1f} s on 1 core; value = 1 / ({R} x s per (request, layer)-step), "
            f"extrapolated from the sample to whole layers")
    info = cpu_info()
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "layer-steps/s", "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": elapsed / K * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "extrapolated": True,
            "timed_work": {"pairs_per_step": P, "pairs_per_layer": R, "layers": L,
                           "ms_per_step": "wall time of one sampled step as run (P pairs), not of a whole step",
                           "seconds_timed": elapsed},
            "config": {"workload": args.workload, "requests": R, "layers": L, "context": w["ctx0"],
                       "top_k": k, "buffer_slots": w["B"]},
            "cpu_baseline": {"value": value, "unit": "layer-steps/s", "cores": 1, "kind": "oracle", "sample": desc,
                             "cache_us_per_layer": R * cache_s[0] / (P * K) * 1e6,
                             "attention_us_per_layer": R * (elapsed - cache_s[0]) / (P * K) * 1e6, **info},
            "e2e": {"value": value, "unit": "layer-steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=56)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (small profiling runs)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--microbatches", type=int, default=1,
                    help="split the requests into this many groups, each running its layers on its own stream; "
                         "the groups' resolves form one chain and their attentions another")
    ap.add_argument("--separate-append", action="store_true",
                    help="append and resolve as two launches instead of the fused hs_append_resolve")
    ap.add_argument("--fetch", choices=["auto", "resolve", "early", "attention"], default="auto",
                    help="who copies the misses host -> HBM: the resolve kernel once it has chosen the victims, "
                         "the resolve with fetch CTAs that start copying while the victims are chosen (early), "
                         "or the attention while it gathers")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--index-share", type=int, default=1,
                    help="layer groups of this size share one selection; their resolves (and host fetches) "
                         "run together on side streams, overlapping the attentions (exact layer-group prefetch)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the headline pass's kernels one by one instead of replaying a captured graph")
    ap.add_argument("--no-alt", action="store_true",
                    help="skip the extra GQA passes: two micro-batches with the miss copies inside the "
                         "attention, and layer groups sharing one selection")
    ap.add_argument("--no-latent", action="store_true",
                    help="skip the shared-latent workloads (stress batch, MLA batch of 8) reported beside the "
                         "default GQA line")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per attention launch from an ncu capture of the same kernel")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    w = dict(WORKLOADS[args.workload])
    if args.layers:
        w["L"] = args.layers
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        out = run_reference(args, w, world, rank)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    out = run_ours(args, w, world, rank, local)
    if args.fetch == "auto" and w["layout"] == 1 and not args.no_alt:
        # the same steps with the miss copies moved into the attention kernel (overlapping the host
        # link with the HBM gather): reported beside the headline, which keeps the copies in the resolve
        # in two micro-batches, so one half's resolve runs while the other half's attention copies
        alt_args = argparse.Namespace(**vars(args))
        alt_args.fetch, alt_args.no_e2e, alt_args.microbatches = "attention", True, 2
        alt = run_ours(alt_args, w, world, rank, local)
        out["fetch_in_attention"] = {k: alt[k] for k in ("value", "unit", "ms_per_step", "us_per_layer", "miss_rate",
                                                         "host_link", "clocks", "errors")}
        out["fetch_in_attention"]["microbatches"] = 2
    if args.fetch == "auto" and w["layout"] == 1 and not args.no_alt and args.index_share == 1 and w["L"] >= 4:
        # a different workload: layer groups of 4 share one selection (as with a shared indexer), so a
        # group's resolves and host fetches start together and overlap the attentions (exact
        # layer-group prefetch); misses copied inside the attention
        grp_args = argparse.Namespace(**vars(args))
        grp_args.fetch, grp_args.no_e2e, grp_args.index_share = "attention", True, 4
        grp = run_ours(grp_args, w, world, rank, local)
        out["layer_group_prefetch"] = {k: grp[k] for k in ("value", "unit", "ms_per_step", "miss_rate", "host_link",
                                                           "clocks", "errors")}
        out["layer_group_prefetch"]["us_per_layer"] = grp["us_per_layer"]["total"]
        out["layer_group_prefetch"]["workload"] = "same sizes; layer groups of 4 share one top-k selection"
    if (args.workload == DEFAULT_WORKLOAD and args.fetch == "auto" and not args.no_alt and not args.no_latent
            and args.microbatches == 1 and args.index_share == 1 and not args.layers):
        # the shared-latent workloads of the same metric, each with its own attention and resolve
        # rooflines (the 64-head tcgen05 attention and its split combine; the resolve's host link)
        latent = {}
        for name in ("stress_b16_l4", "mla_b8"):
            la = argparse.Namespace(**vars(args))
            la.workload, la.no_e2e = name, True
            # at least 256 timed layer-steps: a step of these batches takes tens of microseconds, and a
            # short timed region lets one slow step move the figure by several percent
            la.steps = max(args.steps, 256 // WORKLOADS[name]["L"])
            res = run_ours(la, dict(WORKLOADS[name]), world, rank, local)
            latent[name] = {k: res[k] for k in ("value", "unit", "steps", "ms_per_step", "us_per_layer", "miss_rate",
                                                "roofline", "host_link", "gpu_launches", "clocks", "errors", "config")}
        out["shared_latent"] = latent
    if rank == 0 and not args.no_cpu_baseline:
        per, desc, n, split = oracle_sample(w, steps=min(16, args.warmup + args.steps), seed=99,
                                            budget_s=args.cpu_seconds)
        out["cpu_baseline"] = {"value": 1.0 / (w["R"] * per), "unit": "layer-steps/s", "cores": 1, "kind": "oracle",
                               "sample": desc, **split, **cpu_info()}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
