"""GPU parity: the CUDA library against the oracle, element by element, through the C ABI.

Bit-exact: slot of every selected position (locs), tags, stamps, clocks, per-step misses,
hit/miss/append/host-byte counters, hot-buffer contents and the written-through history.
Attention: max-abs <= 2e-2 and mean-abs <= 2e-3 against fp64 (and within the fp32 bound).
"""
import numpy as np
import pytest

from harness import (OracleRun, Scenario, assert_attn_close, assert_layer_matches_oracle, assert_pool_matches_oracle,
                     bf16_tensor, gpu_step, prefill)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from hierarchical_kv_cache_02_gb300 import (DEVERR_APPEND, DEVERR_DUP, DEVERR_LOC, DEVERR_RANGE, LAYOUT_GQA,
                                             LAYOUT_MLA, HsConfig, HsPool)


def _gqa(R, L, C, k, B, policy=0, kvh=8, G=4, io=64, log=0, P0=0, seed=3, fetch=0):
    """fetch: 0 the resolve copies the misses, 1 the attention does, 2 the resolve with fetch CTAs
    that start copying the misses before the decision ends (early_fetch)."""
    return HsConfig(num_requests=R, num_layers=L, capacity=C, layout=LAYOUT_GQA, num_q_heads=kvh * G,
                    num_kv_heads=kvh, head_dim_qk=128, head_dim_v=128, top_k=k, buffer_slots=B, policy=policy,
                    seed=seed, io_chunk_bytes=io, log_steps=log, shared_prefix=P0, fetch_in_attention=int(fetch == 1),
                    early_fetch=int(fetch == 2))


def _mla(R, L, C, k, B, Hq=16, policy=0, io=64, log=0, P0=0, early=0):
    return HsConfig(num_requests=R, num_layers=L, capacity=C, layout=LAYOUT_MLA, num_q_heads=Hq, num_kv_heads=1,
                    head_dim_qk=576, head_dim_v=512, top_k=k, buffer_slots=B, policy=policy, seed=11,
                    io_chunk_bytes=io, log_steps=log, shared_prefix=P0, early_fetch=early)


def run_and_compare(sc: Scenario, attn_every=1, check_state=True, fused=False):
    cfg = sc.cfg
    pool = HsPool(cfg)
    prefill(pool, sc)
    orc = OracleRun(sc)
    worst = 0.0
    for t in range(sc.steps):
        res = gpu_step(pool, sc, t, attn=(t % attn_every == 0), fused=fused)
        ref = orc.step(t)
        for l in range(cfg.num_layers):
            locs, out = res[l]
            for r in range(cfg.num_requests):
                m, rlocs = ref[(r, l)]
                assert np.array_equal(locs[r], rlocs), (t, r, l)
                if out is not None:
                    worst = max(worst, assert_attn_close(out[r], orc.attention(t, r, l), (t, r, l),
                                                         tight=cfg.layout == LAYOUT_GQA))
            if check_state:
                tag, stamp, clock = pool.read_state(l)
                for r in range(cfg.num_requests):
                    otag, ostamp = orc.caches[(r, l)].slots()
                    assert np.array_equal(tag[r], otag), (t, r, l)
                    assert np.array_equal(stamp[r], ostamp), (t, r, l)
                    assert clock[r] == orc.caches[(r, l)].counters()["clock"]
    st = pool.stats()
    tot = {"hits": 0, "misses": 0, "appends": 0}
    for (r, l), cache in orc.caches.items():
        cnt = cache.counters()
        assert list(st["per_rl"][r, l, :3]) == [cnt["hits"], cnt["misses"], cnt["appends"]], (r, l)
        assert st["per_rl"][r, l, 3] == cnt["misses"] * cfg.record_bytes
        for key in tot:
            tot[key] += cnt[key]
    assert st["error_bits"] == 0 and st["status"] == 0
    # hot buffer holds exactly the history record of every tagged slot; appended history written through
    for l in range(cfg.num_layers):
        tag, _, _ = pool.read_state(l)
        for r in range(cfg.num_requests):
            buf = pool.read_buffer(r, l)
            occ = np.nonzero(tag[r] >= 0)[0]
            assert np.array_equal(buf[occ], sc.hist[(r, l)][tag[r][occ]]), (r, l)
            if sc.appends:
                n = sc.steps
                assert np.array_equal(pool.read_history(r, l, sc.ctx0, n), sc.hist[(r, l)][sc.ctx0:sc.ctx0 + n])
    pool.close()
    return worst


def test_tiny_single_request_mla():
    """1 request, 1 layer, 4096-token context, 576-dim latent, 16 heads, k=256, B=512, LRU,
    64 steps with write-through append; drift keep 90%, recency mean 512."""
    sc = Scenario(_mla(1, 1, 4096 + 64, 256, 512, log=64), ctx0=4096, steps=64, appends=True, keep=0.9,
                  recency_mean=512, seed=1)
    run_and_compare(sc)


@pytest.mark.parametrize("fetch", [0, 1, 2])
@pytest.mark.parametrize("policy", [0, 1, 2, 3])
def test_gqa_policies_ragged(policy, fetch):
    """3 requests x 2 layers, k=300 (not a multiple of the stage), B=640, every policy; misses
    copied by the resolve (fetch=0), by the attention while it gathers (fetch=1), or by the resolve
    with fetch CTAs that start before the decision ends (fetch=2)."""
    B = 300 if policy == 3 else 640
    sc = Scenario(_gqa(3, 2, 3000 + 12, 300, B, policy=policy, fetch=fetch), ctx0=3000, steps=12, appends=True,
                  keep=0.8, recency_mean=200, seed=policy + 1)
    run_and_compare(sc)


@pytest.mark.parametrize("fetch", [0, 1, 2])
@pytest.mark.parametrize("policy", [0, 1, 2, 3])
def test_fused_append_resolve(policy, fetch):
    """hs_append_resolve equals append then resolve: same slots, state, counters and outputs as
    the oracle, for every policy (swap-vanilla empties the appended slot when it is unselected)."""
    B = 300 if policy == 3 else 640
    sc = Scenario(_gqa(3, 2, 3000 + 12, 300, B, policy=policy, fetch=fetch), ctx0=3000, steps=12, appends=True,
                  keep=0.8, recency_mean=200, seed=policy + 41)
    run_and_compare(sc, fused=True)
    # the appended position is not always selected: drop it from some lists (replaced by padding)
    sc = Scenario(_gqa(2, 1, 800 + 10, 64, 96, policy=policy, fetch=fetch), ctx0=800, steps=10, appends=True,
                  keep=0.7, recency_mean=50, seed=policy + 51)
    for t in range(0, 10, 2):
        sc.trace[t, 0, 0][sc.trace[t, 0, 0] == 800 + t] = -1
    run_and_compare(sc, fused=True)
    if policy == 0 and fetch != 1:
        sc = Scenario(_mla(1, 1, 4096 + 16, 256, 512, early=int(fetch == 2)), ctx0=4096, steps=16, appends=True,
                      keep=0.9, recency_mean=512, seed=3)
        run_and_compare(sc, fused=True)


@pytest.mark.parametrize("layout", ["gqa", "gqa_fetch", "gqa_early", "mla"])
def test_request_ranges_on_two_streams(layout):
    """Two micro-batches of one pool on two streams, each request's layers in order: slots, state
    and counters equal the oracle's, outputs are within the attention tolerance of its fp64
    attention, and everything is bit-identical to full-batch calls on a second pool."""
    if layout == "mla":
        cfg = _mla(4, 2, 3000 + 6, 256, 512, Hq=64)
    else:
        cfg = _gqa(4, 2, 3000 + 6, 256, 512, fetch={"gqa": 0, "gqa_fetch": 1, "gqa_early": 2}[layout])
    sc = Scenario(cfg, ctx0=3000, steps=6, appends=True, seed=61)
    full, split = HsPool(cfg), HsPool(cfg)
    prefill(full, sc)
    prefill(split, sc)
    orc = OracleRun(sc)
    R, L = cfg.num_requests, cfg.num_layers
    groups = [(0, 1), (1, 3)]  # uneven on purpose
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for t in range(sc.steps):
        ref = gpu_step(full, sc, t, fused=True)
        oref = orc.step(t)
        outs = []
        torch.cuda.synchronize()
        for (r0, n), st in zip(groups, streams):
            with torch.cuda.stream(st):
                per_layer = []
                for l in range(L):
                    topk = torch.from_numpy(sc.trace[t, l, r0:r0 + n]).cuda()
                    pos = torch.full((n,), sc.ctx0 + t, dtype=torch.int64, device="cuda")
                    rec = bf16_tensor(np.stack([sc.hist[(r, l)][sc.ctx0 + t] for r in range(r0, r0 + n)]), "cuda")
                    q = bf16_tensor(sc.q[t, l, r0:r0 + n], "cuda")
                    locs = split.resolve_range(l, r0, topk, pos=pos, rec=rec, stream=st)
                    out = split.sparse_attn_range(l, r0, q, locs, scale=sc.scale, stream=st)
                    per_layer.append((locs, out, topk, pos, rec, q))
                outs.append(per_layer)
        torch.cuda.synchronize()
        for l in range(L):
            got_locs = np.concatenate([outs[gi][l][0].cpu().numpy() for gi in range(len(groups))])
            got_out = np.concatenate([outs[gi][l][1].cpu().numpy() for gi in range(len(groups))])
            assert_layer_matches_oracle(sc, orc, oref, t, l, got_locs, got_out, "request ranges")
            assert np.array_equal(got_locs, ref[l][0]), (t, l)
            assert np.array_equal(got_out, ref[l][1]), (t, l)
    assert_pool_matches_oracle(split, orc, "request ranges")
    for l in range(L):
        a, b = full.read_state(l), split.read_state(l)
        assert all(np.array_equal(x, y) for x, y in zip(a, b))
    assert np.array_equal(full.stats()["per_rl"], split.stats()["per_rl"])
    full.close()
    split.close()


@pytest.mark.parametrize("fetch", [0, 1, 2])
def test_layer_group_schedule_on_side_streams(fetch):
    """Layer groups sharing one selection (exact layer-group prefetch): the group's resolves run at
    once, each layer on its own stream, and the attentions follow on another stream as their
    resolve completes.  Slots, state and counters equal the oracle's stepped beside it, outputs are
    within the attention tolerance of its fp64 attention, and everything is bit-identical to the
    plain layer-by-layer schedule on a second pool."""
    cfg = _gqa(4, 4, 3000 + 6, 256, 512, fetch=fetch)
    sc = Scenario(cfg, ctx0=3000, steps=6, appends=True, seed=67)
    G = 2
    for l in range(cfg.num_layers):
        sc.trace[:, l] = sc.trace[:, G * (l // G)]
    seq, grp = HsPool(cfg), HsPool(cfg)
    prefill(seq, sc)
    prefill(grp, sc)
    orc = OracleRun(sc)
    R, L = cfg.num_requests, cfg.num_layers
    side = [torch.cuda.Stream() for _ in range(G)]
    astream = torch.cuda.Stream()
    for t in range(sc.steps):
        ref = gpu_step(seq, sc, t, fused=True)
        torch.cuda.synchronize()
        ins = []
        for l in range(L):
            ins.append((torch.from_numpy(sc.trace[t, l]).cuda(),
                        torch.full((R,), sc.ctx0 + t, dtype=torch.int64, device="cuda"),
                        bf16_tensor(np.stack([sc.hist[(r, l)][sc.ctx0 + t] for r in range(R)]), "cuda"),
                        bf16_tensor(sc.q[t, l], "cuda")))
        torch.cuda.synchronize()
        locs = [torch.empty((R, cfg.top_k), dtype=torch.int32, device="cuda") for _ in range(L)]
        outs = [None] * L
        for l0 in range(0, L, G):
            known = torch.cuda.Event()
            known.record(astream)
            done = []
            for j, l in enumerate(range(l0, l0 + G)):
                side[j].wait_event(known)
                topk, pos, rec, _ = ins[l]
                grp.append_resolve(l, pos, rec, topk, locs[l], stream=side[j])
                e = torch.cuda.Event()
                e.record(side[j])
                done.append(e)
            for j, l in enumerate(range(l0, l0 + G)):
                astream.wait_event(done[j])
                with torch.cuda.stream(astream):
                    outs[l] = grp.sparse_attn(l, ins[l][3], locs[l], scale=sc.scale, stream=astream)
        torch.cuda.synchronize()
        oref = orc.step(t)
        for l in range(L):
            got_locs, got_out = locs[l].cpu().numpy(), outs[l].cpu().numpy()
            assert_layer_matches_oracle(sc, orc, oref, t, l, got_locs, got_out, "layer groups")
            assert np.array_equal(got_locs, ref[l][0]), (t, l)
            assert np.array_equal(got_out, ref[l][1]), (t, l)
    assert_pool_matches_oracle(grp, orc, "layer groups")
    for l in range(L):
        a, b = seq.read_state(l), grp.read_state(l)
        assert all(np.array_equal(x, y) for x, y in zip(a, b))
    assert np.array_equal(seq.stats()["per_rl"], grp.stats()["per_rl"])
    seq.close()
    grp.close()


@pytest.mark.parametrize("fetch", [0, 1, 2])
def test_chained_microbatches_in_one_graph(fetch):
    """The bench's two-micro-batch schedule: each half on its own stream, the halves' resolves in one
    chain and their attentions in another, every step captured in one CUDA graph.  Slots, state and
    counters equal the oracle's, outputs are within the attention tolerance of its fp64 attention,
    and everything is bit-identical to full-batch calls on a second pool."""
    R, L, steps = 4, 3, 6
    cfg = _gqa(R, L, 3000 + steps, 256, 512, fetch=fetch)
    sc = Scenario(cfg, ctx0=3000, steps=steps, appends=True, seed=67)
    full, split = HsPool(cfg), HsPool(cfg)
    prefill(full, sc)
    prefill(split, sc)
    refs = [gpu_step(full, sc, t, fused=True) for t in range(steps)]
    dev = "cuda"
    topk = torch.from_numpy(sc.trace).to(dev)                                     # [S][L][R][k]
    q = bf16_tensor(sc.q, dev)                                                     # [S][L][R][Hq][D]
    rec = bf16_tensor(np.stack([np.stack([np.stack([sc.hist[(r, l)][sc.ctx0 + t] for r in range(R)])
                                          for l in range(L)]) for t in range(steps)]), dev)
    pos = (torch.arange(steps, dtype=torch.int64, device=dev) + sc.ctx0).view(steps, 1).expand(steps, R).contiguous()
    locs = torch.empty((steps, L, R, cfg.top_k), dtype=torch.int32, device=dev)
    outs = torch.empty((steps, L, R, cfg.num_q_heads, cfg.head_dim_v), dtype=torch.float32, device=dev)
    groups = [(0, 2), (2, 2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cur = torch.cuda.current_stream()
        ev = torch.cuda.Event()
        ev.record(cur)
        for st in streams:
            st.wait_event(ev)
        last_res = last_att = None
        for t in range(steps):
            for l in range(L):
                for (r0, n), st in zip(groups, streams):
                    with torch.cuda.stream(st):
                        if last_res is not None:
                            st.wait_event(last_res)
                        split.resolve_range(l, r0, topk[t, l, r0:r0 + n], locs[t, l, r0:r0 + n],
                                            pos=pos[t, r0:r0 + n], rec=rec[t, l, r0:r0 + n], stream=st)
                        last_res = torch.cuda.Event()
                        last_res.record(st)
                        if last_att is not None:
                            st.wait_event(last_att)
                        split.sparse_attn_range(l, r0, q[t, l, r0:r0 + n], locs[t, l, r0:r0 + n],
                                                outs[t, l, r0:r0 + n], scale=sc.scale, stream=st)
                        last_att = torch.cuda.Event()
                        last_att.record(st)
        for st in streams:
            ev = torch.cuda.Event()
            ev.record(st)
            cur.wait_event(ev)
    graph.replay()
    torch.cuda.synchronize()
    orc = OracleRun(sc)
    for t in range(steps):
        oref = orc.step(t)
        for l in range(L):
            got_locs, got_out = locs[t, l].cpu().numpy(), outs[t, l].cpu().numpy()
            assert_layer_matches_oracle(sc, orc, oref, t, l, got_locs, got_out, "micro-batches")
            assert np.array_equal(got_locs, refs[t][l][0]), (t, l)
            assert np.array_equal(got_out, refs[t][l][1]), (t, l)
    assert_pool_matches_oracle(split, orc, "micro-batches")
    for l in range(L):
        a, b = full.read_state(l), split.read_state(l)
        assert all(np.array_equal(x, y) for x, y in zip(a, b))
    sf, ss = full.stats(), split.stats()
    assert np.array_equal(sf["per_rl"], ss["per_rl"])
    assert ss["error_bits"] == 0
    full.close()
    split.close()


def test_range_arguments_checked():
    cfg = _gqa(2, 1, 100, 4, 8, kvh=1)
    pool = HsPool(cfg)
    from hierarchical_kv_cache_02_gb300 import HsError
    topk = torch.zeros((2, 4), dtype=torch.int32, device="cuda")
    with pytest.raises(HsError):
        pool.resolve_range(0, 1, topk)  # requests 1..2 of a 2-request pool
    pool.close()


@pytest.mark.parametrize("attn_every", [2, 3])
def test_fetch_in_attention_with_skipped_attention(attn_every):
    """Steps without attention leave copies pending; the next append (or resolve) finishes them,
    so state, slots, buffer contents and later attention still match the oracle."""
    steps = 3 * attn_every + 1  # the last step runs attention, so the final buffer check sees every row
    sc = Scenario(_gqa(2, 2, 2500 + steps, 256, 512, fetch=1), ctx0=2500, steps=steps, appends=True, seed=31)
    run_and_compare(sc, attn_every=attn_every)
    sc = Scenario(_gqa(2, 1, 2500, 256, 512, fetch=1), ctx0=2500, steps=steps, appends=False, seed=32)
    run_and_compare(sc, attn_every=attn_every)


@pytest.mark.parametrize("policy", [0, 2])
def test_mla_64_heads_no_append(policy):
    sc = Scenario(_mla(2, 1, 6000, 512, 1024, Hq=64, policy=policy), ctx0=6000, steps=8, appends=False, keep=0.85,
                  recency_mean=600, seed=5)
    run_and_compare(sc)


@pytest.mark.parametrize("R,k", [(2, 2048), (3, 1024)])
def test_mla_64_heads_long_selections(R, k):
    """Few requests with long selections: 32 (R = 2) or 16 (R = 3) splits of 64 tokens per request
    (one-tile splits: the value blocks stay in place from the score pass), merged by the split
    combine."""
    sc = Scenario(_mla(R, 1, 6000 + 6, k, 2 * k, Hq=64), ctx0=6000, steps=6, appends=True, keep=0.85,
                  recency_mean=800, seed=17)
    run_and_compare(sc, fused=True)


def test_mla_64_heads_multi_tile_splits():
    """Many requests: on 152 SMs, 3 splits per request of 352, 352 and 320 tokens, i.e. three 128-token tiles
    each (the last one ragged), so the score pass of a tile runs while the previous tile's value
    blocks are re-read, and the running max and sums carry across tiles."""
    sc = Scenario(_mla(40, 1, 3000 + 4, 1024, 2048, Hq=64), ctx0=3000, steps=4, appends=True, keep=0.85,
                  recency_mean=400, seed=23)
    run_and_compare(sc, fused=True)


@pytest.mark.parametrize("io", [16, 32, 128])
def test_io_chunk_sizes(io):
    sc = Scenario(_gqa(2, 1, 2000 + 6, 128, 256, kvh=2, G=4, io=io), ctx0=2000, steps=6, appends=True, seed=9)
    run_and_compare(sc)
    sc = Scenario(_gqa(2, 1, 2000 + 6, 128, 256, kvh=2, G=4, io=io, fetch=2), ctx0=2000, steps=6, appends=True, seed=9)
    run_and_compare(sc)


@pytest.mark.parametrize("G", [1, 2, 8])
def test_gqa_group_sizes(G):
    sc = Scenario(_gqa(2, 1, 1500, 96, 200, kvh=4, G=G), ctx0=1500, steps=5, appends=False, seed=G)
    run_and_compare(sc)


@pytest.mark.parametrize("fetch", [0, 1, 2])
def test_shared_prefix_history(fetch):
    """Requests share one prefilled history (read-only); appended tokens are private."""
    sc = Scenario(_gqa(3, 2, 2500 + 8, 200, 400, P0=2500, fetch=fetch), ctx0=2500, steps=8, appends=True, seed=21)
    run_and_compare(sc)


def test_buffer_as_large_as_context_no_misses_after_warmup():
    cfg = _gqa(1, 1, 300, 64, 320, kvh=2, log=20)
    sc = Scenario(cfg, ctx0=300, steps=20, appends=False, keep=0.7, recency_mean=50, seed=4)
    run_and_compare(sc)


@pytest.mark.parametrize("fetch", [0, 1, 2])
def test_small_k_and_b_equal_k(fetch):
    for policy in (0, 3):
        sc = Scenario(_gqa(2, 1, 500, 1, 1, kvh=1, G=4, policy=policy, fetch=fetch), ctx0=500, steps=10,
                      appends=False, seed=7)
        run_and_compare(sc)
        sc = Scenario(_gqa(2, 1, 500, 5, 5, kvh=1, G=4, policy=policy, fetch=fetch), ctx0=500, steps=10,
                      appends=False, seed=8)
        run_and_compare(sc)


@pytest.mark.parametrize("fetch", [0, 2])
@pytest.mark.parametrize("policy", [0, 3])
def test_repeats_of_resident_missing_and_appended_positions(policy, fetch):
    """A repeated position counts at its first occurrence only, whether the position is resident (a
    hit), missing, or the token the fused append has just written."""
    cfg = _gqa(2, 1, 600 + 8, 64, 128, policy=policy, kvh=2, fetch=fetch)
    sc = Scenario(cfg, ctx0=600, steps=5, appends=True, seed=21)
    tr = sc.trace.copy()
    prev = set(tr[1, 0, 0].tolist())                   # resident after step 1 (B = 128 >= 2 k)
    e = next(i for i in range(7) if int(tr[2, 0, 0, i]) in prev)
    tr[2, 0, 0, 7] = tr[2, 0, 0, e]                    # a resident position, repeated
    seen = set(tr[:3, 0, 1].ravel().tolist())
    fresh = next(p for p in range(600) if p not in seen)
    tr[2, 0, 1, 10] = fresh                            # missing, and repeated
    tr[2, 0, 1, 11] = fresh
    tr[3, 0, 0, 1] = 600 + 3                           # the token appended this step, twice
    tr[3, 0, 0, 2] = 600 + 3
    sc.trace = tr
    pool = HsPool(cfg)
    prefill(pool, sc)
    orc = OracleRun(sc)
    for t in range(sc.steps):
        res = gpu_step(pool, sc, t, fused=True)
        ref = orc.step(t)
        for r in range(2):
            assert np.array_equal(res[0][0][r], ref[(r, 0)][1]), (t, r)
            assert_attn_close(res[0][1][r], orc.attention(t, r, 0), (t, r))
    tag, stamp, clock = pool.read_state(0)
    for r in range(2):
        otag, ostamp = orc.caches[(r, 0)].slots()
        assert np.array_equal(tag[r], otag) and np.array_equal(stamp[r], ostamp)
    st = pool.stats()
    assert (st["errors"][:, 0] == DEVERR_DUP).all()
    assert [orc.caches[(r, 0)].counters()["err"] for r in range(2)] == [DEVERR_DUP, DEVERR_DUP]
    assert np.array_equal(st["per_rl"][:, 0, :3], np.array([[orc.caches[(r, 0)].counters()[x] for x in
                                                             ("hits", "misses", "appends")] for r in range(2)]))
    pool.close()


@pytest.mark.parametrize("fetch", [0, 2])
def test_padding_duplicates_and_out_of_range(fetch):
    """Invalid entries are skipped like padding, flagged, and attention ignores them."""
    cfg = _gqa(2, 1, 400, 16, 32, kvh=2, fetch=fetch)
    sc = Scenario(cfg, ctx0=400, steps=3, appends=False, seed=12)
    bad = sc.trace.copy()
    bad[1, 0, 0, 3] = -1
    bad[1, 0, 0, 5] = bad[1, 0, 0, 4]          # duplicate of an earlier entry
    bad[2, 0, 1, 0] = 400                      # out of range
    bad[2, 0, 1, 1] = -7                       # negative, not padding
    sc.trace = bad
    pool = HsPool(cfg)
    prefill(pool, sc)
    orc = OracleRun(sc)
    for t in range(3):
        res = gpu_step(pool, sc, t)
        ref = orc.step(t)
        for r in range(2):
            assert np.array_equal(res[0][0][r], ref[(r, 0)][1])
            assert_attn_close(res[0][1][r], orc.attention(t, r, 0))
    st = pool.stats()
    assert st["status"] == -6
    assert st["errors"][0, 0] == DEVERR_DUP and st["errors"][1, 0] == DEVERR_RANGE
    assert orc.caches[(0, 0)].counters()["err"] == DEVERR_DUP
    pool.stats(reset=True)
    assert pool.stats()["error_bits"] == 0
    pool.close()


def test_append_out_of_range_flags():
    cfg = _gqa(2, 1, 100, 4, 8, kvh=1, P0=50)
    pool = HsPool(cfg)
    pos = torch.tensor([10, 100], dtype=torch.int64, device="cuda")  # below the shared prefix / past capacity
    rec = torch.zeros((2, cfg.record_elems), dtype=torch.bfloat16, device="cuda")
    pool.append(0, pos, rec)
    st = pool.stats()
    assert list(st["errors"][:, 0]) == [DEVERR_APPEND, DEVERR_APPEND] and st["appends"] == 0
    pool.close()


def test_exactness_cold_warm_resident_bit_identical():
    """Summary §3: the output over the hot buffer equals the output over fully resident KV,
    bit for bit, whatever the cache held before."""
    for cfg in (_gqa(3, 1, 5000, 512, 1024), _gqa(3, 1, 5000, 512, 1024, fetch=1),
                _gqa(3, 1, 5000, 512, 1024, fetch=2), _mla(2, 1, 5000, 512, 1024, Hq=32),
                _mla(2, 1, 5000, 512, 1024, Hq=64)):  # 64 heads: the tcgen05 kernel, hot slots vs resident rows
        sc = Scenario(cfg, ctx0=5000, steps=10, appends=False, keep=0.85, recency_mean=300, seed=2)
        warm = HsPool(cfg)
        prefill(warm, sc)
        for t in range(9):
            gpu_step(warm, sc, t, attn=False)
        out_warm = gpu_step(warm, sc, 9)[0][1]
        cold = HsPool(cfg)
        prefill(cold, sc)
        out_cold = gpu_step(cold, sc, 9)[0][1]
        kv = torch.stack([bf16_tensor(sc.hist[(r, 0)]) for r in range(cfg.num_requests)]).cuda()
        q = bf16_tensor(sc.q[9, 0], "cuda")
        locs = torch.from_numpy(sc.trace[9, 0]).cuda()
        out_res = warm.sparse_attn(0, q, locs, scale=sc.scale, kv=kv).cpu().numpy()
        assert warm.stats()["hits"] > 0  # the warm pool served hits
        assert np.array_equal(out_warm, out_cold)
        assert np.array_equal(out_warm, out_res)
        orc = OracleRun(sc)
        for r in range(cfg.num_requests):
            assert_attn_close(out_res[r], orc.attention(9, r, 0), tight=cfg.layout == LAYOUT_GQA)
        warm.close()
        cold.close()


def test_resident_kv_bad_rows_flagged():
    cfg = _gqa(1, 1, 64, 8, 16, kvh=1)
    pool = HsPool(cfg)
    kv = torch.zeros((1, 10, cfg.record_elems), dtype=torch.bfloat16, device="cuda")
    locs = torch.tensor([[0, 1, 2, 10, -1, 3, 4, 5]], dtype=torch.int32, device="cuda")
    q = torch.zeros((1, 4, 128), dtype=torch.bfloat16, device="cuda")
    out = pool.sparse_attn(0, q, locs, kv=kv)
    torch.cuda.synchronize()
    assert pool.stats()["error_bits"] == DEVERR_LOC
    assert torch.count_nonzero(out) == 0
    pool.close()


@pytest.mark.parametrize("fetch", [0, 1, 2])
def test_cuda_graph_replay_matches_eager(fetch):
    """All calls are capturable: one decode step (append, resolve, attention for every layer)
    captured once and replayed gives the eager results bit for bit."""
    cfg = _gqa(2, 2, 3000 + 6, 256, 512, fetch=fetch)
    sc = Scenario(cfg, ctx0=3000, steps=6, appends=True, seed=14)
    eager = HsPool(cfg)
    prefill(eager, sc)
    graphed = HsPool(cfg)
    prefill(graphed, sc)
    R, L = cfg.num_requests, cfg.num_layers
    s_pos = torch.zeros((R,), dtype=torch.int64, device="cuda")
    s_rec = [torch.zeros((R, cfg.record_elems), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    s_topk = [torch.zeros((R, cfg.top_k), dtype=torch.int32, device="cuda") for _ in range(L)]
    s_q = [torch.zeros((R, cfg.num_q_heads, 128), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    s_locs = [torch.zeros((R, cfg.top_k), dtype=torch.int32, device="cuda") for _ in range(L)]
    s_out = [torch.zeros((R, cfg.num_q_heads, 128), dtype=torch.float32, device="cuda") for _ in range(L)]
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for l in range(L):
                graphed.append(l, s_pos, s_rec[l], stream=stream)
                graphed.resolve(l, s_topk[l], s_locs[l], stream=stream)
                graphed.sparse_attn(l, s_q[l], s_locs[l], s_out[l], scale=sc.scale, stream=stream)
    graphed.reset()  # capture does not execute; start both pools cold
    torch.cuda.synchronize()
    for t in range(sc.steps):
        s_pos.fill_(sc.ctx0 + t)
        for l in range(L):
            s_rec[l].copy_(bf16_tensor(np.stack([sc.hist[(r, l)][sc.ctx0 + t] for r in range(R)])))
            s_topk[l].copy_(torch.from_numpy(sc.trace[t, l]))
            s_q[l].copy_(bf16_tensor(sc.q[t, l]))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        ref = gpu_step(eager, sc, t)
        for l in range(L):
            assert np.array_equal(s_locs[l].cpu().numpy(), ref[l][0])
            assert np.array_equal(s_out[l].cpu().numpy(), ref[l][1])
    for l in range(L):
        a, b = eager.read_state(l), graphed.read_state(l)
        assert all(np.array_equal(x, y) for x, y in zip(a, b))
    eager.close()
    graphed.close()


def test_fault_injection_allocations(monkeypatch):
    cfg = _gqa(1, 1, 64, 8, 16, kvh=1)
    from hierarchical_kv_cache_02_gb300 import HsError

    for what, code in (("alloc_host", -2), ("alloc_dev", -3)):
        monkeypatch.setenv("HS_FAULT", what)
        with pytest.raises(HsError) as e:
            HsPool(cfg)
        assert e.value.status == code
    monkeypatch.delenv("HS_FAULT")
    HsPool(cfg).close()


def test_pools_of_different_configurations_share_the_kernels():
    """A kernel's dynamic shared-memory limit is one attribute per process, not per pool: pools of
    different configurations (staging area or not, fetch CTAs, 64-head selections of different
    lengths) created one after another all keep launching, and each matches the oracle."""
    cfgs = [_gqa(2, 1, 2000 + 4, 256, 512), _gqa(2, 1, 2000 + 4, 256, 512, fetch=2),
            _gqa(2, 1, 2000 + 4, 256, 512, fetch=1), _mla(2, 1, 2000 + 4, 512, 1024, Hq=64),
            _mla(2, 1, 2000 + 4, 128, 256, Hq=64, early=1)]
    scs = [Scenario(c, ctx0=2000, steps=4, appends=True, seed=71 + i) for i, c in enumerate(cfgs)]
    pools = [HsPool(c) for c in cfgs]
    for pool, sc in zip(pools, scs):
        prefill(pool, sc)
    orcs = [OracleRun(sc) for sc in scs]
    for t in range(4):
        for pool, sc, orc in zip(pools, scs, orcs):
            res = gpu_step(pool, sc, t, fused=True)
            ref = orc.step(t)
            for l in range(sc.cfg.num_layers):
                assert_layer_matches_oracle(sc, orc, ref, t, l, res[l][0], res[l][1], "pools side by side")
    for pool, orc in zip(pools, orcs):
        assert_pool_matches_oracle(pool, orc, "pools side by side")
        pool.close()


def test_select_beyond_the_bitmap_window():
    """The one-pass victim select covers a window of 131072 keys below the largest; older candidate
    keys send it back to the radix select.  One request, k = 2048 in B = 4096 slots, one new position
    per step and no appends: half the buffer stays empty while the clock passes 131072, and from about
    step 66 on the candidates include positions dropped at the start, whose stamps lie below the
    window (checked on the oracle's state before each step).  Slots, stamps, counters and the last
    step's attention equal the oracle's."""
    k, B, ctx0, steps = 2048, 4096, 20000, 80
    cfg = _gqa(1, 1, ctx0, k, B, kvh=1, G=4)  # LRU: a hit is restamped, so the clock runs ahead
    sc = Scenario(cfg, ctx0=ctx0, steps=steps, appends=False, seed=77)
    rng = np.random.default_rng(77)
    order = rng.permutation(ctx0)
    cur, nxt = [int(x) for x in order[:k]], k
    trace = np.empty((steps, 1, 1, k), dtype=np.int32)
    for t in range(steps):
        if t > 0:  # one selected position replaced by one never selected before: one miss
            cur[int(rng.integers(k))] = int(order[nxt])
            nxt += 1
        trace[t, 0, 0] = cur
    sc.trace = trace
    pool = HsPool(cfg)
    prefill(pool, sc)
    orc = OracleRun(sc)
    beyond = 0
    for t in range(steps):
        tag, stamp = orc.caches[(0, 0)].slots()
        chosen = set(trace[t, 0, 0].tolist())
        keys = [int(s) for tg, s in zip(tag.tolist(), stamp.tolist()) if tg not in chosen]
        nz = [x for x in keys if x != 0]
        if nz and 0 in keys:
            beyond += any(x < max(nz) - 131071 for x in nz)
        elif nz:
            beyond += max(nz) - min(nz) >= 131072
        res = gpu_step(pool, sc, t, attn=(t == steps - 1))
        ref = orc.step(t)
        m, locs = ref[(0, 0)]
        assert np.array_equal(res[0][0][0], locs), t
    assert beyond > 0  # the scenario did reach keys outside the window
    assert_attn_close(res[0][1][0], orc.attention(steps - 1, 0, 0), tight=True)
    assert_pool_matches_oracle(pool, orc, "select window")
    pool.close()
