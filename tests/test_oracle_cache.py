"""Pins of the oracle's cache simulation against things other than itself.

Each test checks a fact that the HiSparse summary (§3-§5) or plain reasoning
fixes, so that a slip in the oracle (a dropped term, a wrong tie-break, an
off-by-one in the stamps) fails at least one of them:
  * hand-worked examples (tests/golden/cache_worked_examples.json);
  * list-based restatements of LRU and FIFO (a recency list / insertion queue
    instead of stamps) agree on the resident set and the eviction order;
  * hits + misses = k; B >= context => no misses after warm-up;
  * B = k: swap-vanilla and LRU misses = |S_t minus S_{t-1}|;
  * Belady equals the exhaustive minimum on tiny traces, and lower-bounds LRU,
    FIFO, random and swap-vanilla;
  * the random policy's key is splitmix64 at the stated counter;
  * a buffer grown on demand (slots [0, cap) only) is the recency list / queue of
    cap entries, equals the full buffer while its growth stays ahead of the
    context, and refuses a step with fewer than k slots.
"""
import itertools
import json
import os
from functools import lru_cache

import numpy as np
import pytest

import oracle
from hierarchical_kv_cache_02_gb300 import inputs


def _load_examples(golden_dir):
    with open(os.path.join(golden_dir, "cache_worked_examples.json")) as f:
        return json.load(f)["examples"]


def test_worked_examples(golden_dir):
    for ex in _load_examples(golden_dir):
        c = oracle.Cache(ex["B"], ex["k"], ex["policy"], C=ex["C"])
        for op in ex["ops"]:
            if "resolve" in op:
                m, locs = c.resolve(op["resolve"])
                assert m == op["misses"], (ex["name"], op)
                assert locs.tolist() == op["locs"], (ex["name"], op)
            else:
                assert c.append(op["append"]) == op["slot"], (ex["name"], op)
            tag, stamp = c.slots()
            assert tag.tolist() == op["tag"], (ex["name"], op)
            assert stamp.tolist() == op["stamp"], (ex["name"], op)
            assert c.counters()["clock"] == op["clock"], (ex["name"], op)
        cnt = c.counters()
        for key, val in ex["totals"].items():
            assert cnt[key] == val, (ex["name"], key)


def _random_trace(rng, T, k, npos):
    return np.stack([rng.choice(npos, size=k, replace=False) for _ in range(T)]).astype(np.int32)


def _lru_list_model(B, trace):
    """Recency list, oldest first.  Per step: hits move to the MRU end in top-k order,
    then each miss evicts (if the buffer is full) the oldest entry not selected this step
    and is appended at the MRU end in top-k order."""
    order, out = [], []
    for S in trace:
        Sset = set(int(x) for x in S)
        resident = set(order)
        hits = [int(s) for s in S if int(s) in resident]
        miss = [int(s) for s in S if int(s) not in resident]
        stale = [p for p in order if p not in Sset]
        free = B - len(order)
        n_evict = max(0, len(miss) - free)
        evicted = set(stale[:n_evict])
        order = [p for p in order if p not in evicted and p not in Sset] + hits + miss
        out.append((len(miss), list(order)))
    return out


def _fifo_queue_model(B, trace):
    """Insertion queue, oldest first; hits do not move; misses evict the oldest unselected entry."""
    queue, out = [], []
    for S in trace:
        Sset = set(int(x) for x in S)
        resident = set(queue)
        miss = [int(s) for s in S if int(s) not in resident]
        stale = [p for p in queue if p not in Sset]
        n_evict = max(0, len(miss) - (B - len(queue)))
        evicted = set(stale[:n_evict])
        queue = [p for p in queue if p not in evicted] + miss
        out.append((len(miss), list(queue)))
    return out


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("B,k,npos", [(4, 2, 8), (6, 3, 10), (8, 3, 20), (16, 5, 40)])
def test_lru_matches_recency_list(seed, B, k, npos):
    rng = np.random.default_rng(seed)
    trace = _random_trace(rng, 30, k, npos)
    c = oracle.Cache(B, k, "lru", C=npos)
    for S, (m_ref, order) in zip(trace, _lru_list_model(B, trace)):
        m, locs = c.resolve(S)
        assert m == m_ref
        tag, stamp = c.slots()
        assert (tag[locs] == S).all()
        occ = tag >= 0
        by_stamp = [int(t) for _, t in sorted(zip(stamp[occ].tolist(), tag[occ].tolist()))]
        assert by_stamp == order


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("B,k,npos", [(4, 2, 8), (6, 3, 10), (16, 5, 40)])
def test_fifo_matches_insertion_queue(seed, B, k, npos):
    rng = np.random.default_rng(100 + seed)
    trace = _random_trace(rng, 30, k, npos)
    c = oracle.Cache(B, k, "fifo", C=npos)
    for S, (m_ref, queue) in zip(trace, _fifo_queue_model(B, trace)):
        m, _ = c.resolve(S)
        assert m == m_ref
        tag, stamp = c.slots()
        occ = tag >= 0
        by_stamp = [int(t) for _, t in sorted(zip(stamp[occ].tolist(), tag[occ].tolist()))]
        assert by_stamp == queue


@pytest.mark.parametrize("policy", ["lru", "fifo", "random", "swap"])
def test_hits_plus_misses_is_k_and_locs_point_at_tags(policy):
    spec = inputs.TraceSpec(ctx0=300, k=32, steps=40, keep=0.8, recency_mean=40, appends=True)
    tr = inputs.drift_traces(spec, 1, 1, seed=11)[:, 0, 0]
    c = oracle.Cache(64, 32, policy, seed=5, C=300 + 40)
    prev = c.counters()
    for t, S in enumerate(tr):
        c.append(300 + t)
        m, locs = c.resolve(S)
        cnt = c.counters()
        assert (cnt["hits"] - prev["hits"]) + (cnt["misses"] - prev["misses"]) == 32
        assert cnt["misses"] - prev["misses"] == m
        tag, stamp = c.slots()
        assert (tag[locs] == S).all()
        assert len(set(tag[tag >= 0].tolist())) == int((tag >= 0).sum())  # no position twice
        assert ((tag < 0) == (stamp == 0)).all()                          # empty <=> stamp 0
        prev = cnt
    assert cnt["clock"] == 1 + 40 * 32 + 40
    assert cnt["appends"] == 40 and cnt["err"] == 0


@pytest.mark.parametrize("policy", ["lru", "fifo", "random", "swap"])
def test_buffer_larger_than_context_has_no_misses_after_warmup(policy):
    npos, k = 24, 6
    rng = np.random.default_rng(3)
    trace = _random_trace(rng, 50, k, npos)
    c = oracle.Cache(npos, k, policy, seed=9, C=npos)
    seen = set()
    for S in trace:
        m, _ = c.resolve(S)
        new = set(S.tolist()) - seen
        if policy == "swap":
            continue
        assert m == len(new)  # only compulsory misses
        seen |= new


@pytest.mark.parametrize("policy", ["swap", "lru"])
def test_b_equals_k_misses_are_set_difference(policy):
    rng = np.random.default_rng(21)
    trace = _random_trace(rng, 40, 5, 12)
    c = oracle.Cache(5, 5, policy, C=12)
    prev = set()
    for S in trace:
        m, _ = c.resolve(S)
        cur = set(S.tolist())
        assert m == len(cur - prev)
        prev = cur


def test_swap_vanilla_keeps_only_current_topk():
    rng = np.random.default_rng(8)
    trace = _random_trace(rng, 30, 4, 30)
    c = oracle.Cache(10, 4, "swap", C=30)
    for S in trace:
        c.resolve(S)
        tag, stamp = c.slots()
        assert sorted(tag[tag >= 0].tolist()) == sorted(S.tolist())


def _exhaustive_min_misses(B, trace):
    """Minimum total misses over every choice of victims, by dynamic programming over resident sets."""
    trace = [tuple(int(x) for x in S) for S in trace]

    @lru_cache(maxsize=None)
    def best(t, resident):
        if t == len(trace):
            return 0
        S = trace[t]
        res = set(resident)
        miss = [s for s in S if s not in res]
        m = len(miss)
        evictable = sorted(p for p in res if p not in S)
        empties = B - len(res)
        out = None
        for n_empty in range(min(m, empties) + 1):
            n_ev = m - n_empty
            if n_ev > len(evictable):
                continue
            for ev in itertools.combinations(evictable, n_ev):
                nxt = frozenset((res - set(ev)) | set(miss))
                v = m + best(t + 1, nxt)
                out = v if out is None else min(out, v)
        return out

    return best(0, frozenset())


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("B,k,npos,T", [(3, 2, 6, 8), (4, 2, 7, 8), (5, 3, 9, 7), (6, 3, 10, 6)])
def test_belady_is_the_exhaustive_minimum(seed, B, k, npos, T):
    rng = np.random.default_rng(1000 * B + seed)
    trace = _random_trace(rng, T, k, npos)
    assert int(oracle.belady(B, trace, npos).sum()) == _exhaustive_min_misses(B, trace)


@pytest.mark.parametrize("seed", range(4))
def test_belady_lower_bounds_online_policies(seed):
    spec = inputs.TraceSpec(ctx0=2000, k=64, steps=60, keep=0.85, recency_mean=128)
    tr = inputs.drift_traces(spec, 1, 1, seed=seed)[:, 0, 0]
    opt = int(oracle.belady(128, tr, 2000).sum())
    for policy in ("lru", "fifo", "random"):
        c = oracle.Cache(128, 64, policy, seed=seed, C=2000)
        tot = sum(c.resolve(S)[0] for S in tr)
        assert tot >= opt, policy
    c = oracle.Cache(64, 64, "swap", C=2000)
    assert sum(c.resolve(S)[0] for S in tr) >= int(oracle.belady(64, tr, 2000).sum())


def test_random_policy_key_is_splitmix64_at_counter():
    """Fill a 6-slot buffer, then one miss: the victim is the unselected slot whose key
    1 + (splitmix64 output at counter ((t*R + r)*L + l)*B + slot) >> 33 is smallest."""
    B, k, R, L, r, l, seed = 6, 6, 3, 2, 1, 1, 77
    c = oracle.Cache(B, k, "random", seed=seed, R=R, L=L, r=r, l=l, C=100)
    c.resolve(np.arange(6, dtype=np.int32))          # t = 0: fills slots 0..5 with 0..5
    S = np.array([0, 1, 2, 3, 4, 50], dtype=np.int32)
    m, locs = c.resolve(S)                           # t = 1: one miss; candidate = slot 5 only
    assert m == 1 and locs[5] == 5
    S2 = np.array([50, 60, 61, 62, 0, 1], dtype=np.int32)  # t = 2: three misses among slots 2, 3, 4
    stream = inputs.splitmix64_stream(seed, 200)     # stream[n-1] = output at counter n
    t = 2
    keys = {}
    for slot in (2, 3, 4):
        n = ((t * R + r) * L + l) * B + slot
        keys[slot] = 1 + (int(stream[n - 1]) >> 33)
    m, locs = c.resolve(S2)
    assert m == 3
    victims = sorted(sorted(keys, key=lambda j: (keys[j], j))[:3])
    assert sorted(locs[1:4].tolist()) == victims == [2, 3, 4]


def test_random_policy_victims_follow_keys():
    """Three of five stale slots are evicted: exactly the three smallest keys."""
    B, k, seed = 8, 3, 12345
    c = oracle.Cache(B, k, "random", seed=seed, R=1, L=1, r=0, l=0, C=100)
    for i in range(0, 9, 3):
        c.resolve(np.array([i, i + 1, i + 2], dtype=np.int32))  # t = 0, 1, 2
    tag_before, _ = c.slots()
    S = np.array([90, 91, 92], dtype=np.int32)                   # t = 3: 3 misses, no hits
    stream = inputs.splitmix64_stream(seed, 64)
    keys = {}
    for slot in range(B):
        if tag_before[slot] < 0:
            keys[slot] = 0
        else:
            keys[slot] = 1 + (int(stream[(3 * B + slot) - 1]) >> 33)
    expect = sorted(sorted(range(B), key=lambda j: (keys[j], j))[:3])
    m, locs = c.resolve(S)
    assert m == 3 and locs.tolist() == expect


def test_validation_bits():
    valid, err = oracle.validate([4, -1, 4, 7, -3, 2], C=7)
    assert valid.tolist() == [True, False, False, False, False, True]
    assert err == oracle.ERR_RANGE | oracle.ERR_DUP


def test_policy_order_on_drift_traces():
    """Shape check against §4's ordering (swap-vanilla worst, LRU best online, Belady lowest,
    doubling B helps LRU) on the synthetic stand-in traces.  The absolute rates of the
    replayed GLM-5.1 traces are not reproduced (parity unpinned)."""
    spec = inputs.TraceSpec(ctx0=20000, k=128, steps=120, keep=0.85, recency_mean=128)
    tr = inputs.drift_traces(spec, 1, 1, seed=4)[:, 0, 0]

    def run(policy, B):
        c = oracle.Cache(B, 128, policy, seed=1, C=20000)
        return sum(c.resolve(S)[0] for S in tr[1:]) if c.resolve(tr[0]) else 0

    swap, lru, fifo, rnd, lru2 = run("swap", 128), run("lru", 256), run("fifo", 256), run("random", 256), run("lru", 512)
    bel = int(oracle.belady(256, tr, 20000)[1:].sum())
    assert swap > fifo >= lru > bel
    assert rnd >= lru
    assert lru2 < lru


# ---- buffers grown on demand: only slots [0, cap) exist ----------------------------------

@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("B,cap,k,npos", [(32, 8, 3, 20), (64, 16, 5, 40), (20, 6, 6, 12)])
def test_capped_lru_is_the_recency_list_of_cap_entries(seed, B, cap, k, npos):
    rng = np.random.default_rng(300 + seed)
    trace = _random_trace(rng, 30, k, npos)
    c = oracle.Cache(B, k, "lru", C=npos)
    c.set_cap(cap)
    for S, (m_ref, order) in zip(trace, _lru_list_model(cap, trace)):
        m, locs = c.resolve(S)
        assert m == m_ref
        assert (locs < cap).all()
        tag, stamp = c.slots()
        assert (tag[cap:] == -1).all() and (stamp[cap:] == 0).all()
        occ = tag >= 0
        assert [int(t) for _, t in sorted(zip(stamp[occ].tolist(), tag[occ].tolist()))] == order


@pytest.mark.parametrize("seed", range(4))
def test_capped_fifo_is_the_insertion_queue_of_cap_entries(seed):
    rng = np.random.default_rng(400 + seed)
    B, cap, k, npos = 40, 10, 4, 30
    trace = _random_trace(rng, 30, k, npos)
    c = oracle.Cache(B, k, "fifo", C=npos)
    c.set_cap(cap)
    for S, (m_ref, queue) in zip(trace, _fifo_queue_model(cap, trace)):
        m, _ = c.resolve(S)
        assert m == m_ref
        tag, stamp = c.slots()
        occ = tag >= 0
        assert [int(t) for _, t in sorted(zip(stamp[occ].tolist(), tag[occ].tolist()))] == queue


@pytest.mark.parametrize("policy", ["lru", "fifo", "random", "swap"])
def test_growth_ahead_of_the_context_equals_the_full_buffer(policy):
    """Empty slots go first, lowest slot first: a buffer whose cap stays >= min(B, context) never
    evicts where the full buffer would not, so every step matches the full buffer exactly."""
    ctx0, k, B, T, page = 40, 8, 128, 60, 16
    spec = inputs.TraceSpec(ctx0=ctx0, k=k, steps=T, keep=0.7, recency_mean=12, appends=True)
    tr = inputs.drift_traces(spec, 1, 1, seed=17)[:, 0, 0]
    full = oracle.Cache(B, k, policy, seed=3, C=ctx0 + T)
    grown = oracle.Cache(B, k, policy, seed=3, C=ctx0 + T)
    for t, S in enumerate(tr):
        ctx = ctx0 + t + 1  # the append makes position ctx0 + t
        grown.set_cap(min(B, -(-max(ctx, k) // page) * page))
        assert full.append(ctx0 + t) == grown.append(ctx0 + t)
        a, b = full.resolve(S), grown.resolve(S)
        assert a[0] == b[0] and np.array_equal(a[1], b[1]), t
        assert all(np.array_equal(x, y) for x, y in zip(full.slots(), grown.slots())), t
    assert full.counters() == grown.counters()


@pytest.mark.parametrize("policy", ["lru", "random"])
def test_fewer_than_k_slots_refuse_the_step(policy):
    c = oracle.Cache(16, 6, policy, C=100)
    c.set_cap(16)
    c.resolve(np.arange(6, dtype=np.int32))
    before = (c.slots(), c.counters())
    c.set_cap(5)
    m, locs = c.resolve(np.arange(10, 16, dtype=np.int32))
    assert m == -1 and (locs == -1).all()
    assert c.append(50) == -1
    tag, stamp = c.slots()
    cnt = c.counters()
    assert np.array_equal(tag, before[0][0]) and np.array_equal(stamp, before[0][1])
    assert cnt["err"] == oracle.ERR_SLOTS
    assert {k_: v for k_, v in cnt.items() if k_ != "err"} == {k_: v for k_, v in before[1].items() if k_ != "err"}
    with pytest.raises(ValueError):
        c.set_cap(17)
