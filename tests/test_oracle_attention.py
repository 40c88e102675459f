"""Pins of the oracle's fp64 attention.

The HiSparse summary (§3) states that attention over the resolved set is exact:
the selected positions, scores and outputs are those of full-resident KV.  So
the oracle's sparse attention must equal DENSE attention over the whole history
with every unselected position masked out -- computed here a different way
(one dense matrix product over all C rows, then a masked softmax), plus closed
forms: k = 1 gives V, zero logits give the mean of V, order does not matter,
padding and invalid entries are ignored, and GQA heads read their own block.
"""
import numpy as np
import pytest

import oracle


def _bits(x):
    """float array -> bf16 bit patterns (round to nearest even) and the exact values they hold."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    vals = (rounded.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return rounded, vals


def _dense_masked(qv, hv, S, scale, kv_heads, Dqk, Dv):
    """Dense attention over all C rows with a -inf mask off the selected set (fp64)."""
    Hq = qv.shape[0]
    C = hv.shape[0]
    mask = np.full(C, -np.inf)
    for s in S:
        if 0 <= s < C:
            mask[s] = 0.0
    out = np.zeros((Hq, Dv))
    group = Hq // kv_heads if kv_heads else Hq
    for h in range(Hq):
        if kv_heads:
            g = h // group
            K = hv[:, g * (Dqk + Dv): g * (Dqk + Dv) + Dqk]
            V = hv[:, g * (Dqk + Dv) + Dqk: (g + 1) * (Dqk + Dv)]
        else:
            K, V = hv[:, :Dqk], hv[:, :Dv]
        z = scale * (K @ qv[h]) + mask
        w = np.exp(z - z.max())
        out[h] = (w / w.sum()) @ V
    return out


@pytest.mark.parametrize("layout", ["mla", "gqa"])
@pytest.mark.parametrize("seed", range(4))
def test_selected_set_equals_dense_masked(layout, seed):
    rng = np.random.default_rng(seed)
    if layout == "mla":
        Hq, kvh, Dqk, Dv = 16, 0, 64, 48
        rec = Dqk
    else:
        Hq, kvh, Dqk, Dv = 8, 2, 16, 24
        rec = kvh * (Dqk + Dv)
    C, k = 300, 37
    qb, qv = _bits(rng.standard_normal((Hq, Dqk)))
    hb, hv = _bits(rng.standard_normal((C, rec)))
    S = rng.choice(C, size=k, replace=False).astype(np.int32)
    scale = 1.0 / np.sqrt(Dqk)
    got = oracle.attention(qb, hb, S, np.float32(scale), kvh, Dqk, Dv)
    ref = _dense_masked(qv, hv, S, float(np.float32(scale)), kvh, Dqk, Dv)
    assert np.max(np.abs(got - ref)) <= 1e-12


def test_single_selection_returns_v_and_zero_logits_average():
    rng = np.random.default_rng(7)
    Hq, Dqk, Dv, C = 4, 32, 16, 50
    qb, _ = _bits(rng.standard_normal((Hq, Dqk)))
    hb, hv = _bits(rng.standard_normal((C, Dqk)))
    out = oracle.attention(qb, hb, np.array([17], np.int32), 0.125, 0, Dqk, Dv)
    assert np.array_equal(out, np.tile(hv[17, :Dv], (Hq, 1)))
    S = np.array([3, 9, 11, 40], np.int32)
    out0 = oracle.attention(np.zeros((Hq, Dqk), np.uint16), hb, S, 0.125, 0, Dqk, Dv)
    assert np.max(np.abs(out0 - hv[S, :Dv].mean(axis=0))) <= 1e-15


def test_two_token_closed_form():
    """out = sigmoid(z1 - z2) V1 + sigmoid(z2 - z1) V2."""
    rng = np.random.default_rng(2)
    Dqk, Dv, C = 8, 8, 5
    qb, qv = _bits(rng.standard_normal((1, Dqk)))
    hb, hv = _bits(rng.standard_normal((C, Dqk)))
    z1, z2 = 0.5 * hv[1] @ qv[0], 0.5 * hv[4] @ qv[0]
    w1 = 1.0 / (1.0 + np.exp(z2 - z1))
    ref = w1 * hv[1] + (1 - w1) * hv[4]
    out = oracle.attention(qb, hb, np.array([4, 1], np.int32), 0.5, 0, Dqk, Dv)
    assert np.max(np.abs(out[0] - ref)) <= 1e-14


def test_order_padding_and_invalid_entries_do_not_matter():
    rng = np.random.default_rng(5)
    Hq, kvh, Dqk, Dv, C = 8, 4, 16, 16, 64
    qb, _ = _bits(rng.standard_normal((Hq, Dqk)))
    hb, _ = _bits(rng.standard_normal((C, kvh * (Dqk + Dv))))
    S = np.array([5, 60, 2, 33, 17], np.int32)
    base = oracle.attention(qb, hb, S, 0.25, kvh, Dqk, Dv)
    perm = oracle.attention(qb, hb, S[::-1].copy(), 0.25, kvh, Dqk, Dv)
    noisy = np.array([-1, 5, 60, 5, 2, 99, 33, -1, 17, 2], np.int32)
    padded = oracle.attention(qb, hb, noisy, 0.25, kvh, Dqk, Dv)
    assert np.max(np.abs(base - perm)) <= 1e-14
    assert np.max(np.abs(base - padded)) <= 1e-14
    empty = oracle.attention(qb, hb, np.array([-1, -1], np.int32), 0.25, kvh, Dqk, Dv)
    assert not empty.any()


def test_gqa_heads_read_their_own_block():
    """Query head h must attend with block h // (Hq / kv_heads): make V of block g equal to g+1
    everywhere and check every head's output is exactly its block's constant."""
    Hq, kvh, Dqk, Dv, C = 8, 4, 8, 8, 20
    rng = np.random.default_rng(1)
    hist = rng.standard_normal((C, kvh * (Dqk + Dv)))
    for g in range(kvh):
        hist[:, g * (Dqk + Dv) + Dqk:(g + 1) * (Dqk + Dv)] = g + 1
    hb, _ = _bits(hist)
    qb, _ = _bits(rng.standard_normal((Hq, Dqk)))
    out = oracle.attention(qb, hb, np.arange(0, C, 3, dtype=np.int32), 0.3, kvh, Dqk, Dv)
    for h in range(Hq):
        assert np.allclose(out[h], h // 2 + 1, rtol=0, atol=1e-14)


def test_mla_value_is_the_leading_slice():
    """In the shared-latent layout V is the first Dv values of the record: with one selected
    record the output equals those values exactly."""
    rng = np.random.default_rng(4)
    hb, hv = _bits(rng.standard_normal((10, 24)))
    qb, _ = _bits(rng.standard_normal((3, 24)))
    out = oracle.attention(qb, hb, np.array([6], np.int32), 1.0, 0, 24, 16)
    assert np.array_equal(out[1], hv[6, :16])


def test_scale_multiplies_logits():
    rng = np.random.default_rng(9)
    qf = rng.standard_normal((2, 16))
    qb, _ = _bits(qf)
    q2b, _ = _bits(2 * qf)  # doubling is exact in bf16
    hb, _ = _bits(rng.standard_normal((30, 16)))
    S = np.arange(0, 30, 2, dtype=np.int32)
    a = oracle.attention(qb, hb, S, 0.5, 0, 16, 16)
    b = oracle.attention(q2b, hb, S, 0.25, 0, 16, 16)
    assert np.max(np.abs(a - b)) <= 1e-14
