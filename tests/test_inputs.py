"""The seeded input generators: published test vectors and the trace shape."""
import numpy as np
import pytest

from hierarchical_kv_cache_02_gb300 import inputs


def test_splitmix64_published_vector():
    # splitmix64 seeded with 1234567: the first outputs of the reference implementation
    # (Steele, Lea and Flood 2014; Vigna's public C version).
    assert inputs.splitmix64_stream(1234567, 3).tolist() == [
        6457827717110365317, 3203168211198807973, 9817491932198370423]


@pytest.mark.parametrize("appends", [False, True])
def test_trace_rows_are_distinct_in_range_and_drift(appends):
    spec = inputs.TraceSpec(ctx0=4096, k=256, steps=64, keep=0.9, recency_mean=512, appends=appends)
    tr = inputs.drift_traces(spec, 2, 3, seed=1)
    assert tr.shape == (64, 3, 2, 256)
    for r in range(2):
        for l in range(3):
            prev = None
            for t in range(64):
                row = tr[t, l, r]
                n = 4096 + (t + 1 if appends else 0)
                assert len(set(row.tolist())) == 256
                assert row.min() >= 0 and row.max() < n
                assert n - 1 in row  # newest position always selected
                if prev is not None:
                    assert len(set(row.tolist()) & prev) >= round(0.9 * 256) - 1
                prev = set(row.tolist())
    # different (r, l) get different traces; the same seed reproduces them
    assert not np.array_equal(tr[:, 0, 0], tr[:, 1, 0])
    assert np.array_equal(tr, inputs.drift_traces(spec, 2, 3, seed=1))


def test_burst_moves_a_contiguous_far_span():
    k = 256
    spec = inputs.TraceSpec(ctx0=100000, k=k, steps=40, keep=0.9, recency_mean=512,
                            burst_every=32, burst_frac=0.4, far_gap=8 * 512)
    tr = inputs.drift_traces(spec, 1, 1, seed=3)[:, 0, 0]
    row = np.sort(tr[32])
    span = round(0.4 * k)
    runs = np.split(row, np.where(np.diff(row) != 1)[0] + 1)
    longest = max(runs, key=len)
    assert len(longest) >= span and longest[0] <= 100000 - 1 - 8 * 512 - span + span
