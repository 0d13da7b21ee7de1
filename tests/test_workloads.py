"""The seeded synthetic inputs both sides are fed: sequence layouts, index
structure (causal, distinct, -1 padded, the stated number of all-padding rows,
the clustered window), determinism, and the bf16 rounding of the values.  The
generator holds none of the method's arithmetic; these checks pin the input
recipe the measurements are quoted on."""
import numpy as np
import pytest

from bwd_sparse_mla_gb300 import workloads as W


def _row_starts(w):
    starts = np.repeat(w.cu_seqlens[:-1], np.diff(w.cu_seqlens))
    return starts.astype(np.int64)


def _check_causal(w, rows):
    idx = w.indices.reshape(w.T, w.topk)[rows].astype(np.int64)
    t = np.asarray(rows, dtype=np.int64)
    s0 = _row_starts(w)[rows]
    k = np.minimum(t - s0 + 1, w.topk)
    valid = idx >= 0
    n = valid.sum(axis=1)
    empty = n == 0
    assert np.all(n[~empty] == k[~empty]), "a row has min(p + 1, topk) valid slots"
    # valid slots first, then -1 padding
    first_pad = np.where(valid.all(axis=1), w.topk, np.argmin(valid, axis=1))
    assert np.all(first_pad[~empty] == n[~empty])
    assert np.all((idx[valid] >= np.broadcast_to(s0[:, None], idx.shape)[valid]))
    assert np.all((idx[valid] <= np.broadcast_to(t[:, None], idx.shape)[valid])), "causal: s0 <= idx <= t"
    srt = np.sort(idx, axis=1)
    dup = (srt[:, 1:] == srt[:, :-1]) & (srt[:, 1:] >= 0)
    assert not dup.any(), "indices of a row are distinct"
    return int(empty.sum())


@pytest.mark.parametrize("config,lens_rule,n_empty", [
    (1, lambda L: L == [256], 4),
    (2, lambda L: all(256 <= x <= 8192 for x in L[:-1]) and 0 < L[-1] <= 8192, round(0.01 * 16384)),
    (4, lambda L: L == [16384], round(0.005 * 16384)),
    (5, lambda L: all(128 <= x <= 32768 for x in L[:-1]) and 0 < L[-1] <= 32768, round(0.01 * 65536)),
])
def test_causal_workloads(config, lens_rule, n_empty):
    w = W.make_workload(config, values=False)
    assert int(w.cu_seqlens[0]) == 0 and int(w.cu_seqlens[-1]) == w.T and np.all(np.diff(w.cu_seqlens) > 0)
    assert lens_rule(list(w.seqlens)) and sum(w.seqlens) == w.T
    assert w.indices.shape == (w.T, 1, w.topk) and w.indices.dtype == np.int32
    rows = np.arange(w.T) if w.T <= 16384 else np.sort(np.random.default_rng(0).choice(w.T, 4096, replace=False))
    empties = _check_causal(w, rows)
    all_empty = int((w.indices.reshape(w.T, w.topk).max(axis=1) < 0).sum())
    assert all_empty == n_empty
    if rows.size == w.T:
        assert empties == n_empty


def test_clustered_workload_windows():
    w = W.make_workload(3, values=False)
    assert list(w.seqlens) == [8192] * 4
    idx = w.indices.reshape(w.T, w.topk).astype(np.int64)
    s0 = _row_starts(w)
    for t in np.random.default_rng(1).choice(w.T, 512, replace=False):
        p = t - s0[t]
        row = idx[t][idx[t] >= 0] - s0[t]
        assert row.size == min(w.topk, p + 1) and np.unique(row).size == row.size
        lo = max(0, p - 511)
        assert set(range(lo, p + 1)) <= set(row.tolist()), "the 512-wide local window is always taken"
        far = row[row < lo]
        assert far.size == min(w.topk - (p + 1 - lo), lo) and np.all(far >= 0)


def test_same_seed_same_inputs_and_values_independent_of_threads():
    a = W.make_custom(1000, 8, 128, [300, 700], seed=5, threads=1)
    b = W.make_custom(1000, 8, 128, [300, 700], seed=5, threads=4)
    for name in ("q", "kv", "dout", "indices"):
        assert np.array_equal(getattr(a, name), getattr(b, name)), name
    c = W.make_custom(1000, 8, 128, [300, 700], seed=6, threads=1)
    assert not np.array_equal(a.q, c.q)


def test_bf16_rounding_is_round_to_nearest_even():
    one = np.float32(1.0)
    cases = {
        one: 0x3F80,
        np.float32(1 + 2.0 ** -8): 0x3F80,              # halfway: ties to the even code
        np.float32(1 + 3 * 2.0 ** -8): 0x3F82,          # halfway between 0x3F81 and 0x3F82
        np.float32(1 + 2.0 ** -8 + 2.0 ** -20): 0x3F81,  # above halfway rounds up
        np.float32(-0.0): 0x8000,
        np.float32(np.inf): 0x7F80,
        np.float32(-2.5): 0xC020,
    }
    got = W.f32_to_bf16_bits(np.array(list(cases), dtype=np.float32))
    assert [int(g) for g in got] == list(cases.values())
    nan = W.f32_to_bf16_bits(np.array([np.nan], dtype=np.float32))[0]
    assert (int(nan) & 0x7F80) == 0x7F80 and (int(nan) & 0x7F) != 0


def test_headline_values_have_the_stated_scales():
    w = W.make_workload(5, values=False)
    assert w.q_std == 8.0
    W.draw_values(w, rows=range(512))
    as_f32 = lambda bits: (bits.astype(np.uint32) << 16).view(np.float32)   # noqa: E731  (bf16 bits -> fp32, exact)
    q = as_f32(w.q.reshape(w.T, -1)[:512])
    kv = as_f32(w.kv.reshape(w.T, -1))
    assert abs(float(q.std()) - 8.0) < 0.1
    assert abs(float(kv.std()) - 1.0) < 0.01
