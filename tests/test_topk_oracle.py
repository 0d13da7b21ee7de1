"""Pin the top-k selection oracle to references other than itself (CPU only):
a hand-worked example, brute-force selection in pure Python on small random
inputs (with ties and NaN), the values torch.topk returns, and structural
properties; then plant plausible mistakes in copies of the oracle and check
that a pin catches each."""
import importlib.util
import os

import numpy as np
import pytest
import torch

import oracle.topk_ref as tk

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "topk_example.txt")


def _golden():
    cu, topk, scores, expect = None, None, [], []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("cu_seqlens"):
            cu = np.array([int(x) for x in line.split()[1:]], np.int32)
        elif line.startswith("topk"):
            topk = int(line.split()[1])
        elif line.startswith("row"):
            left, right = line[3:].split("|")
            scores.append([float(x) for x in left.split()])
            expect.append([int(x) for x in right.split()])
    return np.array(scores), cu, topk, np.array(expect, np.int32)


def _brute(scores, cu, topk):
    """Pure-Python selection: repeatedly take the first largest remaining candidate."""
    T, ncols = scores.shape
    out = np.full((T, 1, topk), -1, np.int32)
    for t in range(T):
        b = max(i for i in range(len(cu) - 1) if cu[i] <= t)
        s0 = int(cu[b])
        cand = list(range(min(t - s0 + 1, ncols)))
        for j in range(min(topk, len(cand))):
            def rank(c):
                v = scores[t, c]
                return (0 if np.isnan(v) else 1, -np.inf if np.isnan(v) else v, -c)
            best = max(cand, key=rank)
            out[t, 0, j] = s0 + best
            cand.remove(best)
    return out


def _random_case(seed, T=60, ncols=40, topk=16, tie_levels=5, nan_frac=0.05):
    rng = np.random.default_rng(seed)
    lens = []
    while sum(lens) < T:
        lens.append(int(rng.integers(1, ncols + 1)))
    lens[-1] -= sum(lens) - T
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    scores = rng.integers(0, tie_levels, size=(T, ncols)).astype(np.float64) / tie_levels   # many ties
    scores[rng.random((T, ncols)) < nan_frac] = np.nan
    return scores, cu, topk


def pin_golden(tk):
    scores, cu, topk, expect = _golden()
    return int((tk.topk_indices(scores, cu, topk)[:, 0, :] != expect).sum())


def pin_brute(tk, seeds=(1, 2, 3)):
    bad = 0
    for s in seeds:
        scores, cu, topk = _random_case(s)
        bad += int((tk.topk_indices(scores, cu, topk) != _brute(scores, cu, topk)).sum())
    return bad


def pin_torch_values(tk, seed=4):
    """The selected scores equal torch.topk's values (sorted, NaN-free rows)."""
    rng = np.random.default_rng(seed)
    T, ncols, topk = 50, 64, 24
    cu = np.array([0, 20, 50], np.int32)
    scores = rng.standard_normal((T, ncols))
    idx = tk.topk_indices(scores, cu, topk)
    bad = 0
    for t in range(T):
        s0 = cu[np.searchsorted(cu, t, side="right") - 1]
        n = t - s0 + 1
        k = min(topk, n)
        vals = torch.topk(torch.from_numpy(scores[t, :n]), k).values.numpy()
        got = scores[t, idx[t, 0, :k] - s0]
        bad += int(not np.array_equal(got, vals)) + int(np.any(idx[t, 0, k:] != -1))
    return bad


def pin_properties(tk, seed=5):
    """Indices lie in [s0, t], are distinct, scores are non-increasing, ties ascend."""
    scores, cu, topk = _random_case(seed, nan_frac=0.0)
    idx = tk.topk_indices(scores, cu, topk)
    bad = 0
    for t in range(scores.shape[0]):
        s0 = cu[np.searchsorted(cu, t, side="right") - 1]
        row = idx[t, 0]
        v = row[row >= 0]
        bad += int(v.size != min(topk, t - s0 + 1, scores.shape[1]))
        bad += int(np.any(v < s0) or np.any(v > t) or np.unique(v).size != v.size)
        sc = scores[t, v - s0]
        bad += int(np.any(np.diff(sc) > 0))
        bad += int(np.any((np.diff(sc) == 0) & (np.diff(v) < 0)))
    return bad


def test_pin_golden():
    assert pin_golden(tk) == 0


def test_pin_brute_force():
    assert pin_brute(tk) == 0


def test_pin_torch_topk_values():
    assert pin_torch_values(tk) == 0


def test_pin_properties():
    assert pin_properties(tk) == 0


MUTANTS = {
    "k not capped at the causal count": ("k = min(topk, n)", "k = min(topk, ncols)"),
    "causal range off by one": ("n = min(t - s0 + 1, ncols)", "n = min(t - s0, ncols)"),
    "ascending order": ('key = np.where(np.isnan(s), np.inf, -s)', 'key = np.where(np.isnan(s), np.inf, s)'),
    "ties by descending column": ('order = np.argsort(key, kind="stable")',
                                  'order = (len(key) - 1 - np.argsort(key[::-1], kind="stable"))'),
    "NaN sorts first": ('key = np.where(np.isnan(s), np.inf, -s)', 'key = np.where(np.isnan(s), -np.inf, -s)'),
    "padding with 0": ("out = np.full((T, 1, topk), -1, dtype=np.int32)", "out = np.full((T, 1, topk), 0, dtype=np.int32)"),
    "local instead of packed rows": ("out[t, 0, :k] = s0 + topk_row(scores[t], n, k)", "out[t, 0, :k] = topk_row(scores[t], n, k)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(tk.__file__).read()
    assert src.count(old) == 1, name
    path = tmp_path / "topk_mutant.py"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location("topk_mutant", path)
    mut = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mut)
    try:
        caught = pin_golden(mut) + pin_brute(mut) + pin_torch_values(mut) + pin_properties(mut)
    except (ValueError, IndexError):      # a shape or index error is caught as well
        caught = 1
    assert caught > 0, name
