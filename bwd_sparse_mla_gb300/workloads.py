"""Seeded synthetic workloads for DSA-style sparse MLA attention.

This module only draws inputs: random values, sequence lengths and top-k
index lists.  It holds none of the attention arithmetic, so both the CUDA
path and the fp64 oracle can consume its output without sharing code.

Shapes follow the GLM-5 sparse-MLA kernels described in the miles PR #2079
summary ("fix -1 index OOB and NaN grads in the GLM-5 sparse-MLA kernel",
key code fragments): every KV row carries a D=512 latent part (also the
value) plus a D_tail=64 rope tail, one KV group is shared by all heads, and
top-k slots that name no key hold the sentinel -1.  The Megatron-Bridge
"GLM-5 DSA option: tilelang (2/2)" PR (Bug fixes) states that the indexer
caps k at the sequence length and pads back to the fixed top-k width with -1,
and that the fused backend runs on the packed thd layout.

Values are drawn as fp32 normals and rounded to bf16 (round to nearest even);
bf16 tensors are carried as their raw uint16 bit patterns.

Five workloads:
  1 tiny        T=256,  H=8,   topk=64,   one sequence, 4 rows all -1
  2 prod-shard  T=16384,H=8,   topk=2048, ragged lengths U{256..8192}, 1% rows all -1
  3 clustered   T=32768,H=16,  topk=2048, 4 x 8192, 512-wide local window + 1536 random
  4 h64         T=16384,H=64,  topk=2048, one sequence, 0.5% rows all -1
  5 headline    T=65536,H=128, topk=2048, log-uniform lengths in [128,32768],
                q ~ N(0, 8^2), 1% rows all -1
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

D_LATENT = 512          # latent width; the latent part is also V
D_TAIL = 64             # rope tail, used only in K
D_QK = D_LATENT + D_TAIL

# rows per independently seeded chunk when drawing large value tensors;
# fixed so the draw does not depend on the number of threads
_CHUNK_TOKENS = 256


@dataclass
class Workload:
    name: str
    T: int
    H: int
    topk: int
    seqlens: list
    scale: float
    q_std: float = 1.0
    seed: int = 0
    # filled by draw()
    cu_seqlens: np.ndarray = field(default=None, repr=False)
    indices: np.ndarray = field(default=None, repr=False)   # int32 [T, 1, topk]
    q: np.ndarray = field(default=None, repr=False)         # bf16 bits [T, H, 576]
    kv: np.ndarray = field(default=None, repr=False)        # bf16 bits [T, 1, 576]
    dout: np.ndarray = field(default=None, repr=False)      # bf16 bits [T, H, 512]

    @property
    def B(self) -> int:
        return len(self.seqlens)

    def n_valid(self) -> int:
        idx = self.indices
        return int(((idx >= 0) & (idx < self.T)).sum())


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest even) and return the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def _normal_bf16(seed: int, stream: int, shape: tuple, std: float, threads: int,
                 rows=None) -> np.ndarray:
    """Draw N(0, std^2) in fp32, round to bf16 bits; chunked over the first axis.

    With `rows`, only the chunks holding those rows are drawn (the others are
    left unset); every drawn value is identical to a full draw."""
    T = shape[0]
    row = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    out = np.empty((T, row), dtype=np.uint16)
    n_chunks = (T + _CHUNK_TOKENS - 1) // _CHUNK_TOKENS
    children = np.random.SeedSequence([seed, stream]).spawn(max(n_chunks, 1))

    def fill(c: int) -> None:
        lo = c * _CHUNK_TOKENS
        hi = min(T, lo + _CHUNK_TOKENS)
        g = np.random.Generator(np.random.PCG64(children[c]))
        x = g.standard_normal((hi - lo, row), dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[lo:hi] = f32_to_bf16_bits(x)

    chunks = range(n_chunks) if rows is None else sorted({int(r) // _CHUNK_TOKENS for r in rows if 0 <= r < T})
    if len(chunks) <= 1 or threads <= 1:
        for c in chunks:
            fill(c)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(fill, chunks))
    return out.reshape(shape)


def _lengths_until(rng: np.random.Generator, total: int, draw) -> list:
    """Draw sequence lengths until they reach `total`; truncate the last one."""
    out = []
    acc = 0
    while acc < total:
        n = int(draw(rng))
        n = min(n, total - acc)
        out.append(n)
        acc += n
    return out


def _causal_uniform_row(rng, s0: int, p: int, topk: int) -> np.ndarray:
    """min(p+1, topk) distinct positions drawn uniformly from [s0, s0+p], random order."""
    n = p + 1
    if n <= topk:
        return (s0 + rng.permutation(n)).astype(np.int32)
    return (s0 + rng.choice(n, size=topk, replace=False, shuffle=True)).astype(np.int32)


def _clustered_row(rng, s0: int, p: int, topk: int, window: int) -> np.ndarray:
    """Local window [p-window+1, p] plus up to topk-window distinct earlier positions."""
    lo = max(0, p - window + 1)
    local = np.arange(lo, p + 1)
    n_far = lo                       # candidates in [0, lo)
    k_far = min(topk - local.size, n_far)
    far = rng.choice(n_far, size=k_far, replace=False, shuffle=True) if k_far > 0 else np.empty(0, np.int64)
    row = np.concatenate([local, far])
    rng.shuffle(row)
    return (s0 + row).astype(np.int32)


def _draw_indices(w: Workload, rng: np.random.Generator, kind: str, empty_frac: float,
                  n_empty: int = 0) -> np.ndarray:
    T, K = w.T, w.topk
    idx = np.full((T, K), -1, dtype=np.int32)
    s0 = 0
    for L in w.seqlens:
        for p in range(L):
            if kind == "causal":
                row = _causal_uniform_row(rng, s0, p, K)
            else:
                row = _clustered_row(rng, s0, p, K, window=512)
            idx[s0 + p, :row.size] = row
        s0 += L
    if n_empty == 0 and empty_frac > 0:
        n_empty = max(1, int(round(empty_frac * T)))
    if n_empty:
        rows = rng.choice(T, size=n_empty, replace=False)
        idx[rows] = -1
    return idx.reshape(T, 1, K)


def make_workload(config: int, seed: int | None = None, threads: int | None = None,
                  values: bool = True) -> Workload:
    """Build workload `config` (1..5).  Seed defaults to 1000 + config."""
    if seed is None:
        seed = 1000 + config
    if threads is None:
        threads = min(32, os.cpu_count() or 1)
    rng = np.random.default_rng(seed)
    scale = 1.0 / math.sqrt(D_QK)
    if config == 1:
        w = Workload("tiny T=256 H=8 topk=64", 256, 8, 64, [256], scale, seed=seed)
        w.indices = _draw_indices(w, rng, "causal", 0.0, n_empty=4)
    elif config == 2:
        lens = _lengths_until(rng, 16384, lambda g: g.integers(256, 8193))
        w = Workload("prod-shard T=16384 H=8 topk=2048 ragged", 16384, 8, 2048, lens, scale, seed=seed)
        w.indices = _draw_indices(w, rng, "causal", 0.01)
    elif config == 3:
        w = Workload("clustered T=32768 H=16 topk=2048 4x8192", 32768, 16, 2048, [8192] * 4, scale, seed=seed)
        w.indices = _draw_indices(w, rng, "clustered", 0.0)
    elif config == 4:
        w = Workload("h64 T=16384 H=64 topk=2048 one sequence", 16384, 64, 2048, [16384], scale, seed=seed)
        w.indices = _draw_indices(w, rng, "causal", 0.005)
    elif config == 5:
        lens = _lengths_until(rng, 65536,
                              lambda g: math.exp(g.uniform(math.log(128), math.log(32768))))
        w = Workload("headline T=65536 H=128 topk=2048 log-uniform ragged", 65536, 128, 2048, lens,
                     scale, q_std=8.0, seed=seed)
        w.indices = _draw_indices(w, rng, "causal", 0.01)
    else:
        raise ValueError(f"unknown workload {config}")
    w.cu_seqlens = np.concatenate([[0], np.cumsum(w.seqlens)]).astype(np.int32)
    assert int(w.cu_seqlens[-1]) == w.T
    if values:
        draw_values(w, threads)
    return w


def draw_values(w: Workload, threads: int | None = None, rows=None) -> None:
    """Draw q, kv and dO.  With `rows`, q and dO are drawn only for the chunks
    holding those tokens (kv is always drawn in full)."""
    if threads is None:
        threads = min(32, os.cpu_count() or 1)
    w.q = _normal_bf16(w.seed, 1, (w.T, w.H, D_QK), w.q_std, threads, rows)
    w.kv = _normal_bf16(w.seed, 2, (w.T, 1, D_QK), 1.0, threads)
    w.dout = _normal_bf16(w.seed, 3, (w.T, w.H, D_LATENT), 1.0, threads, rows)


def make_custom(T: int, H: int, topk: int, seqlens: list, seed: int, kind: str = "causal",
                empty_rows: int = 0, q_std: float = 1.0, scale: float | None = None,
                threads: int = 1) -> Workload:
    """Small custom workload with the same recipe (used by tests)."""
    rng = np.random.default_rng(seed)
    if scale is None:
        scale = 1.0 / math.sqrt(D_QK)
    w = Workload(f"custom T={T} H={H} topk={topk}", T, H, topk, list(seqlens), scale, q_std=q_std, seed=seed)
    assert sum(seqlens) == T
    w.indices = _draw_indices(w, rng, kind, 0.0, n_empty=empty_rows)
    w.cu_seqlens = np.concatenate([[0], np.cumsum(w.seqlens)]).astype(np.int32)
    draw_values(w, threads)
    return w


def truncate(w: Workload, n_tokens: int) -> Workload:
    """The first n_tokens tokens of a workload (a smaller case with the same
    shapes per token): sequences are cut at n_tokens, and slots naming a row
    at or past n_tokens become -1 padding."""
    n = int(n_tokens)
    lens, acc = [], 0
    for L in w.seqlens:
        if acc >= n:
            break
        lens.append(min(L, n - acc))
        acc += lens[-1]
    idx = np.array(w.indices[:n], copy=True)
    idx[idx >= n] = -1
    out = Workload(f"{w.name} (first {n} tokens)", n, w.H, w.topk, lens, w.scale, q_std=w.q_std, seed=w.seed)
    out.indices = idx
    out.cu_seqlens = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    out.q = None if w.q is None else w.q[:n]
    out.kv = None if w.kv is None else w.kv[:n]
    out.dout = None if w.dout is None else w.dout[:n]
    return out


def sample_rows(w: Workload, n: int, seed: int = 7) -> np.ndarray:
    """A fixed stratified row sample: every all-padding row (up to n/8), the
    first and last rows of every sequence (up to n/4), plus uniform rows."""
    rng = np.random.default_rng(seed)
    idx = w.indices.reshape(w.T, w.topk)
    n_valid = ((idx >= 0) & (idx < w.T)).sum(1)
    picks = []
    empty = np.nonzero(n_valid == 0)[0]
    picks.extend(empty[: max(1, n // 8)].tolist())
    edges = []
    for b in range(w.B):
        s, e = int(w.cu_seqlens[b]), int(w.cu_seqlens[b + 1])
        if e > s:
            edges.extend([s, e - 1])
    edges = np.unique(np.array(edges, dtype=np.int64))
    if edges.size > n // 4:
        edges = rng.choice(edges, size=n // 4, replace=False)
    picks.extend(edges.tolist())
    rest = n - len(set(picks))
    if rest > 0:
        picks.extend(rng.choice(w.T, size=min(rest, w.T), replace=False).tolist())
    return np.unique(np.array(picks, dtype=np.int64))
