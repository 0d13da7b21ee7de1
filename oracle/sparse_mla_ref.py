"""fp64 CPU oracle for DSA-style sparse MLA attention, forward and backward.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, obviously correct
statement of what the CUDA path computes.  Only the test suite, the smoke
check and the benchmark's CPU-baseline leg may import it; the product path
never calls it and shares no code with it.

Every tensor is upcast to float64 on entry (bf16 inputs convert exactly).
Loops run over query tokens; per token the work is a handful of dense
products of small matrices (numpy's matmul is the only library step).

Sources (web pages; cited by title and section):
  [I2201]  slime issue #2201, "GLM-5.2 SparseMLA TileLang backward returns NaN
           gradients from finite inputs" -- sections "Strongest repro
           evidence" (the call sparse_mla_bwd(q, kv, tl_out, grad_output,
           indices, tl_lse, sm_scale)) and "Suspected area" (D = 512 latent).
  [PR2079] miles PR #2079 summary, "fix -1 index OOB and NaN gradients in the
           GLM-5 sparse-MLA kernel" -- "implementation breakdown" items 1-3
           and the two "key code fragments" (forward `main`, backward
           `sparse_mla_bwd_kernel`).
  [PR17]   Megatron-Bridge PR #17, "GLM-5 DSA option: tilelang (2/2)" --
           "Bug fixes" (top-k padded to the fixed width with -1; thd layout).

Readings of points the pages leave open:
  * valid slot = index in [0, T); -1 and every other out-of-range value are
    padding and contribute nothing (the pages mask `index != -1` and clamp).
  * duplicate indices in one row count once per slot (a multiset).
  * the returned LSE is the natural-log LSE; for a row with no valid slot the
    running max is taken as 0 and the floored sum 1e-30 gives
    LSE_EMPTY = ln(1e-30) and an exactly-zero output row.
  * the backward takes `out` and `lse` as given (like the kernel call on
    [I2201]) and forms Delta = rowsum(dO * out) from the given `out`.
  * indices address rows of the packed KV token axis directly; cu_seqlens is
    only used to validate that an index lies in its query's own sequence.
"""
from __future__ import annotations

import math

import numpy as np

D_LATENT = 512
D_TAIL = 64
D_QK = D_LATENT + D_TAIL
SUMEXP_FLOOR = 1e-30            # [PR2079] forward fragment: sumexp floored at 1e-30
LSE_EMPTY = math.log(SUMEXP_FLOOR)  # empty max read as 0, so lse = 0 + ln(1e-30)


def bf16_bits_to_f64(u16: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 (exact)."""
    u32 = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def _as_f64(x: np.ndarray) -> np.ndarray:
    if x.dtype == np.uint16:
        return bf16_bits_to_f64(x)
    return np.asarray(x, dtype=np.float64)


def valid_slots(idx_row: np.ndarray, T: int) -> np.ndarray:
    """[PR2079] item 2 and both fragments: mask = index is a real row; the
    kernel clamps the rest and loads an exact-zero key.  Returns the list J of
    KV rows named by the valid slots, in slot order (duplicates kept)."""
    idx_row = np.asarray(idx_row).reshape(-1).astype(np.int64)
    keep = (idx_row >= 0) & (idx_row < T)
    return idx_row[keep]


def fwd_row(q_t: np.ndarray, kv: np.ndarray, J: np.ndarray, scale: float):
    """Forward for one query token.

    q_t [H, 576] f64, kv [T, 576] f64, J valid KV rows.
    Steps in the order of the [PR2079] forward fragment:
      gather K = kv[J] (576 wide: latent + tail), V = kv[J, :512];
      s = scale * q_t K^T;
      running max m (0 when J is empty), sumexp l = sum exp(s - m);
      floor l at 1e-30; out = (exp(s - m) V) / l;  lse = m + ln l.
    """
    H = q_t.shape[0]
    if J.size == 0:
        m = np.zeros(H)
        l = np.maximum(np.zeros(H), SUMEXP_FLOOR)
        out = np.zeros((H, D_LATENT)) / l[:, None]
        return out, m + np.log(l)
    K = kv[J]                           # [n, 576]
    V = K[:, :D_LATENT]                 # the latent part is also the value
    s = scale * (q_t @ K.T)             # [H, n]
    m = s.max(axis=1)
    e = np.exp(s - m[:, None])
    l = np.maximum(e.sum(axis=1), SUMEXP_FLOOR)
    out = (e @ V) / l[:, None]
    return out, m + np.log(l)


def _row(x: np.ndarray, t: int) -> np.ndarray:
    """Row t of a bf16-bit (uint16) or float array, as float64."""
    return bf16_bits_to_f64(x[t]) if x.dtype == np.uint16 else np.asarray(x[t], dtype=np.float64)


def sparse_mla_fwd(q, kv, indices, scale: float, rows=None):
    """Forward over all tokens, or only over the tokens listed in `rows`.

    q [T, H, 576], kv [T, 1, 576] (or [T, 576]), indices [T, 1, topk] int32;
    q and kv may be bf16 bit patterns (uint16) or floats.
    Returns out [n, H, 512] f64 and lse [n, H] f64, where n = T and row i is
    token i, or n = len(rows) and row i is token rows[i].
    """
    T, H = q.shape[0], q.shape[1]
    kvf = _as_f64(kv).reshape(-1, D_QK)
    idx = np.asarray(indices).reshape(T, -1)
    toks = range(T) if rows is None else [int(t) for t in rows]
    out = np.zeros((len(toks), H, D_LATENT))
    lse = np.zeros((len(toks), H))
    for i, t in enumerate(toks):
        out[i], lse[i] = fwd_row(_row(q, t), kvf, valid_slots(idx[t], kvf.shape[0]), scale)
    return out, lse


def delta(out, dout):
    """Delta[t, h] = sum_d dO[t,h,d] * out[t,h,d] over the 512 value dims."""
    return (_as_f64(dout) * _as_f64(out)).sum(axis=-1)


def bwd_row(q_t, kv, out_t, dout_t, lse_t, J, scale: float):
    """Backward for one query token; returns (dq_t [H,576], J, G [n,576]).

    Follows the [PR2079] backward fragment: gather the masked K/V block,
    recompute P from the saved LSE, form dP = dO V^T, dS = P (dP - Delta),
    dQ = scale dS K, and the per-slot KV gradient G that is scatter-added
    into dKV at the slot's row: G[:, :512] = P^T dO + scale dS^T q[:, :512],
    G[:, 512:] = scale dS^T q[:, 512:] (the tail is only part of K).
    """
    H = q_t.shape[0]
    if J.size == 0:
        return np.zeros((H, D_QK)), J, np.zeros((0, D_QK))
    K = kv[J]
    V = K[:, :D_LATENT]
    s = scale * (q_t @ K.T)                     # [H, n]
    P = np.exp(s - lse_t[:, None])              # probabilities from the saved LSE
    dP = dout_t @ V.T                           # [H, n]
    dlt = (dout_t * out_t).sum(axis=1)          # Delta from the given output
    dS = P * (dP - dlt[:, None])
    dq_t = scale * (dS @ K)                     # [H, 576]
    G = scale * (dS.T @ q_t)                    # [n, 576]
    G[:, :D_LATENT] += P.T @ dout_t
    return dq_t, J, G


def sparse_mla_bwd(q, kv, out, dout, lse, indices, scale: float, rows=None):
    """Backward over all tokens, or only over the tokens listed in `rows`.

    q [T, H, 576] and dout [T, H, 512] are full (bf16 bits or floats);
    out and lse hold one entry per processed token: [T, H, 512] / [T, H]
    when rows is None, else [len(rows), H, 512] / [len(rows), H] aligned
    with rows.  Returns dq [n, H, 576] f64 (same row convention as out) and
    dkv [T, 576] f64: the scatter-add of every processed token's per-slot
    gradient into the row its slot names.  Rows no processed slot names stay
    exactly zero.
    """
    T, H = q.shape[0], q.shape[1]
    kvf = _as_f64(kv).reshape(-1, D_QK)
    idx = np.asarray(indices).reshape(T, -1)
    toks = range(T) if rows is None else [int(t) for t in rows]
    dq = np.zeros((len(toks), H, D_QK))
    dkv = np.zeros((kvf.shape[0], D_QK))
    for i, t in enumerate(toks):
        J = valid_slots(idx[t], kvf.shape[0])
        dq[i], J, G = bwd_row(_row(q, t), kvf, _row(out, i), _row(dout, t),
                              np.asarray(lse[i], dtype=np.float64), J, scale)
        if J.size:
            np.add.at(dkv, J, G)
    return dq, dkv


def check_indices(indices, cu_seqlens) -> int:
    """Count top-k entries that are neither the -1 sentinel nor a row of the
    query's own packed sequence [cu_seqlens[b], cu_seqlens[b+1])."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    T = int(cu[-1])
    idx = np.asarray(indices, dtype=np.int64).reshape(T, -1)
    bad = 0
    for b in range(cu.size - 1):
        s, e = cu[b], cu[b + 1]
        blk = idx[s:e]
        ok = (blk == -1) | ((blk >= s) & (blk < e))
        bad += int((~ok).sum())
    return bad
