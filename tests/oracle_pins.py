"""Checks that pin the fp64 oracle to things other than itself.

Each check takes the oracle module as an argument and returns the largest
error it saw, so the same checks can be re-run against deliberately broken
copies of the oracle (tests/test_oracle_pins.py plants those mistakes on the
CPU and confirms that some check catches each one).

Pins used:
  * a library routine: on dense causal inputs (every query lists exactly the
    keys of its own sequence up to itself) sparse attention reduces to causal
    multi-query attention, which torch's scaled_dot_product_attention computes
    in fp64 on the CPU; torch.autograd gives the gradients of <dO, O>.
  * calculus: central finite differences of L = <dO, O(q, kv)>.
  * closed forms: a single valid slot, and n slots naming identical rows.
  * invariants stated by the pages (miles PR #2079 summary, implementation
    breakdown items 2-3): padding slots contribute exactly zero, all-padding
    rows give an exactly-zero output and a finite LSE, and the clamped
    padding write to dKV adds nothing.
"""
from __future__ import annotations

import math

import numpy as np

D = 512
DQK = 576


def _dense_causal_case(seed: int, seqlens=(40, 24), H: int = 4, topk: int = 64, pad_noise=True):
    rng = np.random.default_rng(seed)
    T = sum(seqlens)
    q = rng.standard_normal((T, H, DQK))
    kv = rng.standard_normal((T, DQK))
    dout = rng.standard_normal((T, H, D))
    idx = np.full((T, topk), -1, dtype=np.int64)
    allowed = np.zeros((T, T), dtype=bool)
    s0 = 0
    for L in seqlens:
        for p in range(L):
            t = s0 + p
            row = np.full(topk, -1, dtype=np.int64)
            row[: p + 1] = np.arange(s0, t + 1)
            if pad_noise:
                rng.shuffle(row)            # padding interleaved with real slots
            idx[t] = row
            allowed[t, s0: t + 1] = True
        s0 += L
    return q, kv, dout, idx.astype(np.int32), allowed


def pin_sdpa(orc, seed: int = 1) -> float:
    """Max relative error of the oracle against torch SDPA (fp64, CPU)."""
    import torch
    import torch.nn.functional as F

    q, kv, dout, idx, allowed = _dense_causal_case(seed)
    T, H, _ = q.shape
    scale = 1.0 / math.sqrt(DQK)
    out, lse = orc.sparse_mla_fwd(q, kv, idx, scale)
    dq, dkv = orc.sparse_mla_bwd(q, kv, out, dout, lse, idx, scale)

    tq = torch.tensor(q, dtype=torch.float64).permute(1, 0, 2).unsqueeze(0).requires_grad_(True)
    tkv = torch.tensor(kv, dtype=torch.float64).requires_grad_(True)
    K = tkv.unsqueeze(0).unsqueeze(0).expand(1, H, T, DQK)
    V = tkv[:, :D].unsqueeze(0).unsqueeze(0).expand(1, H, T, D)
    mask = torch.tensor(allowed)
    o = F.scaled_dot_product_attention(tq, K, V, attn_mask=mask, scale=scale)
    logits = (tq @ K.transpose(-1, -2)) * scale
    lse_ref = torch.logsumexp(logits.masked_fill(~mask, float("-inf")), dim=-1)
    tdo = torch.tensor(dout, dtype=torch.float64).permute(1, 0, 2).unsqueeze(0)
    (o * tdo).sum().backward()

    out_ref = o[0].permute(1, 0, 2).detach().numpy()
    lse_ref = lse_ref[0].permute(1, 0).detach().numpy()
    dq_ref = tq.grad[0].permute(1, 0, 2).numpy()
    dkv_ref = tkv.grad.numpy()

    def rel(a, b):
        return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))

    return max(rel(out, out_ref), rel(lse, lse_ref), rel(dq, dq_ref), rel(dkv, dkv_ref))


def _loss(orc, q, kv, dout, idx, scale):
    out, _ = orc.sparse_mla_fwd(q, kv, idx, scale)
    return float((out * dout).sum())


def pin_finite_differences(orc, seed: int = 2, n_coords: int = 10) -> float:
    """Max relative error of the oracle gradient against central differences
    of L = <dO, O>, on random q and kv coordinates (latent and tail)."""
    rng = np.random.default_rng(seed)
    T, H, topk = 10, 2, 8
    q = rng.standard_normal((T, H, DQK)) * 2.0
    kv = rng.standard_normal((T, DQK))
    dout = rng.standard_normal((T, H, D))
    idx = rng.integers(-1, T, size=(T, topk)).astype(np.int32)   # duplicates and -1 allowed
    idx[3] = -1                                                 # one all-padding row
    scale = 1.0 / math.sqrt(DQK)
    out, lse = orc.sparse_mla_fwd(q, kv, idx, scale)
    dq, dkv = orc.sparse_mla_bwd(q, kv, out, dout, lse, idx, scale)

    h = 1e-5
    worst = 0.0
    gscale = max(np.abs(dq).max(), np.abs(dkv).max())
    for _ in range(n_coords):
        for which in ("q_lat", "q_tail", "kv_lat", "kv_tail"):
            if which.startswith("q"):
                t, hh = rng.integers(T), rng.integers(H)
                d = rng.integers(0, D) if which == "q_lat" else rng.integers(D, DQK)
                a = q.copy(); a[t, hh, d] += h
                b = q.copy(); b[t, hh, d] -= h
                fd = (_loss(orc, a, kv, dout, idx, scale) - _loss(orc, b, kv, dout, idx, scale)) / (2 * h)
                an = dq[t, hh, d]
            else:
                named = np.unique(idx[(idx >= 0) & (idx < T)])
                r = rng.choice(named)
                d = rng.integers(0, D) if which == "kv_lat" else rng.integers(D, DQK)
                a = kv.copy(); a[r, d] += h
                b = kv.copy(); b[r, d] -= h
                fd = (_loss(orc, q, a, dout, idx, scale) - _loss(orc, q, b, dout, idx, scale)) / (2 * h)
                an = dkv[r, d]
            worst = max(worst, abs(fd - an) / gscale)
    return worst


def pin_closed_forms(orc, seed: int = 3) -> float:
    """Largest deviation from closed forms:
    * one valid slot j: out = kv[j,:512], lse = scale q.kv[j], dq = 0,
      dkv[j,:512] = sum_h dO, dkv[j,512:] = 0;
    * n slots on identical rows (distinct rows with equal content, and one row
      repeated): out = v, lse = scale q.v + ln n."""
    rng = np.random.default_rng(seed)
    T, H, topk = 16, 3, 8
    scale = 0.125
    q = rng.standard_normal((T, H, DQK))
    kv = rng.standard_normal((T, DQK))
    dout = rng.standard_normal((T, H, D))
    idx = np.full((T, topk), -1, dtype=np.int32)
    err = 0.0
    # one valid slot: token 5 -> row 9, slot position 6
    idx[5, 6] = 9
    out, lse = orc.sparse_mla_fwd(q, kv, idx, scale)
    dq, dkv = orc.sparse_mla_bwd(q, kv, out[[5]], dout, lse[[5]], idx, scale, rows=[5])
    err = max(err, np.abs(out[5] - kv[9, :D][None]).max())
    err = max(err, np.abs(lse[5] - scale * (q[5] @ kv[9])).max())
    err = max(err, np.abs(dq[0]).max())
    err = max(err, np.abs(dkv[9, :D] - dout[5].sum(0)).max())
    err = max(err, np.abs(dkv[9, D:]).max())
    # identical rows: rows 1, 4, 11 share content; token 7 lists them; token 8 lists row 2 three times
    kv2 = kv.copy()
    kv2[4] = kv2[1]
    kv2[11] = kv2[1]
    idx2 = np.full((T, topk), -1, dtype=np.int32)
    idx2[7, [0, 3, 7]] = [1, 4, 11]
    idx2[8, [1, 2, 5]] = [2, 2, 2]
    out2, lse2 = orc.sparse_mla_fwd(q, kv2, idx2, scale)
    err = max(err, np.abs(out2[7] - kv2[1, :D][None]).max())
    err = max(err, np.abs(lse2[7] - (scale * (q[7] @ kv2[1]) + math.log(3))).max())
    err = max(err, np.abs(out2[8] - kv2[2, :D][None]).max())
    err = max(err, np.abs(lse2[8] - (scale * (q[8] @ kv2[2]) + math.log(3))).max())
    return float(err)


def pin_padding_invariants(orc, seed: int = 4) -> float:
    """0.0 when every padding invariant holds exactly, else a positive number.

    * padding slots (-1, T, -7, INT32_MAX) interleaved into a row change
      nothing, bit for bit, in out, lse, dq or dkv;
    * an all-padding row gives out == 0, lse == ln(1e-30), dq == 0;
    * rows no slot names get dkv == 0 exactly."""
    rng = np.random.default_rng(seed)
    T, H, topk = 24, 4, 16
    scale = 1.0 / math.sqrt(DQK)
    q = rng.standard_normal((T, H, DQK))
    kv = rng.standard_normal((T, DQK))
    dout = rng.standard_normal((T, H, D))
    compact = np.full((T, topk), -1, dtype=np.int32)
    noisy = np.full((T, topk), -1, dtype=np.int32)
    junk = np.array([-1, T, -7, 2**31 - 1, T + 3], dtype=np.int64)
    for t in range(T):
        n = rng.integers(0, 9) if t not in (2, 17) else 0
        real = rng.choice(np.arange(0, 20), size=n, replace=False)   # rows 20..23 never named
        compact[t, :n] = real
        slots = np.sort(rng.choice(topk, size=n, replace=False))
        noisy[t] = rng.choice(junk, size=topk)
        noisy[t, slots] = real
    bad = 0.0
    o1, l1 = orc.sparse_mla_fwd(q, kv, compact, scale)
    o2, l2 = orc.sparse_mla_fwd(q, kv, noisy, scale)
    bad += float(np.any(o1 != o2)) + float(np.any(l1 != l2))
    g1 = orc.sparse_mla_bwd(q, kv, o1, dout, l1, compact, scale)
    g2 = orc.sparse_mla_bwd(q, kv, o2, dout, l2, noisy, scale)
    bad += float(np.any(g1[0] != g2[0])) + float(np.any(g1[1] != g2[1]))
    for t in (2, 17):
        bad += float(np.any(o1[t] != 0.0))
        bad += float(np.any(l1[t] != math.log(1e-30)))
        bad += float(np.any(g1[0][t] != 0.0))
    bad += float(np.any(g1[1][20:] != 0.0))
    for arr in (o1, l1, g1[0], g1[1]):
        bad += float(not np.all(np.isfinite(arr)))
    return bad


def pin_sum_rules(orc, seed: int = 5) -> float:
    """Sum rules that follow from sum_j dS = 0 per (token, head) when `out` is
    the exact output:  sum over kv rows of dkv[:, 512:] = 0 and
    sum over kv rows of dkv[:, :512] = sum over non-empty (t, h) of dO[t, h];
    plus max_j s_j <= lse <= max_j s_j + ln(n_valid).  Large logits
    (q ~ N(0, 8^2)) exercise the exponent range."""
    rng = np.random.default_rng(seed)
    T, H, topk = 32, 4, 12
    scale = 1.0 / math.sqrt(DQK)
    q = rng.standard_normal((T, H, DQK)) * 8.0
    kv = rng.standard_normal((T, DQK))
    dout = rng.standard_normal((T, H, D))
    idx = rng.integers(-1, T, size=(T, topk)).astype(np.int32)
    idx[[0, 9]] = -1
    out, lse = orc.sparse_mla_fwd(q, kv, idx, scale)
    dq, dkv = orc.sparse_mla_bwd(q, kv, out, dout, lse, idx, scale)
    nonempty = np.array([np.any((r >= 0) & (r < T)) for r in idx])
    ref_lat = dout[nonempty].sum(axis=(0, 1))
    err = np.abs(dkv[:, D:].sum(0)).max() / np.abs(dkv[:, D:]).max()
    err = max(err, np.abs(dkv[:, :D].sum(0) - ref_lat).max() / np.abs(ref_lat).max())
    for t in range(T):
        J = idx[t][(idx[t] >= 0) & (idx[t] < T)].astype(np.int64)
        if J.size == 0:
            continue
        smax = (scale * q[t] @ kv[J].T).max(axis=1)
        lo = smax - 1e-9
        hi = smax + math.log(J.size) + 1e-9
        if np.any(lse[t] < lo) or np.any(lse[t] > hi):
            err = max(err, 1.0)
    if not all(np.all(np.isfinite(a)) for a in (out, lse, dq, dkv)):
        err = max(err, 1.0)
    return float(err)


def pin_delta_identity(orc, seed: int = 6) -> float:
    """Delta = rowsum(dO * O) equals sum_j P_j dP_j when O is the exact output
    (the identity that lets the backward form Delta from the saved output)."""
    rng = np.random.default_rng(seed)
    T, H, topk = 12, 3, 10
    scale = 1.0 / math.sqrt(DQK)
    q = rng.standard_normal((T, H, DQK))
    kv = rng.standard_normal((T, DQK))
    dout = rng.standard_normal((T, H, D))
    idx = rng.integers(0, T, size=(T, topk)).astype(np.int32)
    out, lse = orc.sparse_mla_fwd(q, kv, idx, scale)
    dl = orc.delta(out, dout)
    err = 0.0
    for t in range(T):
        J = idx[t].astype(np.int64)
        P = np.exp(scale * q[t] @ kv[J].T - lse[t][:, None])
        dP = dout[t] @ kv[J, :D].T
        err = max(err, np.abs((P * dP).sum(1) - dl[t]).max())
    return float(err)


def pin_check_indices(orc) -> float:
    """Hand-counted example: two sequences [0,3) and [3,5), topk=3."""
    cu = np.array([0, 3, 5], dtype=np.int32)
    idx = np.array([
        [0, -1, -1],     # ok
        [1, 0, 3],       # 3 is in the other sequence -> 1 bad
        [2, 5, -1],      # 5 == T -> 1 bad
        [3, 4, -7],      # -7 -> 1 bad
        [0, 4, -1],      # 0 is in the other sequence -> 1 bad
    ], dtype=np.int32)
    return float(abs(orc.check_indices(idx, cu) - 4))
