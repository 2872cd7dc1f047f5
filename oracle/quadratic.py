"""Brute-force quadratic form of the SSD scan (pins the oracle on small inputs).

TEST INFRASTRUCTURE ONLY.

Unrolling the per-token recurrence of the Modular page "mamba2_ssd_scan"
("Per-token recurrence") from an initial state S0 gives, per sequence and head,

    S_i    = exp(sum_{k<=i} a_k) S0 + sum_{j<=i} exp(sum_{k=j+1..i} a_k) dt_j x_j (x) B_j
    y_i    = C_i . S_i + D x_i
           = sum_{j<=i} M[i,j] x_j + exp(sum_{k<=i} a_k) C_i . S0 + D x_i,
    M[i,j] = (C_i . B_j) exp(sum_{k=j+1..i} a_k) dt_j     (j <= i, else 0)

with a_k = A[h] dt_k.  This is the "attention-like" matrix the kernelindex
page "Mamba chunk scan with segsum" refers to, over a whole sequence instead
of one chunk.  Every segment sum is added up term by term along its row
(no differences of prefix sums), C B^T is one fp64 matmul, and softplus is
NumPy's logaddexp(0, v): none of this shares a step with the C recurrence.
Cost is O(L^2) per (sequence, head): keep L to a few hundred.
"""
from __future__ import annotations

import numpy as np


def _widen(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32).astype(np.float64)


def segsum_direct(a: np.ndarray) -> np.ndarray:
    """seg[i, j] = sum_{k=j+1..i} a_k for j <= i (0 on the diagonal), -inf above."""
    L = a.shape[0]
    seg = np.full((L, L), -np.inf)
    for i in range(L):
        seg[i, i] = 0.0
        if i > 0:
            # running sums a_i, a_i + a_{i-1}, ..., a_i + ... + a_1
            seg[i, :i] = np.cumsum(a[i:0:-1])[::-1]
    return seg


def ssd_sequence(xs, d, Ah, Bs, Cs, Dh, S0):
    """One (sequence, head): xs (L,P), d (L,), Bs/Cs (L,N), S0 (P,N) -> (y, S_L)."""
    a = Ah * d
    L = a.shape[0]
    seg = segsum_direct(a)
    M = (Cs @ Bs.T) * np.exp(seg) * d[None, :]
    decay_from_start = np.exp(np.cumsum(a))           # exp(sum_{k<=i} a_k)
    y = M @ xs + decay_from_start[:, None] * (Cs @ S0.T) + Dh * xs
    total = a.sum()
    # exp(sum_{k=j+1..L-1} a_k): the last row of the segment-sum matrix
    tail = np.exp(seg[L - 1, :]) if L > 0 else np.zeros(0)
    S = (xs * (tail * d)[:, None]).T @ Bs + np.exp(total) * S0
    return y, S


def ssd_varlen_fwd(*, x, dt, A, B, C, D, dt_bias, ssm_pool, query_start_loc,
                   has_initial_state, cache_indices, dt_softplus: bool = True):
    """Same interface and outputs as ``recurrence.ssd_varlen_fwd`` (fp64 y,
    fp32 updated copy of the pool)."""
    X = _widen(x)
    DT = _widen(dt)
    Bf = _widen(B)
    Cf = _widen(C)
    T, H, P = X.shape
    G, N = Bf.shape[1], Bf.shape[2]
    pool = np.array(ssm_pool, dtype=np.float32, copy=True)
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    y = np.zeros((T, H, P))
    for b in range(qsl.shape[0] - 1):
        t0, t1 = int(qsl[b]), int(qsl[b + 1])
        slot = int(cache_indices[b])
        init = has_initial_state is not None and bool(has_initial_state[b])
        for h in range(H):
            g = h // (H // G)
            v = DT[t0:t1, h] + (0.0 if dt_bias is None else float(dt_bias[h]))
            d = np.logaddexp(0.0, v) if dt_softplus else v
            S0 = pool[slot, h].astype(np.float64) if init else np.zeros((P, N))
            yb, S = ssd_sequence(X[t0:t1, h], d, float(A[h]), Bf[t0:t1, g], Cf[t0:t1, g],
                                 0.0 if D is None else float(D[h]), S0)
            y[t0:t1, h] = yb
            pool[slot, h] = S.astype(np.float32)
    return y, pool
