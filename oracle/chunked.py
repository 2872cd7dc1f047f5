"""Chunked SSD form in fp64 with a free chunk size (pins chunk-size invariance).

TEST INFRASTRUCTURE ONLY.

The kernelindex page "Mamba chunk scan with segsum" describes the method in
four parts: split the sequence into chunks, an intra-chunk attention-like
block built from segment sums, an inter-chunk state recurrence with
exponential decay, and the sum of diagonal (intra) and off-diagonal (inter)
contributions.  The Modular page "mamba2_ssd_scan" states that this chunked
form is a reformulation of the per-token recurrence and equal to it up to
rounding.  Written out per (sequence, head), with chunks aligned to the
sequence start and, inside a chunk, Acum_i = sum_{k<=i} a_k (a_k = A[h] dt_k):

    CB[i,j]   = C_i . B_j
    Ydiag     = (CB o exp(Acum_i - Acum_j) [j<=i] o dt_j) X
    S_c       = sum_j exp(Acum_last - Acum_j) dt_j x_j (x) B_j     (chunk state)
    Yoff      = exp(Acum_i) C_i . S_prev
    y         = Ydiag + Yoff + D x
    S_prev'   = exp(Acum_last) S_prev + S_c                        (state passing)

This module is independent of the C recurrence; it uses NumPy's cumsum and
matmul.  ``intermediates=True`` also returns every chunk's Acum, S_c and
S_prev so that a GPU stage can be checked on its own.
"""
from __future__ import annotations

import numpy as np


def _widen(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32).astype(np.float64)


def ssd_varlen_fwd(*, x, dt, A, B, C, D, dt_bias, ssm_pool, query_start_loc,
                   has_initial_state, cache_indices, dt_softplus: bool = True,
                   chunk_size: int = 256, intermediates: bool = False):
    X = _widen(x)
    DT = _widen(dt)
    Bf = _widen(B)
    Cf = _widen(C)
    T, H, P = X.shape
    G, N = Bf.shape[1], Bf.shape[2]
    pool = np.array(ssm_pool, dtype=np.float32, copy=True)
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    y = np.zeros((T, H, P))
    inter = []
    Q = int(chunk_size)
    for b in range(qsl.shape[0] - 1):
        t0, t1 = int(qsl[b]), int(qsl[b + 1])
        slot = int(cache_indices[b])
        init = has_initial_state is not None and bool(has_initial_state[b])
        for h in range(H):
            g = h // (H // G)
            S_prev = pool[slot, h].astype(np.float64) if init else np.zeros((P, N))
            for c0 in range(t0, t1, Q):
                c1 = min(c0 + Q, t1)
                v = DT[c0:c1, h] + (0.0 if dt_bias is None else float(dt_bias[h]))
                d = np.logaddexp(0.0, v) if dt_softplus else v
                Acum = np.cumsum(float(A[h]) * d)
                Xc, Bc, Cc = X[c0:c1, h], Bf[c0:c1, g], Cf[c0:c1, g]
                diff = Acum[:, None] - Acum[None, :]
                causal = np.tril(np.ones((c1 - c0, c1 - c0), dtype=bool))
                Lmask = np.where(causal, np.exp(np.where(causal, diff, 0.0)), 0.0)
                Ydiag = ((Cc @ Bc.T) * Lmask * d[None, :]) @ Xc
                Yoff = np.exp(Acum)[:, None] * (Cc @ S_prev.T)
                y[c0:c1, h] = Ydiag + Yoff + (0.0 if D is None else float(D[h])) * Xc
                S_c = (Xc * (np.exp(Acum[-1] - Acum) * d)[:, None]).T @ Bc
                if intermediates:
                    inter.append(dict(seq=b, head=h, start=c0, length=c1 - c0, dt=d,
                                      Acum=Acum, S_chunk=S_c, S_prev=S_prev.copy()))
                S_prev = np.exp(Acum[-1]) * S_prev + S_c
            pool[slot, h] = S_prev.astype(np.float32)
    if intermediates:
        return y, pool, inter
    return y, pool
