"""fp64 NumPy unrolled (transition-matrix) form of the recurrence, for tiny inputs.

TEST INFRASTRUCTURE ONLY (see the package docstring).

One token of the recurrence is an affine map of the state,
    S_t = M_t S_{t-1} + beta_t k_t v_t^T,   M_t = (I - beta_t k_t k_t^T) Diag(exp g_t),
so, by induction,
    S_t = (M_t ... M_1) h0 + sum_{j<=t} (M_t ... M_{j+1}) beta_j k_j v_j^T.
This module forms those products explicitly, from scratch for every t (O(T^2 d_k^3)),
and reads o_t = scale * S_t^T q_t. It shares no loop structure with the oracle: the
oracle never forms a d_k x d_k matrix.
"""
from __future__ import annotations

import numpy as np


def unrolled_forward(q, k, v, a, beta, h0=None, cu_seqlens=None, *, g_min=-5.0,
                     scale=None):
    q, k, v, a, beta = (np.asarray(t, dtype=np.float64) for t in (q, k, v, a, beta))
    N, H, dk = q.shape
    dv = v.shape[2]
    if scale is None:
        scale = dk ** -0.5
    cu = np.array([0, N]) if cu_seqlens is None else np.asarray(cu_seqlens, dtype=np.int64)
    n_seq = len(cu) - 1
    out = np.zeros((N, H, dv))
    hf = np.zeros((n_seq, H, dk, dv))
    I = np.eye(dk)
    for n in range(n_seq):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        for h in range(H):
            S0 = np.zeros((dk, dv)) if h0 is None else np.asarray(h0[n, h], dtype=np.float64)
            gam = np.exp(g_min / (1.0 + np.exp(-a[t0:t1, h])))   # [L, dk]
            M = [(I - beta[t, h] * np.outer(k[t, h], k[t, h])) @ np.diag(gam[t - t0])
                 for t in range(t0, t1)]
            S_t = S0
            for t in range(t0, t1):
                prod = I.copy()
                for i in range(t, t0 - 1, -1):        # M_t ... M_{t0}
                    prod = prod @ M[i - t0]
                S_t = prod @ S0
                for j in range(t0, t + 1):
                    Pj = I.copy()
                    for i in range(t, j, -1):         # M_t ... M_{j+1}
                        Pj = Pj @ M[i - t0]
                    S_t = S_t + Pj @ (beta[j, h] * np.outer(k[j, h], v[j, h]))
                out[t, h] = scale * S_t.T @ q[t, h]
            hf[n, h] = S_t
    return out, hf
