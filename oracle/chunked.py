"""fp64 NumPy restatement of the 16-token chunked algebra.

TEST INFRASTRUCTURE ONLY (see the package docstring). This is not the oracle: the
oracle is the token-by-token recurrence in ``kda_oracle.c``. This module exists to pin
that the chunked form -- the form the GPU library implements -- reaches exactly the
recurrence's result, at fp64, including partial last chunks and gates pinned to the
bound.

Per chunk of L <= C = 16 tokens of one head, with start state S (d_k x d_v):

  g   = g_min * sigmoid(a)                     bounded log-decay per key channel
        ["Demystifying Trillion-Parameter MoE Models", Breakthrough 1 §2]
  G_r = sum_{i<=r} g_i                          cumulative log-decay, reset per chunk;
        the pairwise scale between positions r >= j is exp(G_r - G_j)
        ["From Numerical Stability to Load Balancing", §2.1]
  Q~ = Q*exp(G), K~ = K*exp(G), K^ = K*exp(-G), K' = K*exp(G_L - G)
        exp(+-G) stays within exp(+-80) because 16 * (-5) = -80
        ["From Numerical Stability to Load Balancing", §2.2]
  A  = strict_lower(diag(beta) K~ K^^T)         intra-chunk (diagonal tile) products
  T  = (I + A)^-1                               unit lower triangular
  W  = T diag(beta) K~,   U~ = T diag(beta) V
  P  = lower(Q~ K^^T)                           diagonal included
  U  = U~ - W S                                 needs the state: serial across chunks
  O  = scale (Q~ S + P U)
  S <- Diag(exp G_L) S + K'^T U                 "inter-chunk computation proceeds
        serially through state recurrence" [same page, §2.1]

Rows past L (a partial last chunk) behave as q = k = v = 0, beta = 0, g = 0.
Derivation: unrolling the recurrence over a chunk gives
S_r = Diag(Gamma_r) S_0 + sum_{j<=r} Diag(Gamma_r / Gamma_j) k_j u_j^T with
u_j = beta_j (v_j - (Diag(gamma_j) S_{j-1})^T k_j); collecting the u_j gives
(I + A) U = diag(beta) (V - K~ S_0), which is the U line above.
"""
from __future__ import annotations

import numpy as np

C_DEFAULT = 16


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def inverse_unit_lower(A: np.ndarray, method: str = "solve") -> np.ndarray:
    """(I + A)^-1 for strictly lower-triangular A (n x n).

    ``solve``: forward substitution, row r of T is e_r - sum_{j<r} A[r, j] T[j, :].
    ``doubling``: A is nilpotent (A^n = 0 for n <= 16), so
    (I + A)^-1 = (I - A)(I + A^2)(I + A^4)(I + A^8) exactly.
    """
    n = A.shape[0]
    I = np.eye(n)
    if method == "solve":
        T = np.zeros_like(A)
        for r in range(n):
            T[r] = I[r] - A[r, :r] @ T[:r]
        return T
    if method == "doubling":
        assert n <= 16
        P = I - A
        A2 = A @ A
        P = P @ (I + A2)
        A4 = A2 @ A2
        P = P @ (I + A4)
        A8 = A4 @ A4
        return P @ (I + A8)
    raise ValueError(method)


def chunk_step(q, k, v, a, beta, S, *, g_min=-5.0, scale=None, inverse="solve"):
    """One chunk (rows = tokens, already zero-padded past L). Returns (O, S_next)."""
    C, dk = q.shape
    if scale is None:
        scale = dk ** -0.5
    g = g_min * sigmoid(a)
    G = np.cumsum(g, axis=0)
    GL = G[-1]
    Qt = q * np.exp(G)
    Kt = k * np.exp(G)
    Kh = k * np.exp(-G)
    Kp = k * np.exp(GL[None, :] - G)
    A = np.tril(beta[:, None] * (Kt @ Kh.T), -1)
    T = inverse_unit_lower(A, inverse)
    W = T @ (beta[:, None] * Kt)
    Ut = T @ (beta[:, None] * v)
    P = np.tril(Qt @ Kh.T)
    U = Ut - W @ S
    O = scale * (Qt @ S + P @ U)
    S_next = np.exp(GL)[:, None] * S + Kp.T @ U
    return O, S_next


def chunked_forward(q, k, v, a, beta, h0=None, cu_seqlens=None, *, g_min=-5.0,
                    scale=None, C=C_DEFAULT, inverse="solve"):
    """Chunked fp64 forward over packed sequences; same shapes as the oracle."""
    q, k, v, a, beta = (np.asarray(t, dtype=np.float64) for t in (q, k, v, a, beta))
    N, H, dk = q.shape
    dv = v.shape[2]
    cu = np.array([0, N]) if cu_seqlens is None else np.asarray(cu_seqlens, dtype=np.int64)
    n_seq = len(cu) - 1
    out = np.zeros((N, H, dv))
    hf = np.zeros((n_seq, H, dk, dv))
    for n in range(n_seq):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        for h in range(H):
            S = np.zeros((dk, dv)) if h0 is None else np.array(h0[n, h], dtype=np.float64)
            for c0 in range(t0, t1, C):
                L = min(C, t1 - c0)
                qc = np.zeros((C, dk)); kc = np.zeros((C, dk)); vc = np.zeros((C, dv))
                # padded rows: a = -inf gives g = -0, so exp(g) = 1 (no decay)
                ac = np.full((C, dk), -np.inf); bc = np.zeros(C)
                qc[:L] = q[c0:c0 + L, h]; kc[:L] = k[c0:c0 + L, h]; vc[:L] = v[c0:c0 + L, h]
                ac[:L] = a[c0:c0 + L, h]; bc[:L] = beta[c0:c0 + L, h]
                O, S = chunk_step(qc, kc, vc, ac, bc, S, g_min=g_min, scale=scale,
                                  inverse=inverse)
                out[c0:c0 + L, h] = O[:L]
            hf[n, h] = S
    return out, hf


# ---------------------------------------------------------------------------------
# 64-token serial steps built from the 16-token bounded tiles.
#
# The serial state recurrence can advance B = 64 tokens per step while every
# exponential stays inside the bound of one 16-token tile: the pairwise factor between
# positions r (in tile I) and j (in an earlier tile J) of the step factors as
#   exp(G_r - G_j) = exp(G^I_r) * prod_{J<m<I} gamma_m * exp(G^J_end - G^J_j),
# with G^I the cumulative log-decay restarted at tile I and gamma_m = exp(G^m_end). The
# first and last factors are the tile's own Q~ / K~ and K' scalings (both <= 1), the
# middle one a product of tile decays (<= 1); only the diagonal tiles use
# K^ = K exp(-G^I) <= exp(80) ("From Numerical Stability to Load Balancing", §2.2-2.3:
# the 16-token tile is where the bound is needed). Per step, with the B x B matrices
#   A   strict_lower(diag(beta) [pairwise K K^T with the factors above])
#   P   lower([pairwise Q K^T with the same factors])
#   TB  (I + A)^-1 diag(beta)
#   W   TB K~B,      K~B = K exp(G^B),   Q~B = Q exp(G^B)   (G^B: restarted at the step)
#   Q'  Q~B - P W,   P' = P TB,          K'B = K exp(G^B_end - G^B)
# the step is
#   U = TB V - W S;  O = scale (P' V + Q' S);  S <- Diag(exp G^B_end) S + K'B^T U.
# The output line is scale (Q~B S + P U) with U substituted, so the output depends on
# the start state and V only (not on U).
# ---------------------------------------------------------------------------------

def block_step(q, k, v, a, beta, S, *, g_min=-5.0, scale=None, tile=C_DEFAULT, form="qs_pu"):
    """One serial step over B = q.shape[0] tokens (a multiple of ``tile``), rows past the
    sequence already padded (q = k = v = 0, beta = 0, a = -inf). Returns (O, S_next).
    ``form`` picks one of two equal ways of writing the output: "qs_pu" =
    scale (Q~B S + P U), "pv_qs" = scale (P' V + Q' S) with P' = P TB, Q' = Q~B - P W."""
    B, dk = q.shape
    if scale is None:
        scale = dk ** -0.5
    nt = B // tile
    assert nt * tile == B
    g = g_min * sigmoid(a)
    # per tile: restarted cumulative log-decay and its scaled operands
    Qt, Kt, Kh, Kp, gam = [], [], [], [], []
    for I in range(nt):
        sl = slice(I * tile, (I + 1) * tile)
        G = np.cumsum(g[sl], axis=0)
        GL = G[-1]
        Qt.append(q[sl] * np.exp(G))
        Kt.append(k[sl] * np.exp(G))
        Kh.append(k[sl] * np.exp(-G))
        Kp.append(k[sl] * np.exp(GL[None, :] - G))
        gam.append(np.exp(GL))
    A = np.zeros((B, B))
    P = np.zeros((B, B))
    for I in range(nt):
        rI = slice(I * tile, (I + 1) * tile)
        bI = beta[rI][:, None]
        A[rI, rI] = np.tril(bI * (Kt[I] @ Kh[I].T), -1)
        P[rI, rI] = np.tril(Qt[I] @ Kh[I].T)
        for J in range(I):
            rJ = slice(J * tile, (J + 1) * tile)
            mid = np.ones(dk)
            for m in range(J + 1, I):
                mid = mid * gam[m]
            A[rI, rJ] = bI * ((Kt[I] * mid) @ Kp[J].T)
            P[rI, rJ] = (Qt[I] * mid) @ Kp[J].T
    TB = inverse_unit_lower(A, "solve") @ np.diag(beta)
    # step-level operands: decay from the step start to each tile start (<= 1)
    KtB, QtB, KpB = [], [], []
    pre = np.ones(dk)
    for I in range(nt):
        post = np.ones(dk)
        for m in range(I + 1, nt):
            post = post * gam[m]
        KtB.append(Kt[I] * pre)
        QtB.append(Qt[I] * pre)
        KpB.append(Kp[I] * post)
        pre = pre * gam[I]
    gamB = pre
    KtB, QtB, KpB = (np.concatenate(x, axis=0) for x in (KtB, QtB, KpB))
    W = TB @ KtB
    U = TB @ v - W @ S
    if form == "qs_pu":
        O = scale * (QtB @ S + P @ U)
    elif form == "pv_qs":
        Qp = QtB - P @ W
        Pp = P @ TB
        O = scale * (Pp @ v + Qp @ S)
    else:
        raise ValueError(f"unknown output form {form!r}")
    S_next = gamB[:, None] * S + KpB.T @ U
    return O, S_next


def block_forward(q, k, v, a, beta, h0=None, cu_seqlens=None, *, g_min=-5.0, scale=None,
                  B=64, tile=C_DEFAULT):
    """fp64 forward over packed sequences in serial steps of B tokens (see block_step)."""
    q, k, v, a, beta = (np.asarray(t, dtype=np.float64) for t in (q, k, v, a, beta))
    N, H, dk = q.shape
    dv = v.shape[2]
    cu = np.array([0, N]) if cu_seqlens is None else np.asarray(cu_seqlens, dtype=np.int64)
    n_seq = len(cu) - 1
    out = np.zeros((N, H, dv))
    hf = np.zeros((n_seq, H, dk, dv))
    for n in range(n_seq):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        for h in range(H):
            S = np.zeros((dk, dv)) if h0 is None else np.array(h0[n, h], dtype=np.float64)
            for c0 in range(t0, t1, B):
                L = min(B, t1 - c0)
                qc = np.zeros((B, dk)); kc = np.zeros((B, dk)); vc = np.zeros((B, dv))
                ac = np.full((B, dk), -np.inf); bc = np.zeros(B)
                qc[:L] = q[c0:c0 + L, h]; kc[:L] = k[c0:c0 + L, h]; vc[:L] = v[c0:c0 + L, h]
                ac[:L] = a[c0:c0 + L, h]; bc[:L] = beta[c0:c0 + L, h]
                O, S = block_step(qc, kc, vc, ac, bc, S, g_min=g_min, scale=scale, tile=tile)
                out[c0:c0 + L, h] = O[:L]
            hf[n, h] = S
    return out, hf
