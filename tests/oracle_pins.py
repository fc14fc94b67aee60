"""Pins for the oracle: each checks it against something other than itself.

Every ``pin_*`` function takes ``fwd`` (a callable with the oracle's signature,
``fwd(q, k, v, a, beta, h0, cu) -> (out, h_final)``) and returns the largest relative
error it found (or raises AssertionError for a structural failure). The tests assert
each pin passes on the oracle, and that every planted mutant of the oracle fails at
least one of them.

What pins what:
  pin_brute_force       -- the whole recurrence, against an unrolled product of
                           per-token transition matrices (different algebra), d_k != d_v
                           so a transposed state fails
  pin_first_token       -- T = 1 from a zero state has the closed form
                           o = s beta (k.q) v, S = beta k v^T: pins beta, the output
                           scale d_k^-1/2 and reading the state after the write
  pin_gate_closed_form  -- beta = 0, h0 = I: o_t = s exp(G_t) q_t with g = -5 sigmoid(a);
                           a = 0 gives g = -2.5 exactly, a = +inf the bound -5, a = -inf 0
  pin_bound_value       -- a = +inf for 16 tokens decays by exp(-80) ~ 1.8e-35 (printed)
  pin_beta_zero         -- beta = 0: pure decay of h0 (closed form)
  pin_gla_limit         -- beta -> 0 from h0 = 0: o / beta tends to the gated linear
                           attention parallel form (first order in beta)
  pin_delta_exact_write -- beta = 1, |k| = 1: the write makes S_t^T k_t = v_t exactly
  pin_householder       -- g = 0, v = 0, beta = 2, |k| = 1: each step is a reflection,
                           |S|_F is preserved
  pin_projection        -- g = 0, v = 0, beta = 1: |S|_F never increases
"""
from __future__ import annotations

import math

import numpy as np

from oracle.brute import unrolled_forward

G_MIN = -5.0


def rel(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    nr = np.linalg.norm(ref)
    err = np.linalg.norm(x - ref)
    return err / nr if nr > 0 else err


def _rand(rng, lengths, H, dk, dv, *, h0=True, gate_std=2.0):
    N = sum(lengths)
    q = rng.standard_normal((N, H, dk))
    k = rng.standard_normal((N, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((N, H, dv))
    a = gate_std * rng.standard_normal((N, H, dk))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((N, H))))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    hh = 0.3 * rng.standard_normal((len(lengths), H, dk, dv)) if h0 else None
    return q, k, v, a, beta, hh, cu


def pin_brute_force(fwd, dk=3, dv=5, seed=1):
    rng = np.random.default_rng(seed)
    worst = 0.0
    for lengths, gstd in (([7, 0, 12, 1], 2.0), ([9], 6.0), ([5, 5], 0.5)):
        q, k, v, a, beta, h0, cu = _rand(rng, lengths, 2, dk, dv, gate_std=gstd)
        if gstd == 6.0:   # mix of pinned gates: bound, no decay, finite
            a[::3] = np.inf
            a[1::3] = -np.inf
        o, hf = fwd(q, k, v, a, beta, h0, cu)
        ob, hb = unrolled_forward(q, k, v, a, beta, h0, cu, g_min=G_MIN)
        worst = max(worst, rel(o, ob), rel(hf, hb))
    return worst


def pin_first_token(fwd, dk=4, dv=6, seed=2):
    rng = np.random.default_rng(seed)
    q, k, v, a, beta, _, cu = _rand(rng, [1, 1, 1], 3, dk, dv, h0=False)
    o, hf = fwd(q, k, v, a, beta, None, cu)
    s = dk ** -0.5
    o_ref = s * beta[..., None] * np.einsum("nhk,nhk->nh", k, q)[..., None] * v
    S_ref = beta[..., None, None] * np.einsum("nhk,nhv->nhkv", k, v)
    return max(rel(o, o_ref), rel(hf, S_ref))


def _identity_h0(n_seq, H, d):
    return np.broadcast_to(np.eye(d), (n_seq, H, d, d)).copy()


def pin_gate_closed_form(fwd, d=4, T=20, seed=3):
    rng = np.random.default_rng(seed)
    H = 3
    q = rng.standard_normal((T, H, d))
    k = rng.standard_normal((T, H, d))
    v = rng.standard_normal((T, H, d))
    beta = np.zeros((T, H))
    a = np.empty((T, H, d))
    a[:, 0] = 0.0          # g = -2.5 exactly
    a[:, 1] = np.inf       # g = -5, the bound
    a[:, 2] = -np.inf      # g = 0, no decay
    o, _ = fwd(q, k, v, a, beta, _identity_h0(1, H, d), np.array([0, T]))
    t = np.arange(1, T + 1)[:, None]
    s = d ** -0.5
    worst = 0.0
    for h, g in ((0, -2.5), (1, G_MIN), (2, 0.0)):
        worst = max(worst, rel(o[:, h], s * np.exp(g * t) * q[:, h]))
    return worst


def pin_bound_value(fwd, golden):
    """16 tokens with a = +inf: the state decays by exactly exp(16 g_min) = exp(-80)."""
    d, T = 2, 16
    q = np.ones((T, 1, d))
    z = np.zeros((T, 1, d))
    a = np.full((T, 1, d), np.inf)
    o, hf = fwd(q, z, z, a, np.zeros((T, 1)), _identity_h0(1, 1, d), np.array([0, T]))
    decay = hf[0, 0, 0, 0]
    printed = golden["min_cumulative_decay"]
    assert abs(decay / printed["value"] - 1) <= printed["rtol"], decay
    assert abs(math.log(decay) - golden["worst_chunk_log_decay"]["value"]) < 1e-12
    return rel(decay, math.exp(-80.0))


def pin_beta_zero(fwd, dk=3, dv=4, seed=4):
    rng = np.random.default_rng(seed)
    q, k, v, a, beta, h0, cu = _rand(rng, [11, 6], 2, dk, dv)
    beta[:] = 0.0
    o, hf = fwd(q, k, v, a, beta, h0, cu)
    s = dk ** -0.5
    worst = 0.0
    for n in range(2):
        t0, t1 = cu[n], cu[n + 1]
        for h in range(2):
            G = np.cumsum(G_MIN / (1.0 + np.exp(-a[t0:t1, h])), axis=0)
            o_ref = s * np.einsum("kv,tk->tv", h0[n, h], np.exp(G) * q[t0:t1, h])
            worst = max(worst, rel(o[t0:t1, h], o_ref))
            worst = max(worst, rel(hf[n, h], np.exp(G[-1])[:, None] * h0[n, h]))
    return worst


def pin_gla_limit(fwd, dk=4, dv=3, T=24, eps=1e-7, seed=5):
    rng = np.random.default_rng(seed)
    q, k, v, a, _, _, cu = _rand(rng, [T], 2, dk, dv, h0=False)
    beta = np.full((T, 2), eps)
    o, _ = fwd(q, k, v, a, beta, None, cu)
    s = dk ** -0.5
    worst = 0.0
    for h in range(2):
        G = np.cumsum(G_MIN / (1.0 + np.exp(-a[:, h])), axis=0)
        ref = np.zeros((T, dv))
        for t in range(T):
            for j in range(t + 1):
                ref[t] += s * np.dot(q[t, h] * np.exp(G[t] - G[j]), k[j, h]) * v[j, h]
        worst = max(worst, rel(o[:, h] / eps, ref))
    return worst   # O(eps * T) by construction


def pin_delta_exact_write(fwd, dk=5, dv=3, T=17, seed=6):
    rng = np.random.default_rng(seed)
    q, k, v, a, beta, h0, cu = _rand(rng, [T], 2, dk, dv)
    beta[:] = 1.0
    q = k.copy()          # o_t = s S_t^T k_t, which the write sets to s v_t
    o, _ = fwd(q, k, v, a, beta, h0, cu)
    return rel(o, dk ** -0.5 * v)


def pin_householder(fwd, d=4, T=13, seed=7):
    rng = np.random.default_rng(seed)
    q, k, v, a, beta, h0, cu = _rand(rng, [T], 2, d, d)
    v[:] = 0.0
    a[:] = -np.inf
    beta[:] = 2.0
    worst = 0.0
    for L in (1, 5, T):
        _, hf = fwd(q[:L], k[:L], v[:L], a[:L], beta[:L], h0, np.array([0, L]))
        for h in range(2):
            worst = max(worst, abs(np.linalg.norm(hf[0, h]) / np.linalg.norm(h0[0, h]) - 1))
    return worst


def pin_projection(fwd, d=4, T=12, seed=8):
    rng = np.random.default_rng(seed)
    q, k, v, a, beta, h0, cu = _rand(rng, [T], 1, d, d)
    v[:] = 0.0
    a[:] = -np.inf
    beta[:] = 1.0
    norms = [np.linalg.norm(h0[0, 0])]
    for L in range(1, T + 1):
        _, hf = fwd(q[:L], k[:L], v[:L], a[:L], beta[:L], h0, np.array([0, L]))
        norms.append(np.linalg.norm(hf[0, 0]))
    increase = max(0.0, max(b - a_ for a_, b in zip(norms, norms[1:])))
    # every step must strictly shrink a generic state (k not orthogonal to it)
    assert norms[-1] < norms[0]
    return increase


PINS = {
    "brute_force": (pin_brute_force, 1e-12),
    "first_token": (pin_first_token, 1e-13),
    "gate_closed_form": (pin_gate_closed_form, 1e-13),
    "beta_zero": (pin_beta_zero, 1e-13),
    "gla_limit": (pin_gla_limit, 1e-4),
    "delta_exact_write": (pin_delta_exact_write, 1e-12),
    "householder": (pin_householder, 1e-12),
    "projection": (pin_projection, 1e-12),
}
