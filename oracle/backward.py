"""fp64 gradients of the recurrence by reverse-mode automatic differentiation.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages define the forward operation only; its backward pass is by definition the
gradient of that forward. The function differentiated here is the token-by-token
recurrence, the same definition the C oracle (``kda_oracle.c``) implements:

    g_t = g_min * sigmoid(a_t)                      per key channel, g_min = -5
    S   <- Diag(exp g_t) S
    S   <- S + beta_t k_t (v_t - S^T k_t)^T
    o_t  = scale * S^T q_t                          scale = d_k^-1/2

("From Numerical Stability to Load Balancing", §2.1-2.2; "Demystifying
Trillion-Parameter MoE Models", Breakthrough 1 §2), written as plain PyTorch fp64 CPU
operations one token at a time (all heads at once). ``torch.autograd`` then gives the
gradients of

    L = <dout, out> + <dh_final, h_final>

with respect to q, k, v, the gate logits a, beta and h0 -- the vector-Jacobian product
a backward kernel computes. The forward written here is pinned to the C oracle, and the
gradients to central finite differences and a one-token closed form, in the tests.
"""
from __future__ import annotations

import numpy as np
import torch


def _t(x):
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float64).clone()
    return torch.as_tensor(np.asarray(x, dtype=np.float64)).clone()


def log_decay(a, gate="bounded", g_min=-5.0):
    """Per-channel log-decay g from the gate logits: ``bounded`` is the method's
    g = g_min sigmoid(a) ("Demystifying Trillion-Parameter MoE Models", Breakthrough 1 §2;
    "From Numerical Stability to Load Balancing", §2.2); ``softplus`` is the unbounded
    prior art it replaces, g = -softplus(a) = -log(1 + e^a), which reaches any negative
    value ("Architecture Analysis of Ultra-Long Context Sparse MoE Models", §2.1-2.2;
    "Demystifying Trillion-Parameter MoE Models", Breakthrough 1 §1)."""
    if gate == "bounded":
        return g_min * torch.sigmoid(a)
    if gate == "softplus":
        return -torch.nn.functional.softplus(a)
    raise ValueError(f"unknown gate {gate!r}")


def forward_torch(q, k, v, a, beta, h0, cu, *, g_min=-5.0, scale=None, gate="bounded"):
    """The recurrence on fp64 torch tensors (differentiable). Shapes as
    ``recurrence.kda_forward``; ``cu`` is a sequence of int offsets; ``gate`` selects the
    log-decay (``log_decay``). Returns ``(out [N, H, d_v], h_final [n_seq, H, d_k, d_v])``."""
    N, H, dk = q.shape
    dv = v.shape[2]
    if scale is None:
        scale = dk ** -0.5
    outs, finals = [], []
    for n in range(len(cu) - 1):
        S = h0[n] if h0 is not None else torch.zeros((H, dk, dv), dtype=torch.float64)
        for t in range(int(cu[n]), int(cu[n + 1])):
            gamma = torch.exp(log_decay(a[t], gate, g_min))           # [H, dk]
            S = gamma[:, :, None] * S
            pred = torch.einsum("hkv,hk->hv", S, k[t])               # S^T k
            S = S + beta[t][:, None, None] * torch.einsum("hk,hv->hkv", k[t], v[t] - pred)
            outs.append(scale * torch.einsum("hkv,hk->hv", S, q[t]))  # S^T q
        finals.append(S)
    out = torch.stack(outs) if outs else torch.zeros((0, H, dv), dtype=torch.float64)
    return out, torch.stack(finals)


def kda_backward(q, k, v, a, beta, h0, cu_seqlens, dout, dh_final=None, *, g_min=-5.0,
                 scale=None):
    """Gradients of ``<dout, out> + <dh_final, h_final>``.

    Shapes (packed, token-major): ``q, k, a`` [N, H, d_k]; ``v``, ``dout`` [N, H, d_v];
    ``beta`` [N, H]; ``h0``, ``dh_final`` [n_seq, H, d_k, d_v] or None (zeros);
    ``cu_seqlens`` [n_seq + 1] or None (one sequence). Returns a dict of fp64 numpy
    arrays ``dq, dk, dv, da, dbeta, dh0``.
    """
    q, k, v, a, beta, dout = (_t(x) for x in (q, k, v, a, beta, dout))
    N, H, dk = q.shape
    dv = v.shape[2]
    if cu_seqlens is None:
        cu = [0, N]
    else:
        cu = [int(c) for c in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist")
                               else cu_seqlens)]
    n_seq = len(cu) - 1
    h0 = _t(h0) if h0 is not None else torch.zeros((n_seq, H, dk, dv), dtype=torch.float64)
    leaves = [q, k, v, a, beta, h0]
    for x in leaves:
        x.requires_grad_(True)
    out, hf = forward_torch(q, k, v, a, beta, h0, cu, g_min=g_min, scale=scale)
    loss = (out * dout).sum()
    if dh_final is not None:
        loss = loss + (hf * _t(dh_final)).sum()
    grads = torch.autograd.grad(loss, leaves, allow_unused=True)
    names = ["dq", "dk", "dv", "da", "dbeta", "dh0"]
    return {nm: (g.numpy() if g is not None else np.zeros(x.shape))
            for nm, g, x in zip(names, grads, leaves)}


def kda_forward_gate(q, k, v, a, beta, h0=None, cu_seqlens=None, *, gate="bounded",
                     scale=None):
    """The forward recurrence with either gate (fp64, no gradients). Returns numpy
    ``(out [N, H, d_v], h_final [n_seq, H, d_k, d_v])``."""
    q, k, v, a, beta = (_t(x) for x in (q, k, v, a, beta))
    N = q.shape[0]
    cu = [0, N] if cu_seqlens is None else [int(c) for c in (
        cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
    with torch.no_grad():
        out, hf = forward_torch(q, k, v, a, beta, _t(h0), cu, scale=scale, gate=gate)
    return out.numpy(), hf.numpy()
