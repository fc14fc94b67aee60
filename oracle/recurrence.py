"""ctypes loader for the fp64 token-by-token oracle in ``kda_oracle.c``.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The recurrence, per sequence and head, with S in R^{d_k x d_v}:

    g_t = g_min * sigmoid(a_t)                      per key channel, g_min = -5
    S   <- Diag(exp g_t) S
    S   <- S + beta_t k_t (v_t - S^T k_t)^T
    o_t  = d_k^-1/2 S^T q_t

The bounded gate follows "Demystifying Trillion-Parameter MoE Models", Breakthrough 1
§2 and "From Numerical Stability to Load Balancing", §2.2; the state that decays and
writes key-value outer products follows the latter's §2.1.

Inputs are converted to fp64 before the call; bf16 and fp32 values convert exactly,
so the oracle sees exactly the numbers handed to the GPU.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_libs: dict[int, ctypes.CDLL] = {}


def oracle_library_path(mutant: int = 0) -> str:
    name = "libkda_oracle.so" if mutant == 0 else f"libkda_oracle_mutant{mutant}.so"
    return os.path.join(_BUILD, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile ``kda_oracle.c`` (plain C, -O2, no fast-math) into ``_build/``."""
    out = oracle_library_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           f"-DKDA_ORACLE_MUTANT={int(mutant)}", _SRC, "-o", tmp, "-lpthread", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _load(mutant: int = 0) -> ctypes.CDLL:
    with _lock:
        lib = _libs.get(mutant)
        if lib is None:
            lib = ctypes.CDLL(build(mutant))
            dp = ctypes.POINTER(ctypes.c_double)
            lib.kda_oracle_fwd.argtypes = [dp, dp, dp, dp, dp, dp,
                                           ctypes.POINTER(ctypes.c_int64),
                                           ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_int64, ctypes.c_double, ctypes.c_double,
                                           dp, dp, ctypes.c_int]
            lib.kda_oracle_fwd.restype = ctypes.c_int
            _libs[mutant] = lib
        return lib


def _f64(x) -> np.ndarray:
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor (any dtype, CPU)
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(x):
    if x is None:
        return None
    return x.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def kda_forward(q, k, v, a, beta, h0=None, cu_seqlens=None, *, g_min: float = -5.0,
                scale: float | None = None, threads: int | None = None,
                want_state: bool = True, mutant: int = 0):
    """Run the oracle.

    Shapes (packed, token-major): ``q, k, a`` [N, H, d_k]; ``v`` [N, H, d_v];
    ``beta`` [N, H]; ``h0`` [n_seq, H, d_k, d_v] or None (zeros);
    ``cu_seqlens`` [n_seq + 1] integer offsets or None (one sequence of N tokens).
    ``scale`` defaults to d_k^-1/2. Returns ``(out [N, H, d_v], h_final)`` in fp64;
    ``h_final`` is None when ``want_state`` is False.
    """
    q, k, v, a, beta = (_f64(t) for t in (q, k, v, a, beta))
    N, H, dk = q.shape
    dv = v.shape[2]
    assert k.shape == (N, H, dk) and a.shape == (N, H, dk), "q/k/a shape mismatch"
    assert v.shape == (N, H, dv) and beta.shape == (N, H), "v/beta shape mismatch"
    if cu_seqlens is None:
        cu = np.array([0, N], dtype=np.int64)
    else:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().cpu().numpy()
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    n_seq = cu.shape[0] - 1
    assert cu[0] == 0 and cu[-1] == N and np.all(np.diff(cu) >= 0), "bad cu_seqlens"
    h0 = _f64(h0)
    if h0 is not None:
        assert h0.shape == (n_seq, H, dk, dv), "h0 shape mismatch"
    if scale is None:
        scale = float(dk) ** -0.5
    out = np.zeros((N, H, dv), dtype=np.float64)
    hf = np.zeros((n_seq, H, dk, dv), dtype=np.float64) if want_state else None
    rc = _load(mutant).kda_oracle_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(beta), _ptr(h0),
        cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        n_seq, H, dk, dv, float(g_min), float(scale), _ptr(out), _ptr(hf),
        int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_fwd failed with code {rc}")
    return out, hf


def decode_step(q, k, v, a, beta, state, *, g_min: float = -5.0, scale: float | None = None,
                threads: int | None = None, mutant: int = 0):
    """One recurrent decode step: each of B sequences advances by one token from its own
    state. By definition this is the recurrence run on B one-token sequences started from
    ``state``, so it calls ``kda_forward`` with ``cu_seqlens = [0, 1, ..., B]``.

    ``q, k, a`` [B, H, d_k]; ``v`` [B, H, d_v]; ``beta`` [B, H]; ``state``
    [B, H, d_k, d_v]. Returns ``(out [B, H, d_v], new_state [B, H, d_k, d_v])`` in fp64.
    """
    B = (q.shape[0])
    return kda_forward(q, k, v, a, beta, state, np.arange(B + 1, dtype=np.int64),
                       g_min=g_min, scale=scale, threads=threads, mutant=mutant)
