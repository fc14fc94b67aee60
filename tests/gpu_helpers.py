"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI and
the oracle on exactly the same (seeded) inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import chunked_linear_attention_kda_gb300 as kda
import kda_inputs as K
from oracle import recurrence

# rel-L2 bars: fp32 inputs 1e-4, bf16 inputs 1e-2 (fp32 state and accumulation)
TOL = {torch.float32: 1e-4, torch.bfloat16: 1e-2}


def rel_l2(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    nr = np.linalg.norm(ref)
    e = np.linalg.norm(x - ref)
    return float(e / nr) if nr > 0 else float(e)


def gpu_forward(x: K.KDAInputs, *, path="auto", want_state=True):
    fn = kda.chunk_fwd if path == "auto" else kda.chunk_fwd_simt
    out, hf = fn(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_seqlens,
                 output_final_state=want_state)
    torch.cuda.synchronize()
    return out, hf


def oracle_forward(x: K.KDAInputs, heads=None, want_state=True):
    """fp64 oracle on the CPU copies of the same tensors (optionally a subset of heads)."""
    if heads is not None:
        x = K.slice_heads(x, heads)
    cpu = lambda t: None if t is None else t.detach().to("cpu")  # noqa: E731
    return recurrence.kda_forward(cpu(x.q), cpu(x.k), cpu(x.v), cpu(x.a), cpu(x.beta),
                                  cpu(x.h0), x.cu_host, want_state=want_state)


def to_np(t, heads=None):
    if heads is not None:
        t = t.index_select(1, torch.as_tensor(list(heads), device=t.device))
    return t.detach().to("cpu", torch.float64).numpy()


def assert_finite(*ts):
    for t in ts:
        if t is not None:
            assert bool(torch.isfinite(t).all()), "non-finite values in GPU output"


def per_seq_head_rel(x_gpu, ref, cu, min_len: int = 1):
    """Worst rel-L2 over (sequence, head) of outputs [N, H, d] (sequences shorter than
    ``min_len`` skipped) -- a localised error is not diluted by the whole-tensor norm."""
    x_gpu = np.asarray(x_gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    worst = 0.0
    for s, e in zip(cu[:-1], cu[1:]):
        if e - s < max(1, min_len):
            continue
        d = x_gpu[s:e] - ref[s:e]
        num = np.sqrt((d ** 2).sum(axis=(0, 2)))
        den = np.sqrt((ref[s:e] ** 2).sum(axis=(0, 2)))
        r = np.where(den > 0, num / np.maximum(den, 1e-300), num)
        worst = max(worst, float(r.max()))
    return worst


def per_state_rel(h_gpu, h_ref):
    """Worst rel-L2 over (sequence, head) of final states [n_seq, H, d_k, d_v]."""
    h_gpu = np.asarray(h_gpu, dtype=np.float64)
    h_ref = np.asarray(h_ref, dtype=np.float64)
    num = np.sqrt(((h_gpu - h_ref) ** 2).sum(axis=(2, 3)))
    den = np.sqrt((h_ref ** 2).sum(axis=(2, 3)))
    r = np.where(den > 0, num / np.maximum(den, 1e-300), num)
    return float(r.max()) if r.size else 0.0
