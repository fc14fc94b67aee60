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
