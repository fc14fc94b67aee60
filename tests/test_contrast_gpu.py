"""GPU tests of the contrast variants (``kda_chunk_fwd_variant``): the bounded gate with
either diagonal tile equals the method; the unbounded softplus gate is computed correctly
by the position-pair tile at any decay, while the dense tile -- the method's fast path --
overflows once a chunk's decay passes what fp32 can invert (the failure the bound
removes, reproduced on purpose). Oracle: the fp64 recurrence with the same gate.
"""
import pytest
import torch

import chunked_linear_attention_kda_gb300 as kda
import kda_inputs as K
from oracle import backward as B
from tests.gpu_helpers import TOL, assert_finite, gpu_forward, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


def cpu(t):
    return None if t is None else t.detach().to("cpu")


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def oracle(x, gate):
    return B.kda_forward_gate(cpu(x.q), cpu(x.k), cpu(x.v), cpu(x.a), cpu(x.beta), cpu(x.h0),
                              x.cu_host, gate=gate)


def run(x, gate, diag):
    out, hf = kda.chunk_fwd_variant(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_seqlens,
                                    gate=gate, diag=diag)
    torch.cuda.synchronize()
    return out, hf


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("diag", ["dense", "pairs"])
def test_bounded_gate_either_tile(dtype, diag):
    x = K.make_inputs([40, 17, 0, 64], 2, 64, 64, dtype=dtype, device=DEV, seed=11, h0_std=0.3)
    out, hf = run(x, "bounded", diag)
    assert_finite(out, hf)
    o_ref, h_ref = oracle(x, "bounded")
    eo, eh = rel_l2(f64(out), o_ref), rel_l2(f64(hf), h_ref)
    assert eo <= TOL[dtype] and eh <= TOL[dtype], f"out {eo:.3e}, state {eh:.3e}"


def test_bounded_dense_variant_is_the_simt_forward():
    """Same template instance as the product's fp32 kernel: bit-identical results."""
    x = K.make_inputs([50, 9], 3, 128, 128, dtype=torch.float32, device=DEV, seed=12,
                      h0_std=0.2)
    out, hf = run(x, "bounded", "dense")
    ref_o, ref_h = gpu_forward(x, path="simt")
    assert torch.equal(out, ref_o) and torch.equal(hf, ref_h)


@pytest.mark.parametrize("diag", ["dense", "pairs"])
def test_softplus_gate_moderate_decay(diag):
    """Gate logits ~ N(0, 1): softplus ~ 0.7 per token, a chunk's decay ~ -11, within
    fp32 range either way: both tiles match the unbounded oracle."""
    x = K.make_inputs([33, 48], 2, 64, 64, dtype=torch.float32, device=DEV, seed=13,
                      h0_std=0.3, gate_std=1.0)
    out, hf = run(x, "softplus", diag)
    assert_finite(out, hf)
    o_ref, h_ref = oracle(x, "softplus")
    eo, eh = rel_l2(f64(out), o_ref), rel_l2(f64(hf), h_ref)
    assert eo <= 1e-4 and eh <= 1e-4, f"out {eo:.3e}, state {eh:.3e}"


def extreme(dtype):
    """A decay of -40 per token (softplus(40) = 40) on a band of channels: the chunk's
    cumulative decay reaches -640 there."""
    x = K.make_inputs([32, 20], 2, 64, 64, dtype=dtype, device=DEV, seed=14, h0_std=0.3,
                      gate_std=1.0)
    x.a[:, :, :16] = 40.0
    return x


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_softplus_extreme_decay_pairs_tile_is_exact(dtype):
    x = extreme(dtype)
    out, hf = run(x, "softplus", "pairs")
    assert_finite(out, hf)
    o_ref, h_ref = oracle(x, "softplus")
    eo, eh = rel_l2(f64(out), o_ref), rel_l2(f64(hf), h_ref)
    tol = 1e-4 if dtype == torch.float32 else 1e-2
    assert eo <= tol and eh <= tol, f"out {eo:.3e}, state {eh:.3e}"


def test_softplus_extreme_decay_dense_tile_overflows():
    """The dense tile needs e^-G = e^640 there: it overflows fp32 and the outputs are no
    longer finite."""
    x = extreme(torch.float32)
    out, _ = run(x, "softplus", "dense")
    assert not bool(torch.isfinite(out).all())


def test_bounded_gate_cannot_reach_the_overflow():
    """The same logits through the bounded gate: -5 per token at most, -80 per chunk,
    and the method's tensor-core kernel stays finite and exact."""
    x2 = K.make_inputs([32, 20], 2, 128, 128, dtype=torch.bfloat16, device=DEV, seed=14,
                       h0_std=0.3, gate_std=1.0)
    x2.a[:, :, :16] = 40.0
    out, hf = gpu_forward(x2)
    assert_finite(out, hf)
    o_ref, h_ref = oracle(x2, "bounded")
    assert rel_l2(f64(out), o_ref) <= 1e-2 and rel_l2(f64(hf), h_ref) <= 1e-2
