"""GPU parity of the gate projection (``kda_gate_projection``, tcgen05 GEMM) against the
fp64 oracle ``a = x W^T + b``: tile-exact and ragged shapes (row, column and K tails,
columns not a multiple of 4), no bias, the bench's 64K x 4096 x 4096 problem on sampled
rows, and the projection feeding the forward pass.

Bar: rel-L2 <= 1e-5 on a (bf16 products are exact in fp32; only the fp32 accumulation
order differs from the fp64 sum), 1e-2 for the forward fed by it (bf16 inputs).
"""
import numpy as np
import pytest
import torch

import chunked_linear_attention_kda_gb300 as kda
import kda_inputs as K
from oracle import projection, recurrence
from tests.gpu_helpers import assert_finite, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


def make(M, D, N, bias=True, seed=0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn((M, D), generator=g).to(DEV, torch.bfloat16)
    w = (torch.randn((N, D), generator=g) * D ** -0.5).to(DEV, torch.bfloat16)
    b = torch.randn((N,), generator=g).to(DEV) if bias else None
    return x, w, b


@pytest.mark.parametrize("M,D,N,bias", [(128, 64, 256, True), (300, 256, 384, True),
                                        (1, 8, 4, False), (257, 72, 250, True),
                                        (1000, 512, 4096, False)])
def test_projection_shapes(M, D, N, bias):
    x, w, b = make(M, D, N, bias, seed=M + D + N)
    a = kda.gate_projection(x, w, b)
    torch.cuda.synchronize()
    assert kda.read_device_flags() == 0
    assert_finite(a)
    ref = projection.gate_projection(x, w, b)
    e = rel_l2(a.double().cpu().numpy(), ref)
    assert e <= 1e-5, f"{(M, D, N)}: {e:.3e}"


@pytest.mark.parametrize("M,D,N,bias", [(128, 64, 256, True), (257, 72, 250, True),
                                        (1, 8, 4, False), (1000, 512, 4096, True)])
def test_bf16_output_is_the_fp32_output_rounded(M, D, N, bias):
    """bf16 output (N a multiple of 8 takes the packed stores, else the scalar ones): the
    fp32 result plus bias rounded to nearest even, bit for bit."""
    x, w, b = make(M, D, N, bias, seed=M + 2 * N)
    a32 = kda.gate_projection(x, w, b)
    a16 = kda.gate_projection(x, w, b, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert a16.dtype == torch.bfloat16 and torch.equal(a16, a32.to(torch.bfloat16))


def test_bench_problem_sampled_rows():
    M, D, N = 65536, 4096, 4096
    x, w, b = make(M, D, N, True, seed=3)
    a = kda.gate_projection(x, w, b)
    torch.cuda.synchronize()
    assert kda.read_device_flags() == 0
    rows = torch.tensor([0, 1, 127, 128, 4095, 33333, 65535], device=DEV)
    ref = projection.gate_projection(x[rows], w, b)
    assert rel_l2(a[rows].double().cpu().numpy(), ref) <= 1e-5
    assert_finite(a)


def test_projection_feeds_the_forward():
    """x -> gate logits -> chunked forward (tensor-core kernel), against the oracle given
    the fp64 projection of the same x and W."""
    H, d, D = 4, 128, 256
    base = K.make_inputs([200, 77], H, d, d, dtype=torch.bfloat16, device=DEV, seed=8,
                         h0_std=0.2)
    x, w, b = make(base.n_tok, D, H * d, True, seed=8)
    a = kda.gate_projection(x, w, b).view(base.n_tok, H, d)
    out, hf = kda.chunk_fwd(base.q, base.k, base.v, a, base.beta, base.h0, base.cu_seqlens)
    torch.cuda.synchronize()
    assert_finite(out, hf)
    a_ref = projection.gate_projection(x, w, b).reshape(base.n_tok, H, d)
    cpu = lambda t: t.detach().to("cpu")  # noqa: E731
    o_ref, h_ref = recurrence.kda_forward(cpu(base.q), cpu(base.k), cpu(base.v), a_ref,
                                          cpu(base.beta), cpu(base.h0), base.cu_host)
    assert rel_l2(out.double().cpu().numpy(), o_ref) <= 1e-2
    assert rel_l2(hf.double().cpu().numpy(), h_ref) <= 1e-2
