"""GPU parity of the segment scan (one sequence split in time, segments run side by
side): ``kda_affine_combine`` against fp64 matrix products, and ``segmented_fwd``
against the fp64 oracle on the same seeded inputs, with the bars of the other parity
tests (rel-L2 1e-4 for fp32 inputs, 1e-2 for bf16)."""
import numpy as np
import pytest
import torch

import chunked_linear_attention_kda_gb300 as kda
import kda_inputs as K
from tests.gpu_helpers import TOL, assert_finite, oracle_forward, rel_l2, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("dk,dv", [(128, 128), (16, 16), (64, 32), (7, 5), (128, 33)])
def test_affine_combine_matches_fp64(dk, dv):
    g = torch.Generator(device=DEV)
    g.manual_seed(5)
    H = 3
    M = torch.randn(H, dk, dk, generator=g, device=DEV)
    S = torch.randn(H, dk, dv, generator=g, device=DEV)
    B = torch.randn(H, dk, dv, generator=g, device=DEV)
    O = kda.affine_combine(M, S, B)
    torch.cuda.synchronize()
    f64 = lambda t: t.detach().cpu().double().numpy()  # noqa: E731
    ref = np.einsum("hij,hjk->hik", f64(M), f64(S)) + f64(B)
    assert rel_l2(f64(O), ref) <= 1e-6


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T,segments", [(4096, 4), (1000, 3), (40, 5), (16, 2), (33, 8),
                                        (4096, 1)])
def test_segmented_forward_matches_oracle(dtype, T, segments):
    x = K.make_inputs([T], 4, 128, 128, dtype=dtype, device=DEV, seed=11, h0_std=0.1)
    out, hf = kda.segmented_fwd(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_seqlens,
                                segments=segments)
    torch.cuda.synchronize()
    assert_finite(out, hf)
    o_ref, h_ref = oracle_forward(x)
    eo, eh = rel_l2(to_np(out), o_ref), rel_l2(to_np(hf), h_ref)
    assert eo <= TOL[dtype] and eh <= TOL[dtype], (eo, eh)


def test_segmented_forward_zero_start_and_bound_gates():
    # no h0, half the heads at the decay bound, half without decay
    x = K.make_inputs([2000], 4, 128, 128, device=DEV, seed=12,
                      gate_mean=[6.0, 6.0, -6.0, -6.0], gate_std=[1.0] * 4)
    assert x.h0 is None
    out, hf = kda.segmented_fwd(x.q, x.k, x.v, x.a, x.beta, None, x.cu_seqlens, segments=5)
    torch.cuda.synchronize()
    assert_finite(out, hf)
    o_ref, h_ref = oracle_forward(x)
    eo, eh = rel_l2(to_np(out), o_ref), rel_l2(to_np(hf), h_ref)
    assert eo <= TOL[torch.bfloat16] and eh <= TOL[torch.bfloat16], (eo, eh)


def test_segmented_forward_rejects_packed_inputs():
    x = K.make_inputs([64, 64], 2, 128, 128, device=DEV, seed=1)
    with pytest.raises(ValueError):
        kda.segmented_fwd(x.q, x.k, x.v, x.a, x.beta, None, x.cu_seqlens, segments=2)
