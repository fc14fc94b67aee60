"""The forward pass fed by the gate projection (``kda_chunk_fwd_gated``): bit for bit the
gate projection followed by the forward, for every segment length (cuts inside sequences,
state carried between pieces), and against the fp64 projection + recurrence oracles."""
import numpy as np
import pytest
import torch

import chunked_linear_attention_kda_gb300 as kda
import kda_inputs as K
from tests.gpu_helpers import assert_finite, oracle_forward, per_seq_head_rel, rel_l2, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def layer(x, H, d_model, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    xx = torch.randn((x.n_tok, d_model), generator=g).to(DEV, torch.bfloat16)
    w = (torch.randn((H * 128, d_model), generator=g) * d_model ** -0.5).to(DEV, torch.bfloat16)
    b = torch.randn((H * 128,), generator=g).to(DEV)
    return xx, w, b


@pytest.mark.parametrize("segment", [64, 256, 1000, 1 << 20])
@pytest.mark.parametrize("with_state", [True, False])
def test_equals_projection_then_forward(segment, with_state):
    lengths = [300, 0, 1000, 77, 2100, 64]
    x = K.make_inputs(lengths, 4, 128, 128, device=DEV, seed=41, h0_std=0.2 if with_state else None)
    xx, w, b = layer(x, 4, 256, 42)
    a = kda.gate_projection(xx, w, b).view(x.n_tok, 4, 128)
    ref_o, ref_h = kda.chunk_fwd(x.q, x.k, x.v, a, x.beta, x.h0, x.cu_seqlens,
                                 output_final_state=with_state)
    o, h = kda.chunk_fwd_gated(xx, w, b, x.q, x.k, x.v, x.beta, x.h0, x.cu_seqlens,
                               segment_tokens=segment, output_final_state=with_state)
    torch.cuda.synchronize()
    assert torch.equal(o, ref_o)
    if with_state:
        assert torch.equal(h, ref_h)
    else:
        assert h is None


def test_no_bias_and_repeat_calls():
    x = K.make_inputs([513, 129], 2, 128, 128, device=DEV, seed=43)
    xx, w, _ = layer(x, 2, 128, 44)
    a = kda.gate_projection(xx, w, None).view(x.n_tok, 2, 128)
    ref_o, ref_h = kda.chunk_fwd(x.q, x.k, x.v, a, x.beta, None, x.cu_seqlens)
    ws = torch.empty(kda.load_library().kda_chunk_fwd_gated_workspace_bytes(2, 2, 128, 128, 128),
                     dtype=torch.uint8, device=DEV)
    for _ in range(2):  # the workspace holds the previous call's data: nothing depends on it
        o, h = kda.chunk_fwd_gated(xx, w, None, x.q, x.k, x.v, x.beta, None, x.cu_seqlens,
                                   segment_tokens=128, workspace=ws)
        assert torch.equal(o, ref_o) and torch.equal(h, ref_h)


def test_against_projection_and_recurrence_oracles():
    """fp64 a = x W^T + b (oracle/projection.py), then the fp64 recurrence
    (oracle/kda_oracle.c) on those logits, against the gated forward."""
    from oracle.projection import gate_projection as proj64
    x = K.make_inputs([700, 64, 1300], 4, 128, 128, device=DEV, seed=45, h0_std=0.1)
    xx, w, b = layer(x, 4, 512, 46)
    o, h = kda.chunk_fwd_gated(xx, w, b, x.q, x.k, x.v, x.beta, x.h0, x.cu_seqlens,
                               segment_tokens=512)
    assert_finite(o, h)
    a64 = proj64(xx, w, b).reshape(x.n_tok, 4, 128)
    xo = K.KDAInputs(x.name, x.q, x.k, x.v, torch.from_numpy(a64).float().to(DEV), x.beta, x.h0,
                     x.cu_seqlens, x.cu_host, x.dtype)
    o_ref, h_ref = oracle_forward(xo)
    og, hg = to_np(o), to_np(h)
    assert max(rel_l2(og, o_ref), rel_l2(hg, h_ref), per_seq_head_rel(og, o_ref, x.cu_host, 16)) < 1e-2


def test_no_tokens():
    x = K.make_inputs([0, 0], 2, 128, 128, device=DEV, seed=47, h0_std=0.1)
    xx = torch.empty((0, 128), dtype=torch.bfloat16, device=DEV)
    w = torch.zeros((256, 128), dtype=torch.bfloat16, device=DEV)
    o, h = kda.chunk_fwd_gated(xx, w, None, x.q, x.k, x.v, x.beta, x.h0, x.cu_seqlens)
    assert o.numel() == 0 and torch.equal(h, x.h0)
