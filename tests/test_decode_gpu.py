"""GPU parity of the recurrent decode step (``kda_decode_step``) against the fp64 oracle
on the same seeded inputs: single steps from random states, chains of steps, a decode
that continues a chunked prefill, the degenerate gates and strengths, and the bench's
full batch on sampled (sequence, head) pairs.

Bars as for the forward pass: rel-L2 <= 1e-4 for fp32 inputs, <= 1e-2 for bf16 (fp32
state and arithmetic in both), on the outputs and on the updated states.
"""
import numpy as np
import pytest
import torch

import chunked_linear_attention_kda_gb300 as kda
import kda_inputs as K
from oracle import recurrence
from tests.gpu_helpers import TOL, assert_finite, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


def cpu(t):
    return None if t is None else t.detach().to("cpu")


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def one_token_inputs(B, H, dk, dv, dtype, seed, **kw):
    """B one-token sequences: exactly the decode step's [B, H, ...] layout."""
    return K.make_inputs([1] * B, H, dk, dv, dtype=dtype, device=DEV, seed=seed,
                         h0_std=kw.pop("h0_std", 0.5), **kw)


def check_step(x, tol):
    state = x.h0.clone()
    out = kda.decode_step(x.q, x.k, x.v, x.a, x.beta, state)
    torch.cuda.synchronize()
    assert_finite(out, state)
    o_ref, s_ref = recurrence.decode_step(cpu(x.q), cpu(x.k), cpu(x.v), cpu(x.a),
                                          cpu(x.beta), cpu(x.h0))
    eo, es = rel_l2(f64(out), o_ref), rel_l2(f64(state), s_ref)
    assert eo <= tol and es <= tol, f"out {eo:.3e}, state {es:.3e}"
    return eo, es


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("B,H,dk,dv", [(5, 3, 128, 128), (2, 4, 64, 128), (3, 2, 40, 72),
                                       (1, 1, 1, 1), (7, 1, 128, 17)])
def test_single_step(dtype, B, H, dk, dv):
    check_step(one_token_inputs(B, H, dk, dv, dtype, seed=100 + dk + dv), TOL[dtype])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_chain_of_steps_equals_forward(dtype):
    """T steps, each feeding its state to the next, against the oracle run over the
    T-token sequences (outputs at every step, final state)."""
    B, T, H, d = 3, 40, 4, 128
    x = K.make_inputs([T] * B, H, d, d, dtype=dtype, device=DEV, seed=7, h0_std=0.3)
    state = x.h0.clone()
    outs = []
    for t in range(T):
        rows = torch.arange(B, device=DEV) * T + t
        outs.append(kda.decode_step(x.q[rows].contiguous(), x.k[rows].contiguous(),
                                    x.v[rows].contiguous(), x.a[rows].contiguous(),
                                    x.beta[rows].contiguous(), state))
    torch.cuda.synchronize()
    got = torch.stack(outs, dim=1).reshape(B * T, H, d)
    assert_finite(got, state)
    o_ref, s_ref = recurrence.kda_forward(cpu(x.q), cpu(x.k), cpu(x.v), cpu(x.a),
                                          cpu(x.beta), cpu(x.h0), x.cu_host)
    eo, es = rel_l2(f64(got), o_ref), rel_l2(f64(state), s_ref)
    assert eo <= TOL[dtype] and es <= TOL[dtype], f"out {eo:.3e}, state {es:.3e}"


def test_decode_continues_a_chunked_prefill():
    """Prompt through kda_chunk_fwd (tensor-core kernel), its h_final fed to one decode
    step for the next token: equals the oracle over prompt + token."""
    lengths, H, d = [100, 37, 16], 8, 128
    B = len(lengths)
    full = K.make_inputs([L + 1 for L in lengths], H, d, d, dtype=torch.bfloat16, device=DEV,
                         seed=21, h0_std=0.2)
    cu = full.cu_host
    keep = torch.cat([torch.arange(int(cu[b]), int(cu[b + 1]) - 1) for b in range(B)]).to(DEV)
    last = torch.as_tensor([int(cu[b + 1]) - 1 for b in range(B)], device=DEV)
    pcu = torch.tensor([0] + list(np.cumsum(lengths)), dtype=torch.int32, device=DEV)
    _, hf = kda.chunk_fwd(full.q[keep].contiguous(), full.k[keep].contiguous(),
                          full.v[keep].contiguous(), full.a[keep].contiguous(),
                          full.beta[keep].contiguous(), full.h0, pcu)
    o = kda.decode_step(full.q[last].contiguous(), full.k[last].contiguous(),
                        full.v[last].contiguous(), full.a[last].contiguous(),
                        full.beta[last].contiguous(), hf)
    torch.cuda.synchronize()
    assert_finite(o, hf)
    o_ref, h_ref = recurrence.kda_forward(cpu(full.q), cpu(full.k), cpu(full.v), cpu(full.a),
                                          cpu(full.beta), cpu(full.h0), cu)
    eo = rel_l2(f64(o), o_ref[np.asarray(cu[1:]) - 1])
    eh = rel_l2(f64(hf), h_ref)
    assert eo <= 1e-2 and eh <= 1e-2, f"out {eo:.3e}, state {eh:.3e}"


@pytest.mark.parametrize("case", ["beta_zero", "gate_at_bound", "no_decay", "zero_state"])
def test_degenerate_cases(case):
    x = one_token_inputs(4, 3, 128, 128, torch.float32, seed=31)
    if case == "beta_zero":          # nothing written: pure decay
        x.beta.zero_()
    elif case == "gate_at_bound":    # sigmoid saturates: every channel decays by exp(-5)
        x.a.fill_(60.0)
    elif case == "no_decay":         # sigmoid -> 0: the plain delta rule
        x.a.fill_(-60.0)
    else:
        x.h0.zero_()
    check_step(x, TOL[torch.float32])


def test_bench_batch_sampled():
    """The bench's decode batch (256 sequences x 32 heads, d = 128, bf16) in one call;
    the oracle checks 3 sequences x 4 heads of it."""
    B, H, d = 256, 32, 128
    x = one_token_inputs(B, H, d, d, torch.bfloat16, seed=41, h0_std=0.5)
    state = x.h0.clone()
    out = kda.decode_step(x.q, x.k, x.v, x.a, x.beta, state)
    torch.cuda.synchronize()
    assert_finite(out, state)
    seqs, heads = [0, 127, 255], [0, 13, 22, 31]
    sub = lambda t: cpu(t)[seqs][:, heads].contiguous()  # noqa: E731
    o_ref, s_ref = recurrence.decode_step(sub(x.q), sub(x.k), sub(x.v), sub(x.a),
                                          sub(x.beta), sub(x.h0))
    eo = rel_l2(f64(out)[seqs][:, heads], o_ref)
    es = rel_l2(f64(state)[seqs][:, heads], s_ref)
    assert eo <= 1e-2 and es <= 1e-2, f"out {eo:.3e}, state {es:.3e}"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_state_alignment_selects_either_kernel(dtype):
    """A 16-byte aligned state with d_v a multiple of 4 takes the 16-byte-access kernel; a
    state one float off that boundary takes the scalar kernel. Both meet the oracle's bar
    on the same inputs and agree with each other to fp32 rounding."""
    x = one_token_inputs(6, 5, 128, 128, dtype, seed=57, h0_std=0.5)
    n = x.h0.numel()
    aligned = x.h0.clone()
    shifted = torch.empty(n + 1, device=DEV)[1:].view_as(x.h0)
    shifted.copy_(x.h0)
    assert aligned.data_ptr() % 16 == 0 and shifted.data_ptr() % 16 == 4
    o_ref, s_ref = recurrence.decode_step(cpu(x.q), cpu(x.k), cpu(x.v), cpu(x.a),
                                          cpu(x.beta), cpu(x.h0))
    outs = []
    for st in (aligned, shifted):
        o = kda.decode_step(x.q, x.k, x.v, x.a, x.beta, st)
        torch.cuda.synchronize()
        assert_finite(o, st)
        eo, es = rel_l2(f64(o), o_ref), rel_l2(f64(st), s_ref)
        assert eo <= TOL[dtype] and es <= TOL[dtype], f"out {eo:.3e}, state {es:.3e}"
        outs.append(o.float())
    assert rel_l2(f64(aligned), f64(shifted)) <= 1e-6
    assert rel_l2(f64(outs[0]), f64(outs[1])) <= (1e-6 if dtype == torch.float32 else 1e-2)


def test_empty_batch_is_a_noop():
    x = torch.zeros(0, 2, 128, device=DEV)
    st = torch.zeros(0, 2, 128, 128, device=DEV)
    out = kda.decode_step(x, x, x, x, torch.zeros(0, 2, device=DEV), st)
    assert out.shape == (0, 2, 128)
