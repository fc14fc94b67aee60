"""GPU parity of the backward pass (``kda_chunk_bwd``) against the fp64 reverse-mode
oracle on the same seeded inputs and upstream gradients: every gradient (dq, dk, dv,
dgate_logits, dbeta, dh0) element by element in rel-L2, on ragged varlen packings with
empty and partial chunks, odd head sizes, the degenerate gates and strengths, and the
bench's 64K-token workload through a suffix property.

Bars: rel-L2 <= 1e-4 for fp32 inputs, <= 1e-2 for bf16 inputs (fp32 arithmetic).
"""
import numpy as np
import pytest
import torch

import chunked_linear_attention_kda_gb300 as kda
import kda_inputs as K
from oracle import backward as B
from tests.gpu_helpers import TOL, assert_finite, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"
NAMES = ["dq", "dk", "dv", "da", "dbeta", "dh0"]


def cpu(t):
    return None if t is None else t.detach().to("cpu")


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def upstream(x, seed, with_dhf=True):
    g = torch.Generator(device="cpu").manual_seed(seed)
    dout = torch.randn((x.n_tok, x.n_heads, x.d_v), generator=g).to(DEV, x.dtype)
    dhf = torch.randn((x.n_seq, x.n_heads, x.d_k, x.d_v), generator=g).to(DEV) if with_dhf \
        else None
    return dout, dhf


def check(x, seed=0, with_dhf=True, tol=None):
    dout, dhf = upstream(x, seed, with_dhf)
    got = kda.chunk_bwd(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_seqlens, dout, dhf)
    torch.cuda.synchronize()
    assert_finite(*got)
    ref = B.kda_backward(cpu(x.q), cpu(x.k), cpu(x.v), cpu(x.a), cpu(x.beta), cpu(x.h0),
                         x.cu_host, cpu(dout), cpu(dhf))
    tol = TOL[x.dtype] if tol is None else tol
    errs = {nm: rel_l2(f64(g), ref[nm]) for nm, g in zip(NAMES, got)}
    bad = {nm: e for nm, e in errs.items() if not e <= tol}
    assert not bad, f"{x.name}: {errs}"
    return errs


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_ragged_varlen_d32(dtype):
    x = K.make_inputs([1, 15, 0, 16, 17, 40], 2, 32, 32, dtype=dtype, device=DEV, seed=1,
                      h0_std=0.3)
    check(x, seed=1)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_d128_two_sequences(dtype):
    x = K.make_inputs([50, 33], 2, 128, 128, dtype=dtype, device=DEV, seed=2, h0_std=0.3)
    check(x, seed=2)


def test_odd_head_sizes():
    x = K.make_inputs([23, 9], 3, 40, 72, dtype=torch.float32, device=DEV, seed=3, h0_std=0.2)
    check(x, seed=3)


def test_no_h0_no_dh_final():
    x = K.make_inputs([37], 2, 64, 64, dtype=torch.float32, device=DEV, seed=4)
    check(x, seed=4, with_dhf=False)


@pytest.mark.parametrize("case", ["beta_zero", "gate_at_bound", "no_decay"])
def test_degenerate_cases(case):
    x = K.make_inputs([20, 16], 2, 32, 32, dtype=torch.float32, device=DEV, seed=5,
                      h0_std=0.3)
    if case == "beta_zero":
        x.beta.zero_()
    elif case == "gate_at_bound":
        x.a.fill_(40.0)
    else:
        x.a.fill_(-40.0)
    check(x, seed=5)


def test_context_64k_suffix():
    """The 64K-token, 32-head workload in one backward call. The gradients of the last
    256 tokens, and the state gradient at their start, are those of the last 256 tokens
    run alone from the state the first 65280 tokens leave (same upstream gradients): the
    oracle checks that suffix on two heads, its start state taken from the fp32 SIMT
    forward of the prefix."""
    x = K.make_workload(3, DEV)
    dout, dhf = upstream(x, 6)
    got = kda.chunk_bwd(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_seqlens, dout, dhf,
                        want_dh0=False)
    torch.cuda.synchronize()
    assert_finite(*got[:5])
    T, t1, heads = x.n_tok, x.n_tok - 256, [5, 26]
    pre = K.prefix(x, t1)
    _, s1 = kda.chunk_fwd_simt(pre.q, pre.k, pre.v, pre.a, pre.beta, pre.h0, pre.cu_seqlens)
    torch.cuda.synchronize()
    hsel = lambda t: cpu(t)[:, heads].contiguous()  # noqa: E731
    ref = B.kda_backward(hsel(x.q[t1:]), hsel(x.k[t1:]), hsel(x.v[t1:]), hsel(x.a[t1:]),
                         hsel(x.beta[t1:]), hsel(s1), [0, T - t1], hsel(dout[t1:]), hsel(dhf))
    for nm, g in zip(NAMES[:5], got[:5]):
        e = rel_l2(f64(g[t1:])[:, heads], ref[nm])
        assert e <= 1e-2, f"{nm}: {e:.3e}"


def test_kernel_timing_records_every_call():
    """The per-kernel event timing the bench reports: four positive kernel times summed
    over exactly the calls made while recording, and results unchanged by recording."""
    x = K.make_inputs([70, 33], 2, 128, 128, dtype=torch.bfloat16, device=DEV, seed=8,
                      h0_std=0.3)
    dout, dhf = upstream(x, 8)
    ref = kda.chunk_bwd(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_seqlens, dout, dhf)
    kda.bwd_timing_start(8)
    for _ in range(3):
        got = kda.chunk_bwd(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_seqlens, dout, dhf)
    ms, calls = kda.bwd_timing_read()
    # the serial passes share one launch on this path: their time is in ms[1]
    assert calls == 3 and ms[0] > 0 and ms[1] > 0 and ms[3] > 0 and ms[2] >= 0, (ms, calls)
    kda.chunk_bwd(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_seqlens, dout, dhf)  # not recorded
    assert kda.bwd_timing_read()[1] == 3
    torch.cuda.synchronize()
    for r, g in zip(ref, got):
        assert torch.equal(r, g)


def test_many_sequences_per_cta():
    """Seven sequences (one empty, some shorter than a chunk) over 8 heads: about 3500
    (chunk, head) items, so every CTA of the chunk-parallel kernels walks across sequence
    ends and the gap slots between them. Sequences are independent: the oracle checks the
    three short ones on two heads."""
    lens = [2000, 0, 700, 17, 1200, 5, 3000]
    x = K.make_inputs(lens, 8, 128, 128, dtype=torch.bfloat16, device=DEV, seed=21,
                      h0_std=0.3)
    dout, dhf = upstream(x, 21)
    got = kda.chunk_bwd(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_seqlens, dout, dhf)
    torch.cuda.synchronize()
    assert_finite(*got)
    heads = [1, 6]
    for n in (2, 3, 5):
        t0, t1 = x.cu_host[n], x.cu_host[n + 1]
        sel = lambda t: cpu(t)[t0:t1][:, heads].contiguous()  # noqa: E731
        ref = B.kda_backward(sel(x.q), sel(x.k), sel(x.v), sel(x.a), sel(x.beta),
                             cpu(x.h0)[n:n + 1][:, heads], [0, t1 - t0], sel(dout),
                             cpu(dhf)[n:n + 1][:, heads])
        for nm, g in zip(NAMES[:5], got[:5]):
            e = rel_l2(f64(g[t0:t1])[:, heads], ref[nm])
            assert e <= TOL[torch.bfloat16], f"sequence {n} {nm}: {e:.3e}"
        e = rel_l2(f64(got[5][n:n + 1])[:, heads], ref["dh0"])
        assert e <= TOL[torch.bfloat16], f"sequence {n} dh0: {e:.3e}"


def test_unaligned_workspace_takes_the_fp32_kernels():
    """A workspace 4 bytes off a 16-byte boundary (allowed: 4-byte alignment) rules out
    the bulk copies, so bf16 d = 128 runs on the fp32 kernels: still exact to the bar."""
    x = K.make_inputs([50, 33], 2, 128, 128, dtype=torch.bfloat16, device=DEV, seed=22,
                      h0_std=0.3)
    dout, dhf = upstream(x, 22)
    lib = kda.load_library()
    nbytes = lib.kda_chunk_bwd_workspace_bytes(x.n_tok, x.n_seq, 2, 128, 128)
    raw = torch.empty(nbytes + 16, dtype=torch.uint8, device=DEV)
    ws = raw[4:4 + nbytes]
    assert ws.data_ptr() % 16 == 4
    got = kda.chunk_bwd(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_seqlens, dout, dhf,
                        workspace=ws)
    torch.cuda.synchronize()
    ref = B.kda_backward(cpu(x.q), cpu(x.k), cpu(x.v), cpu(x.a), cpu(x.beta), cpu(x.h0),
                         x.cu_host, cpu(dout), cpu(dhf))
    for nm, g in zip(NAMES, got):
        e = rel_l2(f64(g), ref[nm])
        assert e <= TOL[torch.bfloat16], f"{nm}: {e:.3e}"
