"""GPU tests of the two host-memory entry points: ``kda_chunk_fwd_from_host`` (copy in,
compute, copy out on one stream) and ``kda_chunk_fwd_from_host_pipelined`` (segments whose
copies overlap the computation, a cut sequence's state carried in fp32 between pieces).

Both must give exactly -- bit for bit -- what ``kda_chunk_fwd`` gives on the same inputs
already on the device: the pipelined call runs the same kernels on the same 16-token
chunks (every cut lies on a sequence's chunk grid). One case is also checked against the
fp64 oracle at the usual bars, and the launch counter confirms that the forward kernels
ran once per piece.
"""
import pytest
import torch

import chunked_linear_attention_kda_gb300 as kda
import kda_inputs as K
from tests.gpu_helpers import TOL, assert_finite, oracle_forward, rel_l2, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def host_buffers(x, want_state=True, with_h0=True):
    pin = lambda t: None if t is None else t.detach().to("cpu").pin_memory()  # noqa: E731
    host = {"q": pin(x.q), "k": pin(x.k), "v": pin(x.v), "gate_logits": pin(x.a),
            "beta": pin(x.beta), "h0": pin(x.h0) if with_h0 else None,
            "cu_seqlens": pin(x.cu_seqlens)}
    h_out = torch.full((x.n_tok, x.n_heads, x.d_v), float("nan"), dtype=x.dtype).pin_memory()
    h_hf = (torch.full((x.n_seq, x.n_heads, x.d_k, x.d_v), float("nan")).pin_memory()
            if want_state else None)
    dev = {k: (torch.empty_like(v, device=DEV) if v is not None else None)
           for k, v in host.items()}
    dev["out"] = torch.empty(h_out.shape, dtype=x.dtype, device=DEV)
    dev["h_final"] = torch.empty(h_hf.shape, device=DEV) if want_state else None
    return host, h_out, h_hf, dev


def run_host(x, n_segments=None, want_state=True, with_h0=True):
    host, h_out, h_hf, dev = host_buffers(x, want_state, with_h0)
    args = (host["q"], host["k"], host["v"], host["gate_logits"], host["beta"], host["h0"],
            host["cu_seqlens"], h_out, h_hf, dev)
    if n_segments is None:
        kda.chunk_fwd_from_host(*args)
    else:
        kda.chunk_fwd_from_host_pipelined(*args, n_segments=n_segments)
    torch.cuda.synchronize()
    return h_out, h_hf


def device_reference(x, want_state=True, with_h0=True):
    out, hf = kda.chunk_fwd(x.q, x.k, x.v, x.a, x.beta, x.h0 if with_h0 else None,
                            x.cu_seqlens, output_final_state=want_state)
    torch.cuda.synchronize()
    return out.cpu(), None if hf is None else hf.cpu()


def assert_same(got, ref):
    for g, r in zip(got, ref):
        if r is None:
            assert g is None
            continue
        assert g.dtype == r.dtype and g.shape == r.shape
        assert torch.equal(g.view(torch.int16 if g.dtype == torch.bfloat16 else torch.int32),
                           r.view(torch.int16 if r.dtype == torch.bfloat16 else torch.int32))


CASES = {
    # name: (lengths, H, d_k, d_v, dtype)
    "one-sequence-tc": ([8192], 4, 128, 128, torch.bfloat16),
    "ragged-tc": ([700, 0, 2000, 17, 1200, 5, 3000], 3, 128, 128, torch.bfloat16),
    "ragged-fp32-simt": ([300, 0, 517, 33], 2, 128, 128, torch.float32),
    "d64-bf16-simt": ([1000, 250], 2, 64, 64, torch.bfloat16),
    "d40x72-fp32": ([129, 0, 400], 2, 40, 72, torch.float32),
    "uncuttable-d36-bf16": ([500, 77], 1, 36, 36, torch.bfloat16),  # 72-byte rows: one piece
}


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("n_segments", [1, 3, 16, 64])
def test_pipelined_equals_device_call(case, n_segments):
    lens, H, dk, dv, dt = CASES[case]
    x = K.make_inputs(lens, H, dk, dv, dtype=dt, device=DEV, seed=len(lens) * 31 + dk,
                      h0_std=0.5)
    ref = device_reference(x)
    got = run_host(x, n_segments)
    assert_finite(*got)
    assert_same(got, ref)


@pytest.mark.parametrize("case", ["one-sequence-tc", "ragged-tc", "ragged-fp32-simt"])
def test_serial_host_entry_equals_device_call(case):
    lens, H, dk, dv, dt = CASES[case]
    x = K.make_inputs(lens, H, dk, dv, dtype=dt, device=DEV, seed=7, h0_std=0.5)
    assert_same(run_host(x), device_reference(x))


@pytest.mark.parametrize("want_state,with_h0", [(False, True), (True, False), (False, False)])
def test_pipelined_without_h0_or_h_final(want_state, with_h0):
    x = K.make_inputs([3000, 1, 900], 2, 128, 128, device=DEV, seed=11, h0_std=0.5)
    ref = device_reference(x, want_state, with_h0)
    got = run_host(x, 8, want_state, with_h0)
    assert_same(got, ref)


def test_pipelined_no_tokens_copies_h0_to_h_final():
    x = K.make_inputs([0, 0], 2, 128, 128, device=DEV, seed=3, h0_std=0.5)
    out, hf = run_host(x, 4)
    assert out.numel() == 0
    assert torch.equal(hf, x.h0.cpu())


def test_pipelined_against_the_oracle_and_launch_count():
    """bf16 ragged packing with cut sequences, checked against the fp64 oracle on two heads;
    the forward kernels ran once per piece of the plan (plus one offsets kernel)."""
    lens = [2500, 0, 37, 4100]
    x = K.make_inputs(lens, 4, 128, 128, device=DEV, seed=21, h0_std=0.5)
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    pieces = kda.fwd_pipeline_plan(cu, 8)
    assert any(p[5] for p in pieces), "the case must cut a sequence"
    n0 = kda.kernel_launch_count()
    out, hf = run_host(x, 8)
    launched = kda.kernel_launch_count() - n0
    assert launched == len(pieces) + 1
    heads = [0, 3]
    o_ref, h_ref = oracle_forward(x, heads=heads)
    eo = rel_l2(to_np(out, heads), o_ref)
    eh = rel_l2(to_np(hf, heads), h_ref)
    assert eo <= TOL[torch.bfloat16] and eh <= TOL[torch.bfloat16], f"out {eo:.3e}, h {eh:.3e}"


def test_pipelined_repeated_calls_reuse_the_workspace():
    """Back-to-back calls on one stream with different inputs in the same host buffers:
    each call's results are those of its own inputs."""
    x1 = K.make_inputs([5000, 3000], 2, 128, 128, device=DEV, seed=41, h0_std=0.5)
    x2 = K.make_inputs([5000, 3000], 2, 128, 128, device=DEV, seed=42, h0_std=0.5)
    host, h_out, h_hf, dev = host_buffers(x1)
    results = []
    for x in (x1, x2, x1):
        for name, t in (("q", x.q), ("k", x.k), ("v", x.v), ("gate_logits", x.a),
                        ("beta", x.beta), ("h0", x.h0)):
            host[name].copy_(t.cpu())
        kda.chunk_fwd_from_host_pipelined(host["q"], host["k"], host["v"],
                                          host["gate_logits"], host["beta"], host["h0"],
                                          host["cu_seqlens"], h_out, h_hf, dev, n_segments=6)
        torch.cuda.synchronize()
        results.append((h_out.clone(), h_hf.clone()))
    assert_same(results[0], device_reference(x1))
    assert_same(results[1], device_reference(x2))
    assert_same(results[2], results[0])
