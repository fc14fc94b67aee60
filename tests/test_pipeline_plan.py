"""The pipelined forward's schedule on the host, without a GPU: the pieces that
``kda_chunk_fwd_pipeline_plan`` returns (the ones ``kda_chunk_fwd_from_host_pipelined``
runs) cover every token once and in order, read each sequence's h0 once and write its
h_final once, hand a cut sequence's state from one segment to the next, cut only on the
sequence's 64-token step grid, and fit the workspace's offset table; executed piece by
piece on the fp64 oracle with the device's offset rule and carried states, they reproduce
one whole-input run bit for bit; plus the pipelined call's host validation (no pointer is
dereferenced, no kernel launched).
"""
import ctypes

import numpy as np
import pytest
import torch

import chunked_linear_attention_kda_gb300 as kda
import kda_inputs as K
from chunked_linear_attention_kda_gb300 import build as kbuild


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kda.load_library()


pytestmark = pytest.mark.usefixtures("lib")   # the library is built before any test


def check_plan(cu, n_segments):
    cu = [int(c) for c in cu]
    n_seq, n_tok = len(cu) - 1, cu[-1]
    plan = kda.fwd_pipeline_plan(cu, n_segments)
    # tokens: contiguous, in order, each once
    t = 0
    for (t0, t1, n0, n1, h0c, hfc, seg) in plan:
        assert t0 == t and t1 >= t0
        t = t1
    assert t == n_tok
    # segments: non-decreasing, at most n_segments, at most 3 pieces each
    segs = [p[6] for p in plan]
    assert segs == sorted(segs) and (not segs or segs[-1] < n_segments)
    assert all(segs.count(s) <= 3 for s in set(segs))
    h0_reads = np.zeros(n_seq, int)
    hf_writes = np.zeros(n_seq, int)
    carried = None  # (sequence, segment) of the state in flight
    for (t0, t1, n0, n1, h0c, hfc, seg) in plan:
        assert 0 <= n0 < n1 <= n_seq
        if h0c or hfc:   # part of one cut sequence
            assert n1 - n0 == 1 and cu[n0] <= t0 and t1 <= cu[n0 + 1]
        else:            # a run of whole sequences
            assert t0 == cu[n0] and t1 == cu[n1]
        if h0c:
            assert n1 - n0 == 1 and carried == (n0, seg - 1), "carried state from the previous segment"
            assert cu[n0] < t0
            carried = None
        else:
            h0_reads[n0:n1] += 1
            assert t0 == cu[n0]
        if hfc:
            assert n1 - n0 == 1 and carried is None and t1 < cu[n0 + 1]
            carried = (n0, seg)
        else:
            hf_writes[n0:n1] += 1
            assert t1 == cu[n1]
        # every piece starts on its first sequence's 64-token step grid
        assert (t0 - cu[n0]) % 64 == 0
    assert carried is None
    assert (h0_reads == 1).all() and (hf_writes == 1).all()
    # the workspace's offset table holds every piece's n1 - n0 + 1 entries
    assert sum(p[3] - p[2] + 1 for p in plan) <= n_seq + 5 * n_segments + 1
    return plan


def test_one_long_sequence_cuts_into_equal_segments():
    plan = check_plan([0, 65536], 16)
    assert len(plan) == 16
    assert [(p[0], p[1]) for p in plan] == [(4096 * i, 4096 * (i + 1)) for i in range(16)]
    assert [(p[4], p[5]) for p in plan] == [(0, 1)] + [(1, 1)] * 14 + [(1, 0)]


def test_hand_worked_plan_with_an_empty_sequence():
    # 205 tokens: sequences of 5, 0 and 200 tokens; 4 segments. Target cuts 51, 102, 153
    # fall in the third sequence (start 5) and move down to 5 + 64 j: 5, 69, 133.
    plan = check_plan([0, 5, 5, 205], 4)
    assert plan == [(0, 5, 0, 2, 0, 0, 0), (5, 69, 2, 3, 0, 1, 1), (69, 133, 2, 3, 1, 1, 2),
                    (133, 205, 2, 3, 1, 0, 3)]
    # 40 tokens cut into 4: every target lies within 64 tokens of the third sequence's
    # start, so the only cut left is that start
    assert check_plan([0, 5, 5, 40], 4) == [(0, 5, 0, 2, 0, 0, 0), (5, 40, 2, 3, 0, 0, 1)]


@pytest.mark.parametrize("n_segments", [1, 2, 3, 7, 16, 64])
def test_random_packings(n_segments):
    rng = np.random.default_rng(1234 + n_segments)
    for trial in range(60):
        n_seq = int(rng.integers(1, 12))
        kind = trial % 3
        if kind == 0:      # mixed lengths with empty sequences
            lens = rng.integers(0, 300, n_seq) * (rng.random(n_seq) > 0.2)
        elif kind == 1:    # one long sequence among short ones
            lens = rng.integers(0, 20, n_seq)
            lens[rng.integers(0, n_seq)] = int(rng.integers(500, 5000))
        else:              # all empty or tiny
            lens = rng.integers(0, 3, n_seq)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        check_plan(cu, n_segments)


def test_no_tokens_runs_the_empty_sequences_once():
    plan = check_plan([0, 0, 0, 0], 8)
    assert plan == [(0, 0, 0, 3, 0, 0, 0)]


@pytest.mark.parametrize("cu,n_segments", [([0, 5, 3], 2), ([1, 5], 2), ([0, 5], 0),
                                            ([0, 5], 65)])
def test_plan_rejects_invalid_input(cu, n_segments):
    with pytest.raises(kda.KDAError):
        kda.fwd_pipeline_plan(cu, n_segments)


def test_workspace_bytes(lib):
    def al(b):
        return (b + 255) // 256 * 256
    for n_seq, H, d, S in [(1, 32, 128, 16), (17, 16, 128, 64), (0, 1, 1, 1), (5, 3, 40, 7)]:
        got = kda.fwd_pipelined_workspace_bytes(n_seq, H, d, d, S)
        assert got == 2 * al(H * d * d * 4) + al((n_seq + 5 * S + 1) * 4)
    assert kda.fwd_pipelined_workspace_bytes(1, 32, 128, 128, 0) == 0
    assert kda.fwd_pipelined_workspace_bytes(1, 32, 128, 128, 65) == 0
    assert kda.fwd_pipelined_workspace_bytes(-1, 32, 128, 128, 4) == 0


def _call(lib, ws_bytes, n_segments, ws_ptr=1 << 20, cu=(0, 64), n_tok=64):
    # every call here fails host validation: the fake pointers are never dereferenced
    fake = ctypes.c_void_p(1 << 16)   # 16-byte aligned
    host_cu = (ctypes.c_int32 * len(cu))(*cu)
    return lib.kda_chunk_fwd_from_host_pipelined(
        fake, fake, fake, fake, fake, None, ctypes.cast(host_cu, ctypes.c_void_p), fake, None,
        fake, fake, fake, fake, fake, None, fake, fake, None, ctypes.c_void_p(ws_ptr), ws_bytes,
        n_tok, len(cu) - 1, 2, 128, 128, n_segments, kda.KDA_BF16, None)


def test_pipelined_host_validation(lib):
    need = kda.fwd_pipelined_workspace_bytes(1, 2, 128, 128, 4)
    assert _call(lib, need, 0) == 1                     # n_segments outside [1, 64]
    assert _call(lib, need, 65) == 1
    assert _call(lib, need - 1, 4) == 1                 # workspace too small
    assert _call(lib, need, 4, ws_ptr=(1 << 20) + 16) == 1   # workspace not 256-byte aligned
    assert _call(lib, need, 4, cu=(0, 63)) == 1          # cu_seqlens does not end at n_tok
    assert b"cu_seqlens" in lib.kda_last_error()
    assert _call(lib, need, 4, cu=(0, 40, 30, 64)) == 1  # cu_seqlens decreases
    assert _call(lib, need, 4, cu=(2, 64)) == 1           # cu_seqlens does not start at 0


def run_plan_on_the_oracle(x, n_segments):
    """Execute the plan the way the pipelined entry point does -- each piece one forward
    call on its token range, with cu_seqlens clamp(cu[n0 + k], t0, t1) - t0, its start state
    from h0 or the carried state and its final state to h_final or the carried state --
    with the fp64 oracle standing in for the kernels."""
    from oracle import recurrence
    cu = [int(c) for c in x.cu_host]
    f64 = lambda t: None if t is None else t.detach().to("cpu", torch.float64).numpy()  # noqa: E731
    q, k, v, a, beta, h0 = (f64(t) for t in (x.q, x.k, x.v, x.a, x.beta, x.h0))
    out = np.full((x.n_tok, x.n_heads, x.d_v), np.nan)
    hf = np.full((x.n_seq, x.n_heads, x.d_k, x.d_v), np.nan)
    carry = [None, None]
    for (t0, t1, n0, n1, h0c, hfc, seg) in kda.fwd_pipeline_plan(cu, n_segments):
        local = [min(max(cu[n0 + j], t0), t1) - t0 for j in range(n1 - n0 + 1)]
        start = carry[seg & 1][None] if h0c else (None if h0 is None else h0[n0:n1])
        o, h = recurrence.kda_forward(q[t0:t1], k[t0:t1], v[t0:t1], a[t0:t1], beta[t0:t1],
                                      start, local)
        out[t0:t1] = o
        if hfc:
            carry[(seg + 1) & 1] = h[0]
        else:
            hf[n0:n1] = h
    return out, hf


@pytest.mark.parametrize("n_segments", [2, 5, 16, 64])
@pytest.mark.parametrize("lens,with_h0", [([2000], False), ([300, 0, 517, 33, 0], True),
                                          ([0, 900, 16, 17, 1000], True), ([0, 0], True)])
def test_executing_the_plan_reproduces_the_whole_run(n_segments, lens, with_h0):
    from oracle import recurrence
    x = K.make_inputs(lens, 2, 8, 6, dtype=torch.float32, seed=sum(lens) + n_segments,
                      h0_std=0.3 if with_h0 else None)
    o_ref, h_ref = recurrence.kda_forward(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_host)
    out, hf = run_plan_on_the_oracle(x, n_segments)
    # the carried fp64 state continues the token recurrence exactly: equal bit for bit
    assert np.array_equal(out, o_ref) and np.array_equal(hf, h_ref)
