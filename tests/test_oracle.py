"""The oracle against its pins (CPU only).

The oracle is the fp64 token-by-token recurrence in ``oracle/kda_oracle.c``. Nothing
here compares it with itself: every check is a closed form, an invariant, a different
algebra (unrolled transition products, the 16-token chunked form), or a number printed
by the source pages (``golden/bound_arithmetic.json``).
"""
import inspect
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import recurrence
from oracle.chunked import block_forward, chunked_forward, inverse_unit_lower
from tests import oracle_pins as P

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "bound_arithmetic.json")))


def oracle_fwd(mutant=0):
    def fwd(q, k, v, a, beta, h0, cu):
        return recurrence.kda_forward(q, k, v, a, beta, h0, cu, mutant=mutant, threads=2)
    return fwd


# ---------------------------------------------------------------- printed numbers

def test_golden_bound_arithmetic():
    g = GOLDEN
    C = g["tile_tokens"]["value"]
    gmin = g["g_min"]["value"]
    assert C * gmin == g["worst_chunk_log_decay"]["value"] == -80.0
    lo, hi = math.exp(C * gmin), math.exp(-C * gmin)
    for key, val in (("min_cumulative_decay", lo), ("max_reciprocal_decay", hi)):
        assert abs(val / g[key]["value"] - 1) <= g[key]["rtol"], (key, val)
    bf = torch.finfo(torch.bfloat16)
    # the printed normal-range top is bf16's (and fp32's) largest finite value
    assert abs(bf.max / g["normal_range_top"]["value"] - 1) <= g["normal_range_top"]["rtol"]
    # "a representable range of roughly 1e-38 to 3e38", shared by bf16 and fp32
    for fi in (bf, torch.finfo(torch.float32)):
        assert math.floor(math.log10(fi.tiny)) == math.floor(
            math.log10(g["bf16_fp32_range_low"]["value"]))
        assert math.floor(math.log10(fi.max)) == math.floor(
            math.log10(g["bf16_fp32_range_high"]["value"]))
    # exp(+-80) are finite, normal bf16 numbers
    hi_bf = torch.tensor(hi, dtype=torch.float32).to(torch.bfloat16).float().item()
    lo_bf = torch.tensor(lo, dtype=torch.float32).to(torch.bfloat16).float().item()
    assert math.isfinite(hi_bf) and abs(hi_bf / hi - 1) < 2 ** -8
    assert lo_bf >= bf.tiny and abs(lo_bf / lo - 1) < 2 ** -8
    # "about three orders of magnitude of headroom above the BF16 lower bound"
    assert round(math.log10(lo / bf.tiny)) == g["headroom_above_bf16_floor_orders"]["value"]
    # the 15-power reading: exp(-g_min * 15) = exp(75), also representable
    assert -gmin * (C - 1) == g["fifteen_power_bound_exponent"]["value"]
    assert math.exp(75.0) < hi < bf.max
    # single-step floor exp(-5) ~ 0.0067 and "forgetting has exceeded 99%"
    step = math.exp(gmin)
    assert abs(step / g["single_step_decay_floor"]["value"] - 1) <= 0.01
    assert 1 - step > g["forgetting_at_bound_exceeds"]["value"]
    # the unbounded counter-example: -40 per step, -640 per chunk, 1/Gamma = inf
    span = C * g["unbounded_step_example"]["value"]
    assert span == g["unbounded_chunk_example"]["value"]
    for dt in (torch.float32, torch.bfloat16):
        Gam = torch.exp(torch.tensor(span, dtype=dt))
        assert Gam.item() == 0.0 and torch.isinf(1.0 / Gam).item()
        assert torch.isfinite(torch.exp(torch.tensor(-C * gmin, dtype=dt))).item()


def test_oracle_bound_value():
    assert P.pin_bound_value(oracle_fwd(), GOLDEN) < 1e-13


# ---------------------------------------------------------------- pins

@pytest.mark.parametrize("name", sorted(P.PINS))
def test_oracle_pin(name):
    fn, tol = P.PINS[name]
    err = fn(oracle_fwd())
    assert err <= tol, f"{name}: {err:.3e} > {tol:.0e}"


def _run_pin_for_mutant(name, fwd, square):
    fn, tol = P.PINS[name]
    kw = {}
    if square:
        params = inspect.signature(fn).parameters
        if "dk" in params and "dv" in params:
            kw = {"dk": 4, "dv": 4}
    try:
        return fn(fwd, **kw) <= tol
    except AssertionError:
        return False


@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5, 6])
def test_planted_mistakes_are_caught(mutant):
    """Each mutant plants one plausible mistake in a copy of the oracle (decay after
    the write, output before the write, transposed state, flipped correction sign,
    bound dropped from the gate, output scale dropped); at least one pin must fail."""
    recurrence.build(mutant)
    fwd = oracle_fwd(mutant)
    square = mutant == 3   # the transposed-read mutant is only memory-safe for d_k == d_v
    passed = {name: _run_pin_for_mutant(name, fwd, square) for name in P.PINS}
    try:
        passed["bound_value"] = P.pin_bound_value(fwd, GOLDEN) < 1e-13
    except AssertionError:
        passed["bound_value"] = False
    assert not all(passed.values()), f"mutant {mutant} passed every pin: {passed}"


# ---------------------------------------------------------------- chunked algebra

@pytest.mark.parametrize("T", [1, 15, 16, 17, 53, 64])
@pytest.mark.parametrize("d", [4, 8, 16])
@pytest.mark.parametrize("gate", ["random", "bound", "mixed"])
def test_chunked_algebra_equals_recurrence(T, d, gate):
    rng = np.random.default_rng(100 + T * 7 + d)
    lengths = [T, max(1, T // 3)]
    q, k, v, a, beta, h0, cu = P._rand(rng, lengths, 2, d, d + 2)
    if gate == "bound":
        a[:] = np.inf                      # g = -5 exactly on every channel
    elif gate == "mixed":
        a[:, 0] = np.inf
        a[:, 1] = rng.normal(6.0, 1.0, size=a[:, 1].shape)
    o_ref, h_ref = recurrence.kda_forward(q, k, v, a, beta, h0, cu)
    for inverse in ("solve", "doubling"):
        o, hf = chunked_forward(q, k, v, a, beta, h0, cu, inverse=inverse)
        assert P.rel(o, o_ref) < 1e-12 and P.rel(hf, h_ref) < 1e-12, inverse


@pytest.mark.parametrize("T", [1, 16, 17, 63, 64, 65, 130, 200])
@pytest.mark.parametrize("gate", ["random", "bound", "mixed"])
def test_block_steps_of_64_tokens_equal_recurrence(T, gate):
    """Serial steps of 64 tokens assembled from 16-token bounded tiles (cross-tile factors
    all <= 1) reach the recurrence's result, including partial steps, at the bound."""
    rng = np.random.default_rng(300 + T)
    lengths = [T, max(1, T // 3)]
    q, k, v, a, beta, h0, cu = P._rand(rng, lengths, 2, 8, 6)
    if gate == "bound":
        a[:] = np.inf
    elif gate == "mixed":
        a[:, 0] = np.inf
        a[:, 1] = rng.normal(-6.0, 1.0, size=a[:, 1].shape)
    o_ref, h_ref = recurrence.kda_forward(q, k, v, a, beta, h0, cu)
    o, hf = block_forward(q, k, v, a, beta, h0, cu)
    assert P.rel(o, o_ref) < 1e-12 and P.rel(hf, h_ref) < 1e-12
    assert np.isfinite(o).all() and np.isfinite(hf).all()


def test_block_step_output_forms_agree():
    """scale (Q~B S + P U) and scale (P' V + Q' S) are the same output: one step from a
    random state, and whole runs of steps, against the recurrence."""
    from oracle.chunked import block_step
    rng = np.random.default_rng(44)
    B, dk, dv = 64, 8, 6
    q, k, v = rng.standard_normal((B, dk)), rng.standard_normal((B, dk)), rng.standard_normal((B, dv))
    a, beta = rng.normal(0.0, 2.0, (B, dk)), rng.uniform(0.1, 0.9, B)
    S = rng.standard_normal((dk, dv))
    o1, s1 = block_step(q, k, v, a, beta, S, form="qs_pu")
    o2, s2 = block_step(q, k, v, a, beta, S, form="pv_qs")
    assert P.rel(o1, o2) < 1e-12 and P.rel(s1, s2) < 1e-12
    # the step from S equals the recurrence from h0 = S
    o_ref, h_ref = recurrence.kda_forward(q[:, None], k[:, None], v[:, None], a[:, None], beta[:, None],
                                          S[None, None], [0, B])
    assert P.rel(o1, o_ref[:, 0]) < 1e-12 and P.rel(s1, h_ref[0, 0]) < 1e-12


def test_doubling_inverse_is_exact():
    rng = np.random.default_rng(11)
    for _ in range(5):
        A = np.tril(rng.standard_normal((16, 16)), -1)
        ref = np.linalg.inv(np.eye(16) + A)
        for m in ("solve", "doubling"):
            T = inverse_unit_lower(A, m)
            assert np.abs(T - ref).max() / np.abs(ref).max() < 1e-12


# ---------------------------------------------------------------- host-side behaviour

def test_packing_equals_separate_calls():
    rng = np.random.default_rng(12)
    lengths = [5, 0, 33, 16, 1]
    q, k, v, a, beta, h0, cu = P._rand(rng, lengths, 3, 6, 4)
    o, hf = recurrence.kda_forward(q, k, v, a, beta, h0, cu)
    for n, L in enumerate(lengths):
        s, e = cu[n], cu[n + 1]
        o1, h1 = recurrence.kda_forward(q[s:e], k[s:e], v[s:e], a[s:e], beta[s:e],
                                        h0[n:n + 1], [0, L])
        assert np.array_equal(o[s:e], o1) and np.array_equal(hf[n], h1[0])
    assert np.array_equal(hf[1], h0[1])          # empty sequence keeps h0


def test_resume_equals_one_run():
    rng = np.random.default_rng(13)
    T = 50
    q, k, v, a, beta, h0, cu = P._rand(rng, [T], 2, 5, 5)
    o, hf = recurrence.kda_forward(q, k, v, a, beta, h0, cu)
    for t1 in (1, 16, 23):
        oa, ha = recurrence.kda_forward(q[:t1], k[:t1], v[:t1], a[:t1], beta[:t1], h0, [0, t1])
        ob, hb = recurrence.kda_forward(q[t1:], k[t1:], v[t1:], a[t1:], beta[t1:], ha,
                                        [0, T - t1])
        assert np.allclose(np.concatenate([oa, ob]), o, rtol=0, atol=1e-13)
        assert np.allclose(hb, hf, rtol=0, atol=1e-13)


def test_thread_count_does_not_change_result():
    rng = np.random.default_rng(14)
    q, k, v, a, beta, h0, cu = P._rand(rng, [40, 7, 19], 4, 8, 8)
    r1 = recurrence.kda_forward(q, k, v, a, beta, h0, cu, threads=1)
    r8 = recurrence.kda_forward(q, k, v, a, beta, h0, cu, threads=8)
    assert np.array_equal(r1[0], r8[0]) and np.array_equal(r1[1], r8[1])


def test_rejects_bad_offsets():
    rng = np.random.default_rng(15)
    q, k, v, a, beta, _, _ = P._rand(rng, [4], 1, 2, 2)
    with pytest.raises(AssertionError):
        recurrence.kda_forward(q, k, v, a, beta, None, [0, 3, 2])


# ---------------------------------------------------------------- decode step

def test_decode_steps_chain_to_the_forward_pass():
    """T decode steps from h0, each feeding the next its state, reproduce the T-token
    forward pass of every sequence (the recurrence consumes tokens one at a time)."""
    rng = np.random.default_rng(16)
    B, T, H, dk, dv = 3, 7, 2, 5, 4
    q, k, v, a, beta, h0, cu = P._rand(rng, [T] * B, H, dk, dv)
    o_ref, h_ref = recurrence.kda_forward(q, k, v, a, beta, h0, cu)
    state = h0.copy()
    outs = []
    for t in range(T):
        rows = [b * T + t for b in range(B)]
        o, state = recurrence.decode_step(q[rows], k[rows], v[rows], a[rows], beta[rows], state)
        outs.append(o)
    got = np.stack(outs, axis=1).reshape(B * T, H, dv)   # [B, T] -> packed token order
    assert np.allclose(got, o_ref, rtol=0, atol=1e-13)
    assert np.allclose(state, h_ref, rtol=0, atol=1e-13)


def test_decode_step_pure_decay_closed_form():
    """beta = 0 writes nothing and a saturated gate decays every channel by exactly
    exp(-5): the state becomes exp(-5) S and the output d_k^-1/2 exp(-5) S^T q."""
    rng = np.random.default_rng(17)
    B, H, dk, dv = 2, 3, 6, 5
    q = rng.standard_normal((B, H, dk))
    k = rng.standard_normal((B, H, dk))
    v = rng.standard_normal((B, H, dv))
    a = np.full((B, H, dk), 80.0)            # sigmoid(80) = 1 to double precision
    beta = np.zeros((B, H))
    S = rng.standard_normal((B, H, dk, dv))
    o, S1 = recurrence.decode_step(q, k, v, a, beta, S)
    assert np.allclose(S1, math.exp(-5.0) * S, rtol=1e-14, atol=0)
    want = math.exp(-5.0) / math.sqrt(dk) * np.einsum("bhkv,bhk->bhv", S, q)
    assert np.allclose(o, want, rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- backward oracle

from oracle import backward as B  # noqa: E402


def test_backward_oracle_forward_is_the_recurrence():
    """The function the backward oracle differentiates equals the pinned C oracle."""
    rng = np.random.default_rng(21)
    q, k, v, a, beta, h0, cu = P._rand(rng, [6, 0, 17], 2, 5, 4)
    o_ref, h_ref = recurrence.kda_forward(q, k, v, a, beta, h0, cu)
    t = lambda x: torch.as_tensor(x)  # noqa: E731
    o, hf = B.forward_torch(t(q), t(k), t(v), t(a), t(beta), t(h0), list(cu))
    assert np.allclose(o.numpy(), o_ref, rtol=0, atol=1e-13)
    assert np.allclose(hf.numpy(), h_ref, rtol=0, atol=1e-13)


def _loss(q, k, v, a, beta, h0, cu, dout, dhf):
    o, hf = recurrence.kda_forward(q, k, v, a, beta, h0, cu)
    return float(np.sum(o * dout) + np.sum(hf * dhf))


def test_backward_oracle_matches_finite_differences():
    """Central differences of the C oracle's loss, element by element for every input
    (independent of automatic differentiation)."""
    rng = np.random.default_rng(22)
    lengths, H, dk, dv = [5, 0, 3], 2, 3, 2
    q, k, v, a, beta, h0, cu = P._rand(rng, lengths, H, dk, dv)
    N = sum(lengths)
    dout = rng.standard_normal((N, H, dv))
    dhf = rng.standard_normal((len(lengths), H, dk, dv))
    g = B.kda_backward(q, k, v, a, beta, h0, cu, dout, dhf)
    args = {"dq": q, "dk": k, "dv": v, "da": a, "dbeta": beta, "dh0": h0}
    eps = 1e-6
    for name, x in args.items():
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            keep = x[idx]
            x[idx] = keep + eps
            lp = _loss(q, k, v, a, beta, h0, cu, dout, dhf)
            x[idx] = keep - eps
            lm = _loss(q, k, v, a, beta, h0, cu, dout, dhf)
            x[idx] = keep
            fd[idx] = (lp - lm) / (2 * eps)
        err = np.abs(g[name] - fd).max() / max(np.abs(fd).max(), 1e-12)
        assert err < 1e-7, (name, err)


def test_backward_oracle_one_token_closed_form():
    """One token from a zero state: S = beta k v^T, o = s beta (q.k) v, so
    dv = s beta (q.k) dO, dbeta = s (q.k)(v.dO), dq = s beta (v.dO) k,
    dk = s beta (v.dO) q, da = 0 (the decay multiplies a zero state); and since
    S_1 = (I - beta k k^T) Diag(gamma) S_0 + beta k v^T, dh0 = Diag(gamma) (I - beta k k^T)
    s q dO^T."""
    rng = np.random.default_rng(23)
    H, dk, dv = 3, 4, 5
    q = rng.standard_normal((1, H, dk))
    k = rng.standard_normal((1, H, dk))
    v = rng.standard_normal((1, H, dv))
    a = rng.standard_normal((1, H, dk))
    beta = rng.uniform(0.1, 0.9, (1, H))
    dO = rng.standard_normal((1, H, dv))
    g = B.kda_backward(q, k, v, a, beta, None, [0, 1], dO)
    s = dk ** -0.5
    qk = np.einsum("hk,hk->h", q[0], k[0])
    vdo = np.einsum("hv,hv->h", v[0], dO[0])
    b = beta[0]
    assert np.allclose(g["dv"][0], (s * b * qk)[:, None] * dO[0], atol=1e-14)
    assert np.allclose(g["dbeta"][0], s * qk * vdo, atol=1e-14)
    assert np.allclose(g["dq"][0], (s * b * vdo)[:, None] * k[0], atol=1e-14)
    assert np.allclose(g["dk"][0], (s * b * vdo)[:, None] * q[0], atol=1e-14)
    assert np.allclose(g["da"], 0.0, atol=1e-15)
    gam = np.exp(-5.0 / (1.0 + np.exp(-a[0])))
    for h in range(H):
        Ph = np.eye(dk) - b[h] * np.outer(k[0, h], k[0, h])
        want = gam[h][:, None] * (Ph @ (s * np.outer(q[0, h], dO[0, h])))
        assert np.allclose(g["dh0"][0, h], want, atol=1e-13)


# ---------------------------------------------------------------- unbounded contrast gate

def test_softplus_gate_oracle_equals_the_c_oracle_reparameterised():
    """g = -softplus(a) is g_min sigmoid(a') with g_min = -1000 and
    a' = logit(softplus(a) / 1000): the C oracle, given those, runs the softplus-gated
    recurrence, and must agree with the torch loop's softplus gate."""
    rng = np.random.default_rng(24)
    q, k, v, a, beta, h0, cu = P._rand(rng, [9, 20], 2, 5, 4)
    a = a * 3.0
    o, hf = B.kda_forward_gate(q, k, v, a, beta, h0, cu, gate="softplus")
    sp = np.logaddexp(0.0, a)                   # softplus, stable
    r = sp / 1000.0
    a2 = np.log(r) - np.log1p(-r)              # logit
    o2, hf2 = recurrence.kda_forward(q, k, v, a2, beta, h0, cu, g_min=-1000.0)
    assert np.allclose(o, o2, rtol=0, atol=1e-11)
    assert np.allclose(hf, hf2, rtol=0, atol=1e-11)


def test_bounded_gate_of_the_torch_loop_is_the_c_oracle():
    rng = np.random.default_rng(25)
    q, k, v, a, beta, h0, cu = P._rand(rng, [13], 3, 4, 6)
    o, hf = B.kda_forward_gate(q, k, v, a, beta, h0, cu, gate="bounded")
    o2, hf2 = recurrence.kda_forward(q, k, v, a, beta, h0, cu)
    assert np.allclose(o, o2, rtol=0, atol=1e-13) and np.allclose(hf, hf2, rtol=0, atol=1e-13)


def test_unbounded_chunk_overflows_where_the_bound_cannot():
    """A log-decay of -40 per token over a 16-token chunk gives G = -640 and
    exp(-G) = exp(640), which overflows fp32 and bf16; the bound keeps |G| <= 80 and
    exp(80) = 5.54e34 finite in both."""
    assert np.isinf(np.float32(np.exp(np.float64(640.0))))
    assert float(torch.tensor(640.0).exp().to(torch.bfloat16)) == float("inf")
    assert np.isfinite(np.float32(np.exp(80.0)))
    assert np.isfinite(float(torch.tensor(80.0).exp().to(torch.bfloat16)))
    a = torch.tensor(40.0, dtype=torch.float64)
    assert abs(float(B.log_decay(a, "softplus")) + 40.0) < 1e-15  # softplus(40) = 40 + 4e-18
    assert float(B.log_decay(torch.tensor(1e6, dtype=torch.float64), "bounded")) >= -5.0


# ---------------------------------------------------------------- gate projection oracle

def test_gate_projection_oracle_brute_force_and_exact_integers():
    """The fp64 product against a triple loop, and exactly on small integers (every
    partial sum an integer below 2^53)."""
    from oracle import projection
    rng = np.random.default_rng(26)
    x = rng.standard_normal((5, 7))
    w = rng.standard_normal((3, 7))
    b = rng.standard_normal(3)
    a = projection.gate_projection(x, w, b)
    for i in range(5):
        for j in range(3):
            ref = b[j]
            for kk in range(7):
                ref += x[i, kk] * w[j, kk]
            assert abs(a[i, j] - ref) < 1e-12
    xi = rng.integers(-50, 50, (6, 64)).astype(np.float64)
    wi = rng.integers(-50, 50, (4, 64)).astype(np.float64)
    ai = projection.gate_projection(xi, wi)
    assert np.array_equal(ai, (xi[:, None, :] * wi[None, :, :]).sum(-1))
    assert np.array_equal(projection.gate_projection(xi, wi, None), ai)
