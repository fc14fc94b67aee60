"""Seeded synthetic inputs for the KDA chunked forward.

This module is shared by the oracle side and the CUDA side of the tests and by the
benchmark. It holds input recipes only -- shapes, seeds and value distributions --
and none of the method's arithmetic (no gate, no decay, no state).

Layout (packed, token-major, contiguous):
    q, k, a : [N_tok, H, d_k]     v : [N_tok, H, d_v]     beta : [N_tok, H]
    h0      : [n_seq, H, d_k, d_v] float32 or None (zero start state)
    cu_seqlens : int32 [n_seq + 1] on the device, plus a host copy ``cu_host``.

Workloads (the context ladder 8K -> 64K -> 256K -> 1M of "Architecting Long-Context
LLMs", §5.1, sets the lengths; there is no dataset):
    0 tiny-fp32      B=1 H=1  T=64      d=16   all fp32, h0 = 0
    1 single-bf16    B=1 H=4  T=4096    d=128  h0 ~ N(0, 0.1^2)
    2 bound-stress   B=2 H=16 T=8192    d=128  heads [0,8): a ~ N(+6,1), [8,16): a ~ N(-6,1)
    3 context-64K    B=1 H=32 T=65536   d=128  h0 = 0
    4 varlen-1M      H=16 d=128, 16 lengths ~ U{4096..131072} then one of 1,048,576,
                     per-sequence h0 ~ N(0, 0.1^2)
    5 context-256K   B=1 H=32 T=262144  d=128  h0 = 0 (the ladder's 256K point)
    6 delta-64K      B=1 H=32 T=65536   d=128  a ~ N(-6,1) on every head (g ~ -0.012: a
                     near-pure delta rule, little decay to damp rounding in the state),
                     h0 ~ N(0, 0.1^2)
Common distributions: q, k ~ N(0,1) then L2-normalised per token and head in fp32
(x / max(|x|_2, 1e-6)) before the cast; v ~ N(0,1); beta = sigmoid(N(0,1));
gate logits a ~ N(0, 2^2) unless stated. q/k/v (and the output) are bf16 except in
workload 0; a, beta, h0 and the final state are fp32 everywhere.
Generation order inside one torch.Generator on the tensors' device, seeded with
1000 + workload index: q, k, v, beta, a, h0. Workload 4 draws its lengths first from a
CPU generator with the same seed, so the packing does not depend on the device.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import torch

SEED_BASE = 1000

WORKLOADS = {
    0: "tiny-fp32-B1-H1-T64-d16",
    1: "single-seq-bf16-B1-H4-T4096-d128",
    2: "decay-bound-stress-B2-H16-T8192-d128",
    3: "context-64K-B1-H32-T65536-d128",
    4: "packed-varlen-1M-H16-d128",
    5: "context-256K-B1-H32-T262144-d128",
    6: "near-delta-rule-64K-B1-H32-T65536-d128",
}


@dataclasses.dataclass
class KDAInputs:
    name: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    a: torch.Tensor
    beta: torch.Tensor
    h0: Optional[torch.Tensor]
    cu_seqlens: torch.Tensor          # int32, on the tensors' device
    cu_host: list                     # python ints
    dtype: torch.dtype                # q/k/v/out dtype

    @property
    def n_tok(self) -> int:
        return self.q.shape[0]

    @property
    def n_seq(self) -> int:
        return len(self.cu_host) - 1

    @property
    def n_heads(self) -> int:
        return self.q.shape[1]

    @property
    def d_k(self) -> int:
        return self.q.shape[2]

    @property
    def d_v(self) -> int:
        return self.v.shape[2]

    def lengths(self) -> list:
        return [self.cu_host[i + 1] - self.cu_host[i] for i in range(self.n_seq)]


def _normal(shape, gen, device, mean=0.0, std=1.0):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x


def _l2_normalised(shape, gen, device, dtype):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    n = torch.linalg.vector_norm(x, dim=-1, keepdim=True).clamp_min_(1e-6)
    return x.div_(n).to(dtype)


def make_inputs(lengths: Sequence[int], n_heads: int, d_k: int, d_v: int, *,
                dtype=torch.bfloat16, device="cpu", seed: int = 0,
                gate_mean=0.0, gate_std=2.0, h0_std: Optional[float] = None,
                name: str = "custom", gen: Optional[torch.Generator] = None) -> KDAInputs:
    """Generic recipe. ``gate_mean`` / ``gate_std`` may be per-head sequences."""
    device = torch.device(device)
    if gen is None:
        gen = torch.Generator(device=device)
        gen.manual_seed(seed)
    lengths = [int(x) for x in lengths]
    N = sum(lengths)
    H = n_heads
    q = _l2_normalised((N, H, d_k), gen, device, dtype)
    k = _l2_normalised((N, H, d_k), gen, device, dtype)
    v = _normal((N, H, d_v), gen, device).to(dtype)
    beta = torch.sigmoid(_normal((N, H), gen, device))
    if isinstance(gate_mean, (int, float)) and isinstance(gate_std, (int, float)):
        a = _normal((N, H, d_k), gen, device, gate_mean, gate_std)
    else:
        means = torch.as_tensor(list(gate_mean), dtype=torch.float32, device=device)
        stds = torch.as_tensor(list(gate_std), dtype=torch.float32, device=device)
        a = _normal((N, H, d_k), gen, device)
        a.mul_(stds.view(1, H, 1)).add_(means.view(1, H, 1))
    h0 = None
    if h0_std is not None:
        h0 = _normal((len(lengths), H, d_k, d_v), gen, device, 0.0, h0_std)
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + L)
    cu_dev = torch.tensor(cu, dtype=torch.int32, device=device)
    return KDAInputs(name, q, k, v, a, beta, h0, cu_dev, cu, dtype)


def workload_lengths(index: int, gen: Optional[torch.Generator] = None) -> list:
    if index == 0:
        return [64]
    if index == 1:
        return [4096]
    if index == 2:
        return [8192, 8192]
    if index == 3:
        return [65536]
    if index == 4:
        # lengths come from a CPU generator so they do not depend on the device
        g = torch.Generator()
        g.manual_seed(SEED_BASE + 4 if gen is None else gen.initial_seed())
        lens = torch.randint(4096, 131072 + 1, (16,), generator=g)
        return [int(x) for x in lens.tolist()] + [1 << 20]
    if index == 5:
        return [1 << 18]
    if index == 6:
        return [65536]
    raise ValueError(f"unknown workload {index}")


def make_workload(index: int, device="cpu", seed: Optional[int] = None,
                  max_len: Optional[int] = None) -> KDAInputs:
    """Workload ``index`` (0..6) exactly as listed in the module docstring.
    ``max_len`` truncates every sequence (same recipe, fewer tokens), for host-side
    samples of the large workloads."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(SEED_BASE + index if seed is None else seed)
    lengths = workload_lengths(index, gen)
    if max_len is not None:
        lengths = [min(L, max_len) for L in lengths]
    name = WORKLOADS[index]
    if index == 0:
        return make_inputs(lengths, 1, 16, 16, dtype=torch.float32, device=device,
                           name=name, gen=gen)
    if index == 1:
        return make_inputs(lengths, 4, 128, 128, device=device, h0_std=0.1, name=name,
                           gen=gen)
    if index == 2:
        H = 16
        means = [6.0] * (H // 2) + [-6.0] * (H // 2)
        return make_inputs(lengths, H, 128, 128, device=device, gate_mean=means,
                           gate_std=[1.0] * H, name=name, gen=gen)
    if index == 3:
        return make_inputs(lengths, 32, 128, 128, device=device, name=name, gen=gen)
    if index == 4:
        return make_inputs(lengths, 16, 128, 128, device=device, h0_std=0.1, name=name,
                           gen=gen)
    if index == 5:
        return make_inputs(lengths, 32, 128, 128, device=device, name=name, gen=gen)
    if index == 6:
        return make_inputs(lengths, 32, 128, 128, device=device, gate_mean=-6.0, gate_std=1.0,
                           h0_std=0.1, name=name, gen=gen)
    raise ValueError(index)


def workload_size(index: int) -> dict:
    """Token and token-head counts without generating any tensor."""
    lens = workload_lengths(index)
    H = {0: 1, 1: 4, 2: 16, 3: 32, 4: 16, 5: 32, 6: 32}[index]
    return {"tokens": sum(lens), "heads": H, "token_heads": sum(lens) * H,
            "n_seq": len(lens)}


def slice_heads(x: KDAInputs, heads: Sequence[int]) -> KDAInputs:
    """A view of a subset of heads (contiguous copies), for sampled oracle checks."""
    idx = torch.as_tensor(list(heads), dtype=torch.long, device=x.q.device)
    sel = lambda t: t.index_select(1, idx).contiguous()  # noqa: E731
    h0 = None if x.h0 is None else x.h0.index_select(1, idx).contiguous()
    return KDAInputs(x.name, sel(x.q), sel(x.k), sel(x.v), sel(x.a),
                     x.beta.index_select(1, idx).contiguous(), h0, x.cu_seqlens,
                     list(x.cu_host), x.dtype)


def prefix(x: KDAInputs, max_len: int) -> KDAInputs:
    """Re-pack the first ``max_len`` tokens of every sequence (causal prefixes)."""
    parts = []
    lens = []
    for i in range(x.n_seq):
        s, e = x.cu_host[i], x.cu_host[i + 1]
        L = min(e - s, max_len)
        parts.append((s, s + L))
        lens.append(L)
    cat = lambda t: torch.cat([t[s:e] for s, e in parts], 0).contiguous()  # noqa: E731
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)
    cu_dev = torch.tensor(cu, dtype=torch.int32, device=x.q.device)
    return KDAInputs(x.name + f"-prefix{max_len}", cat(x.q), cat(x.k), cat(x.v),
                     cat(x.a), cat(x.beta), x.h0, cu_dev, cu, x.dtype)


__all__ = ["KDAInputs", "make_inputs", "make_workload", "workload_size", "slice_heads",
           "prefix", "WORKLOADS", "SEED_BASE"]
