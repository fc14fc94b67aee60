"""Multi-rank host logic on CPU with the gloo backend (world size 2).

The forward function on each rank is the fp64 oracle (test infrastructure); what is
under test is the partitioning and the state hand-off, which are the same on GPUs.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from chunked_linear_attention_kda_gb300 import sharding
from oracle import recurrence
from tests import oracle_pins as P


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_fwd(q, k, v, a, beta, h0, cu):
    o, hf = recurrence.kda_forward(q, k, v, a, beta, h0, cu.tolist(), threads=1)
    return torch.from_numpy(o), torch.from_numpy(hf)


def _inputs(seed, lengths, H=2, dk=4, dv=3):
    rng = np.random.default_rng(seed)
    q, k, v, a, beta, h0, cu = P._rand(rng, lengths, H, dk, dv)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x))  # noqa: E731
    return t(q), t(k), t(v), t(a), t(beta), t(h0), torch.from_numpy(cu)


def test_partition_sequences_covers_each_once_and_balances():
    lengths = [5, 100, 3, 40, 40, 1, 77, 0, 12]
    for world in (1, 2, 3, 4, 8, 12):
        parts = sharding.partition_sequences(lengths, world)
        assert len(parts) == world and parts[0][0] == 0 and parts[-1][1] == len(lengths)
        assert all(a <= b for a, b in parts) and all(parts[i][1] == parts[i + 1][0]
                                                     for i in range(world - 1))
    tokens = [sum(lengths[a:b]) for a, b in sharding.partition_sequences(lengths, 2)]
    assert max(tokens) - min(tokens) <= max(lengths)


def test_partition_heads_and_segments():
    assert sharding.partition_heads(10, 3) == [(0, 4), (4, 7), (7, 10)]
    assert sharding.partition_heads(2, 4) == [(0, 1), (1, 2), (2, 2), (2, 2)]
    segs = sharding.segment_bounds(1000, 3)
    assert segs[0][0] == 0 and segs[-1][1] == 1000
    assert all(b % 16 == 0 for _, b in segs[:-1])


def _run_ranks(fn, world=2):
    port = _free_port()
    mp.spawn(fn, args=(world, port), nprocs=world, join=True)


def _sequence_shard_rank(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    lengths = [7, 33, 0, 16, 50, 1]
    q, k, v, a, beta, h0, cu = _inputs(21, lengths)
    b, e = sharding.partition_sequences(lengths, world)[rank]
    s, t = int(cu[b]), int(cu[e])
    cu_r = cu[b:e + 1] - cu[b]
    o, hf = _oracle_fwd(q[s:t], k[s:t], v[s:t], a[s:t], beta[s:t], h0[b:e], cu_r)
    # the check gathers results; the forward pass itself exchanged nothing
    outs = [None] * world
    dist.all_gather_object(outs, (b, e, s, t, o.numpy(), hf.numpy()))
    if rank == 0:
        o_ref, h_ref = _oracle_fwd(q, k, v, a, beta, h0, cu)
        for b_, e_, s_, t_, o_, h_ in outs:
            assert np.array_equal(o_, o_ref.numpy()[s_:t_])
            assert np.array_equal(h_, h_ref.numpy()[b_:e_])
    dist.destroy_process_group()


def test_sequence_sharding_two_ranks_gloo():
    _run_ranks(_sequence_shard_rank)


def _time_split_rank(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    T = 83
    q, k, v, a, beta, h0, cu = _inputs(22, [T])
    s, t = sharding.segment_bounds(T, world)[rank]
    seg = {"q": q[s:t], "k": k[s:t], "v": v[s:t], "gate_logits": a[s:t], "beta": beta[s:t],
           "cu_seqlens": torch.tensor([0, t - s])}
    start = h0.clone() if rank == 0 else torch.empty_like(h0)
    o, hf = sharding.time_split_forward(_oracle_fwd, seg, start, rank, world)
    outs = [None] * world
    dist.all_gather_object(outs, (s, t, o.numpy(), hf.numpy()))
    if rank == 0:
        o_ref, h_ref = _oracle_fwd(q, k, v, a, beta, h0, cu)
        got = np.concatenate([x[2] for x in sorted(outs, key=lambda x: x[0])])
        assert np.abs(got - o_ref.numpy()).max() < 1e-12
        assert np.abs(outs[-1][3] - h_ref.numpy()).max() < 1e-12
    dist.destroy_process_group()


def test_time_split_state_handoff_two_ranks_gloo():
    _run_ranks(_time_split_rank)


def _affine_split_rank(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    T = 101
    q, k, v, a, beta, h0, cu = _inputs(23, [T], H=2, dk=4, dv=3)
    s, t = sharding.segment_bounds(T, world)[rank]
    seg = {"q": q[s:t], "k": k[s:t], "v": v[s:t], "gate_logits": a[s:t], "beta": beta[s:t],
           "cu_seqlens": torch.tensor([0, t - s])}
    start = h0.clone() if rank == 0 else torch.full_like(h0, float("nan"))  # only rank 0's counts
    combine = lambda M, S, B: torch.einsum("hij,hjk->hik", M, S) + B  # noqa: E731
    o, hf = sharding.affine_time_split_forward(_oracle_fwd, combine, seg, start, rank, world)
    outs = [None] * world
    dist.all_gather_object(outs, (s, t, o.numpy(), hf.numpy()))
    if rank == 0:
        o_ref, h_ref = _oracle_fwd(q, k, v, a, beta, h0, cu)
        got = np.concatenate([x[2] for x in sorted(outs, key=lambda x: x[0])])
        assert np.abs(got - o_ref.numpy()).max() < 1e-10
        assert np.abs(outs[-1][3] - h_ref.numpy()).max() < 1e-10
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_affine_time_split_parallel_segments_gloo(world):
    _run_ranks(_affine_split_rank, world=world)


def test_time_split_needs_receive_buffer():
    with pytest.raises(ValueError):
        sharding.time_split_forward(_oracle_fwd, {}, None, 1, 2)
