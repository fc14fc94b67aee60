"""The bench's arithmetic on the CPU: the algorithmic bytes and flops its roofline divides
by (against the per-token figures derived from the operation's tensors and products), the
recorded-traffic lookup, and the parity figure it reports (the timed run's output against
the oracle on the sampled prefixes: zero for the oracle's own output, a planted error
inside the sample caught, rows outside the sample ignored).
"""
import numpy as np
import torch

import bench
import kda_inputs as K
from oracle import recurrence


def test_bytes_per_token_head():
    # bf16 q, k, v, o (4 x 256 B) + fp32 gate logits (512 B) + fp32 beta (4 B)
    assert bench.bytes_per_token_head(128, 128, 2) == 1540
    # the tiny fp32 case, d = 16: 4 x 16 x 4 + 16 x 4 + 4
    assert bench.bytes_per_token_head(16, 16, 4) == 324


def test_flops_per_token_head():
    # W S, Q~ S, K'^T U: 3 x 2 x 128^2; K~K^^T, Q~K^^T: 2 x 2 x 16 x 128; TB K~: 2 x 16 x 128;
    # TB V, P U: 2 x 2 x 16 x 128
    assert bench.flops_per_token_head(128, 128) == 3 * 2 * 128 * 128 + 6 * 16 * 128 + 4 * 16 * 128


def test_workload_bytes_and_decode_bytes():
    x = K.make_inputs([64], 1, 16, 16, dtype=torch.float32, seed=0)
    assert bench.algorithmic_bytes(x) == 64 * 324 + 16 * 16 * 4        # h_final, no h0
    x = K.make_inputs([40, 0, 9], 2, 16, 16, dtype=torch.float32, seed=0, h0_std=0.1)
    assert bench.algorithmic_bytes(x) == 49 * 2 * 324 + 2 * 3 * 2 * 16 * 16 * 4
    # the 64K workload: 65536 tokens x 32 heads x 1540 B + one h_final of 32 x 64 KiB
    assert 65536 * 32 * 1540 + 32 * 128 * 128 * 4 == 3231711232
    # one decode step per (sequence, head): fp32 state read and written, q/k/v/o, gate, beta
    assert bench.decode_bytes_per_seq_head(128, 128, 2) == 8 * 128 * 128 + 2 * 512 + 512 + 4


def test_recorded_traffic_needs_the_current_digest():
    digest = bench.kernel_source_digest()
    assert len(digest) == 16
    # a workload nobody recorded has no traffic figure
    assert bench.recorded_traffic("no-such-workload") is None


def test_prefix_parity_figure():
    x = K.make_inputs([300, 0, 1000, 50], 2, 16, 16, dtype=torch.float32, seed=3, h0_std=0.1)
    o, _ = recurrence.kda_forward(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_host)
    out = torch.from_numpy(o).float()
    tokens = 200
    px = K.prefix(x, tokens)
    o_ref, _ = recurrence.kda_forward(px.q, px.k, px.v, px.a, px.beta, px.h0, px.cu_host)
    whole, worst = bench.prefix_rel_l2(x, out, tokens, o_ref)
    assert whole < 1e-6 and worst < 1e-6
    bad = out.clone()
    bad[300 + 150] += 1.0          # inside sequence 2's first 200 tokens
    assert min(bench.prefix_rel_l2(x, bad, tokens, o_ref)) > 1e-2
    late = out.clone()
    late[300 + 250] += 1.0         # sequence 2 beyond the sample: not compared
    assert max(bench.prefix_rel_l2(x, late, tokens, o_ref)) < 1e-6
    # a whole-sequence sample compares every row
    o_all, _ = recurrence.kda_forward(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_host)
    assert np.isclose(bench.prefix_rel_l2(x, bad, 1000, o_all)[0],
                      np.linalg.norm(bad.numpy() - o_all) / np.linalg.norm(o_all))


def test_worst_head_is_not_diluted():
    """An error confined to one (sequence, head) pair: the worst-pair figure is that
    pair's own rel-L2, several times the whole-sample figure."""
    x = K.make_inputs([64, 64], 4, 16, 16, dtype=torch.float32, seed=4)
    o, _ = recurrence.kda_forward(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_host)
    bad = torch.from_numpy(o).float()
    bad[64:128, 2] *= 1.01         # sequence 1, head 2: 1% off
    whole, worst = bench.prefix_rel_l2(x, bad, 64, o)
    assert np.isclose(worst, 0.01, rtol=1e-4)
    assert whole < worst / 2


def test_state_parity_figure():
    r = np.random.default_rng(0).standard_normal((3, 4, 8, 8))
    g = torch.from_numpy(r).float()
    whole, worst = bench.state_rel_l2(g, r)
    assert whole < 1e-6 and worst < 1e-6
    g[1, 3] *= 1.02
    whole, worst = bench.state_rel_l2(g, r)
    assert np.isclose(worst, 0.02, rtol=1e-4) and whole < worst / 2
