"""Failure detection on the GPU without any fault: a pipeline wait that can never
complete gives up after its limit, sets the device status word and returns; a healthy
forward pass leaves the word clear. Also the launch counter the benchmark reports."""
import pytest
import torch

import chunked_linear_attention_kda_gb300 as kda
import kda_inputs as K

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports():
    returned, flags = kda.selftest_bounded_wait(limit_cycles=2_000_000)  # about 1 ms
    assert returned == 1, "the never-completing wait must give up, not complete"
    assert flags & 1, "giving up must set bit 0 of the device status word"
    assert kda.read_device_flags() == 0, "reading with reset clears the word"


def test_healthy_forward_leaves_status_clear():
    kda.read_device_flags(reset=True)
    x = K.make_inputs([300, 17], 4, 128, 128, device="cuda", seed=31, h0_std=0.1)
    kda.chunk_fwd(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_seqlens)
    assert kda.read_device_flags() == 0


def test_one_launch_per_call():
    x = K.make_inputs([100], 2, 128, 128, device="cuda", seed=32)
    n0 = kda.kernel_launch_count()
    for _ in range(3):
        kda.chunk_fwd(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_seqlens)
    torch.cuda.synchronize()
    assert kda.kernel_launch_count() - n0 == 3
