"""The no-allocation backward entry point (``kda_chunk_bwd_static_scratch``): its
checkpoints live in the library's fixed device scratch array instead of a caller
workspace. It must give exactly the results of ``kda_chunk_bwd`` -- the same kernels on
the same data -- on two calls in a row (the second finds the first call's contents in the
scratch, which nothing may depend on), and refuse problems larger than the scratch
before doing any device work. Collected last: it leaves the scratch array of the
loaded library in use by nothing else.
"""
import ctypes

import pytest
import torch

import chunked_linear_attention_kda_gb300 as kda
import kda_inputs as K

FAKE = 0x100000


def test_oversize_problem_is_refused_on_the_host():
    lib = kda.load_library(build_if_missing=True)
    P = ctypes.c_void_p
    n_tok, H, d = 1 << 20, 32, 128        # ~17 GB of checkpoints, far above 64 MiB
    assert lib.kda_chunk_bwd_workspace_bytes(n_tok, 1, H, d, d) > (64 << 20)
    st = lib.kda_chunk_bwd_static_scratch(*[P(FAKE * (i + 1)) for i in range(15)],
                                          n_tok, 1, H, d, d, 1, None)
    assert st == 2, lib.kda_last_error()
    assert "static scratch" in lib.kda_last_error().decode()


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_same_results_as_the_workspace_entry_point_twice(dtype):
    lengths, H, d = [40, 0, 17, 64], 2, 128
    x = K.make_inputs(lengths, H, d, d, dtype=dtype, device="cuda", seed=9, h0_std=0.3)
    g = torch.Generator(device="cpu").manual_seed(9)
    dout = torch.randn((x.n_tok, H, d), generator=g).to("cuda", dtype)
    dhf = torch.randn((x.n_seq, H, d, d), generator=g).to("cuda")
    lib = kda.load_library()
    assert lib.kda_chunk_bwd_workspace_bytes(x.n_tok, x.n_seq, H, d, d) <= (64 << 20)
    # an unrelated, larger problem first, so the scratch holds other data when the
    # compared calls run
    y = K.make_inputs([300, 129], 4, d, d, dtype=dtype, device="cuda", seed=31, h0_std=0.5)
    ydout = torch.randn((y.n_tok, 4, d), generator=g).to("cuda", dtype)
    kda.chunk_bwd_static_scratch(y.q, y.k, y.v, y.a, y.beta, y.h0, y.cu_seqlens, ydout, None)
    ref = kda.chunk_bwd(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_seqlens, dout, dhf)
    for _ in range(2):
        got = kda.chunk_bwd_static_scratch(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_seqlens,
                                           dout, dhf)
        torch.cuda.synchronize()
        for r, o in zip(ref, got):
            assert torch.equal(r, o)


@pytest.mark.gpu
def test_a_call_allocates_no_device_memory():
    """Around one call through the C ABI (outputs allocated beforehand), neither torch's
    allocator nor the device's free memory changes."""
    lengths, H, d = [100, 37], 2, 128
    x = K.make_inputs(lengths, H, d, d, device="cuda", seed=10, h0_std=0.3)
    dout = torch.randn((x.n_tok, H, d), device="cuda").to(x.dtype)
    grads = [torch.empty_like(t) for t in (x.q, x.k, x.v, x.a, x.beta)]
    dh0 = torch.empty((x.n_seq, H, d, d), dtype=torch.float32, device="cuda")
    lib = kda.load_library()
    P = ctypes.c_void_p
    ptr = lambda t: P(t.data_ptr()) if t is not None else None  # noqa: E731

    def call():
        st = lib.kda_chunk_bwd_static_scratch(
            ptr(x.q), ptr(x.k), ptr(x.v), ptr(x.a), ptr(x.beta), ptr(x.h0), ptr(x.cu_seqlens),
            ptr(dout), None, *[ptr(t) for t in grads], ptr(dh0), x.n_tok, x.n_seq, H, d, d,
            kda.KDA_BF16, P(torch.cuda.current_stream().cuda_stream))
        assert st == 0, lib.kda_last_error()
        torch.cuda.synchronize()

    call()   # modules and the scratch address resolved on the first call
    alloc0, (free0, _) = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()
    call()
    alloc1, (free1, _) = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()
    assert alloc1 == alloc0 and free1 == free0
