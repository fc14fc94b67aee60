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
    ref = kda.chunk_bwd(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_seqlens, dout, dhf)
    for _ in range(2):
        got = kda.chunk_bwd_static_scratch(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_seqlens,
                                           dout, dhf)
        torch.cuda.synchronize()
        for r, o in zip(ref, got):
            assert torch.equal(r, o)
