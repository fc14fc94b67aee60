"""Device-side checks through the C ABI: the cu_seqlens validator (bad offsets are made
on the host and handed only to the validator, never to a forward kernel) and the
non-finite counter, on values planted on the host."""
import pytest
import torch

import chunked_linear_attention_kda_gb300 as kda
import kda_inputs as K

pytestmark = pytest.mark.gpu
DEV = "cuda"
INT_MAX = 2**31 - 1


@pytest.mark.parametrize("cu,n_tok,bits,first", [
    ([0, 5, 5, 40], 40, 0, INT_MAX),          # valid, with an empty sequence
    ([0], 0, 0, INT_MAX),                     # no sequence at all
    ([1, 5, 40], 40, 1, 0),                   # does not start at 0
    ([0, 9, 5, 40], 40, 2, 1),                # decreases between entries 1 and 2
    ([0, 5, 40], 41, 4, 2),                   # does not end at n_tok
    ([3, 2, 1], 7, 1 | 2 | 4, 0),             # everything wrong
])
def test_validate_cu_seqlens(cu, n_tok, bits, first):
    t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    assert kda.validate_cu_seqlens(t, n_tok) == (bits, first)


def test_validate_long_offsets_finds_the_first_decrease():
    cu = torch.arange(0, 100001, 10, dtype=torch.int32)
    cu[5000] = cu[4999] - 1
    cu[7000] = 0
    assert kda.validate_cu_seqlens(cu.to(DEV), int(cu[-1])) == (2, 4999)


def test_count_nonfinite_planted():
    x = torch.randn(100003, dtype=torch.float32)
    x[[0, 17, 99999, 100002]] = torch.tensor([float("nan"), float("inf"), float("-inf"), float("nan")])
    y = torch.randn(4097).to(torch.bfloat16)
    y[[4, 4096]] = torch.tensor([float("inf"), float("nan")]).to(torch.bfloat16)
    assert kda.count_nonfinite(x.to(DEV)) == 4
    assert kda.count_nonfinite(y.to(DEV)) == 2
    assert kda.count_nonfinite(x.to(DEV), y.to(DEV), None) == 6
    assert kda.count_nonfinite(torch.zeros(0, device=DEV)) == 0


def test_forward_at_the_bound_has_no_nonfinite_output():
    """The check the bounded gate exists to pass: every channel at g = -5 exactly."""
    x = K.make_inputs([1000, 300], 8, 128, 128, device=DEV, seed=21, h0_std=0.1)
    x.a.fill_(float("inf"))
    out, hf = kda.chunk_fwd(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_seqlens)
    assert kda.count_nonfinite(out, hf) == 0
    lib = kda.load_library()
    import ctypes
    scratch = torch.zeros(1, dtype=torch.int64, device=DEV)
    cnt = ctypes.c_uint64(7)
    st = lib.kda_check_outputs(ctypes.c_void_p(out.data_ptr()), out.numel(), kda.KDA_BF16,
                               ctypes.c_void_p(hf.data_ptr()), hf.numel(),
                               ctypes.c_void_p(scratch.data_ptr()), ctypes.byref(cnt),
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0 and cnt.value == 0
    out.view(-1)[123] = float("nan")
    st = lib.kda_check_outputs(ctypes.c_void_p(out.data_ptr()), out.numel(), kda.KDA_BF16,
                               ctypes.c_void_p(hf.data_ptr()), hf.numel(),
                               ctypes.c_void_p(scratch.data_ptr()), ctypes.byref(cnt),
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 4 and cnt.value == 1
