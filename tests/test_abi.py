"""The C ABI without a GPU: the library builds, loads, exports every symbol that
``include/kda.h`` declares, and rejects bad arguments on the host before any CUDA call.

Only calls that fail host validation (or have nothing to do) are made here, so no
pointer is ever dereferenced and no kernel is launched.
"""
import ctypes
import os
import re

import pytest

import chunked_linear_attention_kda_gb300 as kda
from chunked_linear_attention_kda_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kda.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert declared_functions() == sorted(kda.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_has_no_torch_or_python_dependency():
    out = os.popen(f"ldd {kbuild.LIB}").read()
    assert "torch" not in out and "python" not in out


def test_version_and_status_strings(lib):
    assert lib.kda_version() >= 100
    for s in range(5):
        assert lib.kda_status_string(s).decode().startswith(kda.STATUS[s])
    assert lib.kda_status_string(99) == b"unknown kda_status"


FAKE = 0x100000  # 16-byte aligned, never dereferenced by these calls


def call(lib, *, q=FAKE, k=FAKE, v=FAKE, a=FAKE, beta=FAKE, h0=None, cu=FAKE, out=FAKE,
         hf=None, n_tok=64, n_seq=1, H=2, dk=128, dv=128, dtype=1, symbol="kda_chunk_fwd"):
    P = ctypes.c_void_p
    return getattr(lib, symbol)(P(q), P(k), P(v), P(a), P(beta), P(h0), P(cu), P(out),
                                P(hf), n_tok, n_seq, H, dk, dv, dtype, None)


@pytest.mark.parametrize("symbol", ["kda_chunk_fwd", "kda_chunk_fwd_simt"])
@pytest.mark.parametrize("kw,status", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(a=None), 1),
    (dict(beta=None), 1), (dict(out=None), 1), (dict(cu=None), 1),
    (dict(n_tok=-1), 1), (dict(n_seq=-1), 1), (dict(H=0), 1), (dict(dk=0), 1),
    (dict(dv=-3), 1), (dict(n_seq=0), 1),          # tokens but no sequence
    (dict(dk=129), 2), (dict(dv=256), 2), (dict(dtype=7), 2),
    (dict(q=FAKE + 2), 1), (dict(out=FAKE + 8), 1), (dict(a=FAKE + 4), 1),
    (dict(hf=FAKE + 2), 1), (dict(beta=FAKE + 1), 1), (dict(cu=FAKE + 2), 1),
])
def test_host_validation(lib, symbol, kw, status):
    st = call(lib, symbol=symbol, **kw)
    assert st == status, (kw, st, lib.kda_last_error())
    assert lib.kda_last_error().decode() != ""


def test_nothing_to_do_is_ok(lib):
    assert call(lib, n_tok=0, n_seq=0) == 0
    assert lib.kda_last_error() == b""


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(16, 1, 16)
    with pytest.raises(ValueError):
        kda.chunk_fwd(x, x, x, x, torch.zeros(16, 1))


def combine(lib, *, M=FAKE, S=FAKE + 256, B=FAKE + 512, O=FAKE + 768, H=2, dk=128, dv=128):
    P = ctypes.c_void_p
    return lib.kda_affine_combine(P(M), P(S), P(B), P(O), H, dk, dv, None)


@pytest.mark.parametrize("kw,status", [
    (dict(M=None), 1), (dict(S=None), 1), (dict(B=None), 1), (dict(O=None), 1),
    (dict(H=0), 1), (dict(dk=0), 1), (dict(dv=-1), 1), (dict(dk=129), 2), (dict(dv=200), 2),
    (dict(M=FAKE + 2), 1), (dict(O=FAKE), 1), (dict(O=FAKE + 512), 1),
])
def test_affine_combine_host_validation(lib, kw, status):
    st = combine(lib, **kw)
    assert st == status, (kw, st, lib.kda_last_error())
    assert lib.kda_last_error().decode() != ""


def test_binding_refuses_cpu_combine():
    import torch
    m = torch.zeros(1, 4, 4)
    with pytest.raises(ValueError):
        kda.affine_combine(m, m, m)


def decode(lib, *, q=FAKE, k=2 * FAKE, v=3 * FAKE, a=4 * FAKE, beta=5 * FAKE, state=6 * FAKE,
           out=8 * FAKE, n_seq=2, H=2, dk=128, dv=128, dtype=1):
    P = ctypes.c_void_p
    return lib.kda_decode_step(P(q), P(k), P(v), P(a), P(beta), P(state), P(out), n_seq, H, dk,
                               dv, dtype, None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(a=None), 1),
    (dict(beta=None), 1), (dict(state=None), 1), (dict(out=None), 1),
    (dict(n_seq=-1), 1), (dict(H=0), 1), (dict(dk=0), 1), (dict(dv=-2), 1),
    (dict(dk=129), 2), (dict(dv=256), 2), (dict(dtype=5), 2),
    (dict(q=FAKE + 1), 1), (dict(dtype=0, v=3 * FAKE + 2), 1), (dict(a=4 * FAKE + 2), 1),
    (dict(state=6 * FAKE + 1), 1),
    (dict(state=FAKE + 256), 1),          # state overlaps q
    (dict(out=6 * FAKE + 4096), 1),       # out inside the state
    (dict(out=5 * FAKE), 1),              # out on beta
])
def test_decode_step_host_validation(lib, kw, status):
    st = decode(lib, **kw)
    assert st == status, (kw, st, lib.kda_last_error())
    assert lib.kda_last_error().decode() != ""


def test_decode_step_nothing_to_do_is_ok(lib):
    assert decode(lib, n_seq=0) == 0


def test_binding_refuses_cpu_decode():
    import torch
    x = torch.zeros(1, 1, 16)
    with pytest.raises(ValueError):
        kda.decode_step(x, x, x, x, torch.zeros(1, 1), torch.zeros(1, 1, 16, 16))


def bwd(lib, *, q=FAKE, k=2 * FAKE, v=3 * FAKE, a=4 * FAKE, beta=5 * FAKE, h0=None, cu=6 * FAKE,
        dout=7 * FAKE, dhf=None, dq=8 * FAKE, dk_=9 * FAKE, dv_=10 * FAKE, da=11 * FAKE,
        db=12 * FAKE, dh0=None, ws=16 * FAKE, ws_bytes=None, n_tok=64, n_seq=1, H=2, dk=128,
        dv=128, dtype=1):
    P = ctypes.c_void_p
    if ws_bytes is None:
        ws_bytes = lib.kda_chunk_bwd_workspace_bytes(n_tok, n_seq, H, dk, dv) if n_tok >= 0 else 0
    return lib.kda_chunk_bwd(P(q), P(k), P(v), P(a), P(beta), P(h0), P(cu), P(dout), P(dhf),
                             P(dq), P(dk_), P(dv_), P(da), P(db), P(dh0), P(ws), ws_bytes,
                             n_tok, n_seq, H, dk, dv, dtype, None)


def test_backward_workspace_size(lib):
    # per (chunk slot, head): two fp32 states and the chunk's products (K', W, Q~ 16 x d_k,
    # U~ 16 x d_v, P 16 x 16, gamma_L d_k); slots = (n_tok >> 4) + n_seq + 1
    per = 2 * 128 * 128 + 3 * 16 * 128 + 16 * 128 + 16 * 16 + 128
    assert lib.kda_chunk_bwd_workspace_bytes(64, 1, 2, 128, 128) == 6 * 2 * per * 4
    assert lib.kda_chunk_bwd_workspace_bytes(-1, 1, 2, 128, 128) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), 1), (dict(dout=None), 1), (dict(dq=None), 1), (dict(dk_=None), 1),
    (dict(dv_=None), 1), (dict(da=None), 1), (dict(db=None), 1), (dict(ws=None), 1),
    (dict(ws_bytes=1024), 1), (dict(cu=None), 1), (dict(H=0), 1), (dict(dk=129), 2),
    (dict(dtype=9), 2), (dict(dq=8 * FAKE + 1), 1), (dict(da=11 * FAKE + 2), 1),
    (dict(ws=16 * FAKE + 2), 1),
    (dict(dq=FAKE), 1),                  # dq on q
    (dict(ws=10 * FAKE + 64), 1),        # workspace inside dv
    (dict(db=11 * FAKE), 1),             # dbeta on dgate_logits
])
def test_backward_host_validation(lib, kw, status):
    st = bwd(lib, **kw)
    assert st == status, (kw, st, lib.kda_last_error())
    assert lib.kda_last_error().decode() != ""


def test_backward_nothing_to_do_is_ok(lib):
    assert bwd(lib, n_tok=0, n_seq=0) == 0


@pytest.mark.parametrize("gate,diag,status", [(2, 0, 1), (-1, 0, 1), (0, 2, 1), (1, 7, 1)])
def test_variant_rejects_unknown_gate_or_path(lib, gate, diag, status):
    P = ctypes.c_void_p
    st = lib.kda_chunk_fwd_variant(P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), None, P(FAKE),
                                   P(FAKE), None, 64, 1, 2, 128, 128, 1, gate, diag, None)
    assert st == status and lib.kda_last_error().decode() != ""


def proj(lib, *, x=FAKE, w=2 * FAKE, b=None, a=4 * FAKE, n_tok=64, d=128, n_out=256):
    P = ctypes.c_void_p
    return lib.kda_gate_projection(P(x), P(w), P(b), P(a), n_tok, d, n_out, None)


@pytest.mark.parametrize("kw,status", [
    (dict(x=None), 1), (dict(w=None), 1), (dict(a=None), 1), (dict(n_tok=-1), 1),
    (dict(d=0), 1), (dict(n_out=0), 1), (dict(d=100), 2), (dict(x=FAKE + 8), 1),
    (dict(a=4 * FAKE + 4), 1), (dict(b=3 * FAKE + 2), 1), (dict(a=FAKE + 64), 1),
    (dict(a=2 * FAKE), 1),
])
def test_gate_projection_host_validation(lib, kw, status):
    st = proj(lib, **kw)
    assert st == status, (kw, st, lib.kda_last_error())
    assert lib.kda_last_error().decode() != ""


def test_gate_projection_nothing_to_do_is_ok(lib):
    assert proj(lib, n_tok=0) == 0


def proj_out(lib, *, x=FAKE, w=2 * FAKE, b=None, a=4 * FAKE, dt=1, n_tok=64, d=128, n_out=256):
    P = ctypes.c_void_p
    return lib.kda_gate_projection_out(P(x), P(w), P(b), P(a), dt, n_tok, d, n_out, None)


@pytest.mark.parametrize("kw,status", [
    (dict(dt=2), 2), (dict(dt=-1), 2), (dict(a=None), 1), (dict(a=4 * FAKE + 8), 1),
    (dict(d=100), 2), (dict(x=FAKE + 8), 1), (dict(b=3 * FAKE + 2), 1),
    # bf16 output of 64 x 256: 32 KiB from 4 FAKE, overlapping x (64 x 128 bf16 at FAKE)
    (dict(a=FAKE + 64), 1),
])
def test_gate_projection_out_host_validation(lib, kw, status):
    st = proj_out(lib, **kw)
    assert st == status, (kw, st, lib.kda_last_error())
    assert lib.kda_last_error().decode() != ""


@pytest.mark.parametrize("capacity", [0, -3, 1025])
def test_backward_timing_rejects_capacity(lib, capacity):
    assert lib.kda_bwd_timing_start(capacity) == 1


def test_backward_timing_read_rejects_null(lib):
    ms = (ctypes.c_float * 4)()
    calls = ctypes.c_int(0)
    assert lib.kda_bwd_timing_read(None, ctypes.byref(calls)) == 1
    assert lib.kda_bwd_timing_read(ms, None) == 1


# ---------------------------------------------------------------- device-side checks

@pytest.mark.parametrize("kw,status", [
    (dict(cu=None), 1), (dict(st=None), 1), (dict(n_seq=-1), 1), (dict(n_tok=-5), 1),
    (dict(cu=FAKE + 2), 1), (dict(st=FAKE + 1), 1),
])
def test_validate_cu_seqlens_host_validation(lib, kw, status):
    a = dict(cu=FAKE, n_seq=3, n_tok=100, st=FAKE)
    a.update(kw)
    P = ctypes.c_void_p
    st = lib.kda_validate_cu_seqlens(P(a["cu"]), a["n_seq"], a["n_tok"], P(a["st"]), None)
    assert st == status and lib.kda_last_error().decode() != ""


@pytest.mark.parametrize("kw,status", [
    (dict(x=None), 1), (dict(cnt=None), 1), (dict(n=-1), 1), (dict(dtype=5), 2),
    (dict(x=FAKE + 2, dtype=0), 1), (dict(x=FAKE + 1, dtype=1), 1), (dict(cnt=FAKE + 4), 1),
])
def test_count_nonfinite_host_validation(lib, kw, status):
    a = dict(x=FAKE, n=10, dtype=1, cnt=FAKE)
    a.update(kw)
    P = ctypes.c_void_p
    st = lib.kda_count_nonfinite(P(a["x"]), a["n"], a["dtype"], P(a["cnt"]), None)
    assert st == status and lib.kda_last_error().decode() != ""


def test_check_outputs_host_validation(lib):
    P = ctypes.c_void_p
    cnt = ctypes.c_uint64(0)
    assert lib.kda_check_outputs(P(FAKE), 10, 1, None, 0, None, ctypes.byref(cnt), None) == 1
    assert lib.kda_check_outputs(P(FAKE), 10, 1, None, 0, P(FAKE), None, None) == 1
    assert lib.kda_check_outputs(None, 10, 1, None, 0, P(FAKE), ctypes.byref(cnt), None) == 1
    assert lib.kda_check_outputs(P(FAKE), -1, 1, None, 0, P(FAKE), ctypes.byref(cnt), None) == 1


def gated(lib, *, x=FAKE, w=2 * FAKE, b=None, D=256, q=3 * FAKE, k=4 * FAKE, v=5 * FAKE,
          beta=6 * FAKE, h0=None, cu=7 * FAKE, host_cu="default", out=8 * FAKE, hf=None,
          ws=9 * FAKE, ws_bytes=None, n_tok=64, n_seq=1, H=2, dk=128, dv=128, seg=64, dtype=1):
    P = ctypes.c_void_p
    hc = (ctypes.c_int32 * 2)(0, n_tok) if host_cu == "default" else host_cu
    if ws_bytes is None:
        ws_bytes = lib.kda_chunk_fwd_gated_workspace_bytes(n_seq, H, dk, dv, max(seg, 64))
    return lib.kda_chunk_fwd_gated(P(x), P(w), P(b), D, P(q), P(k), P(v), P(beta), P(h0), P(cu),
                                   hc, P(out), P(hf), P(ws), ws_bytes, n_tok, n_seq, H, dk, dv,
                                   seg, dtype, None)


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=0), 2),                       # bf16 only
    (dict(seg=63), 1),                        # segments of at least one 64-token step
    (dict(D=12), 2),                          # d_model a multiple of 8
    (dict(x=None), 1), (dict(w=None), 1), (dict(x=FAKE + 8), 1), (dict(b=FAKE + 2), 1),
    (dict(q=None), 1), (dict(dk=129), 2),     # the forward's own rules
    (dict(host_cu=None), 1),
    (dict(host_cu=(ctypes.c_int32 * 2)(0, 63)), 1),   # does not end at n_tok
    (dict(ws=None), 1), (dict(ws_bytes=256), 1), (dict(ws=9 * FAKE + 16), 1),
])
def test_gated_forward_host_validation(lib, kw, status):
    st = gated(lib, **kw)
    assert st == status, (kw, st, lib.kda_last_error())
    assert lib.kda_last_error().decode() != ""


def test_gated_workspace_size(lib):
    # two carried states of H x 128 x 128 fp32, the offsets table, one slot of
    # (segment + 64) tokens x H x d_k fp32 gate logits, each 256-byte aligned
    H, seg, n_seq = 32, 4096, 1
    carry = H * 128 * 128 * 4
    table = ((n_seq + 5 * 64 + 1) * 4 + 255) // 256 * 256
    slot = (seg + 64) * H * 128 * 4
    assert lib.kda_chunk_fwd_gated_workspace_bytes(n_seq, H, 128, 128, seg) == 2 * carry + table + slot
    assert lib.kda_chunk_fwd_gated_workspace_bytes(n_seq, H, 128, 128, 32) == 0
    assert lib.kda_chunk_fwd_gated_workspace_bytes(-1, H, 128, 128, seg) == 0
