"""GB300 (sm_103a) chunked forward pass of gated delta-rule linear attention with the
lower-bounded decay g = -5*sigmoid(a) (Kimi Delta Attention style).

This package is a thin ctypes binding of the C ABI in ``include/kda.h``: it checks
tensor metadata, passes raw pointers and the current CUDA stream, and allocates
outputs with torch. Every step of the computation runs in the library's CUDA kernels;
there is no CPU path. If the compiled library is missing, every call raises.

    out, h_final = chunk_fwd(q, k, v, gate_logits, beta, h0=None, cu_seqlens=None)

Shapes (packed, token-major, contiguous): q, k, gate_logits [N, H, d_k]; v [N, H, d_v];
beta [N, H]; h0 / h_final [n_seq, H, d_k, d_v] fp32; cu_seqlens int32 [n_seq + 1]
(None = one sequence of N tokens). q/k/v/out are bf16 or fp32; gate_logits, beta and
the states are fp32.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build_mod

__all__ = ["validate_cu_seqlens", "count_nonfinite", "chunk_fwd", "chunk_fwd_simt", "chunk_fwd_from_host",
           "chunk_fwd_from_host_pipelined", "fwd_pipeline_plan", "fwd_pipelined_workspace_bytes",
           "affine_combine",
           "segmented_fwd", "decode_step", "chunk_bwd", "chunk_bwd_static_scratch",
           "bwd_timing_start", "bwd_timing_read", "chunk_fwd_variant", "gate_projection",
           "chunk_fwd_gated",
           "load_library",
           "kernel_launch_count", "read_device_flags", "selftest_bounded_wait",
           "library_path", "KDAError", "EXPORTED_SYMBOLS", "STATUS"]

STATUS = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED", 3: "KDA_ERR_CUDA",
          4: "KDA_ERR_NONFINITE"}
KDA_F32, KDA_BF16 = 0, 1
EXPORTED_SYMBOLS = ("kda_version", "kda_status_string", "kda_last_error",
                    "kda_kernel_launch_count", "kda_read_device_flags",
                    "kda_selftest_bounded_wait", "kda_chunk_fwd",
                    "kda_chunk_fwd_simt", "kda_chunk_fwd_from_host", "kda_affine_combine",
                    "kda_decode_step", "kda_chunk_bwd_workspace_bytes", "kda_chunk_bwd",
                    "kda_chunk_bwd_static_scratch", "kda_bwd_timing_start",
                    "kda_bwd_timing_read", "kda_chunk_fwd_variant", "kda_gate_projection",
                    "kda_chunk_fwd_from_host_pipelined", "kda_chunk_fwd_pipelined_workspace_bytes",
                    "kda_chunk_fwd_pipeline_plan", "kda_validate_cu_seqlens",
                    "kda_count_nonfinite", "kda_check_outputs",
                    "kda_chunk_fwd_gated_workspace_bytes", "kda_chunk_fwd_gated",
                    "kda_gate_projection_out")

_lock = threading.Lock()
_lib = None


class KDAError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__(f"{STATUS.get(status, status)}: {detail}")


def library_path() -> str:
    """The in-tree build, unless KDA_GB300_LIBRARY names another build of the same
    library (for A/B comparisons of kernel variants)."""
    return os.environ.get("KDA_GB300_LIBRARY") or _build_mod.LIB


def load_library(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load ``libkda_gb300.so``. Raises if it is absent (unless asked to build)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(
                    f"CUDA library {path} is not built; run "
                    "`python -c 'import __graft_entry__ as g; g.build()'` first")
            _build_mod.build()
        lib = ctypes.CDLL(path)
        P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        fwd_args = [P] * 9 + [I64, I32, I32, I32, I32, ctypes.c_int, P]
        for name in ("kda_chunk_fwd", "kda_chunk_fwd_simt"):
            fn = getattr(lib, name)
            fn.argtypes = fwd_args
            fn.restype = ctypes.c_int
        lib.kda_chunk_fwd_variant.argtypes = fwd_args[:-1] + [I32, I32, P]
        lib.kda_chunk_fwd_variant.restype = ctypes.c_int
        lib.kda_gate_projection.argtypes = [P, P, P, P, I64, I32, I32, P]
        lib.kda_gate_projection.restype = ctypes.c_int
        lib.kda_chunk_fwd_from_host.argtypes = [P] * 18 + [I64, I32, I32, I32, I32,
                                                          ctypes.c_int, P]
        lib.kda_chunk_fwd_from_host.restype = ctypes.c_int
        lib.kda_chunk_fwd_from_host_pipelined.argtypes = [P] * 19 + [
            ctypes.c_size_t, I64, I32, I32, I32, I32, I32, ctypes.c_int, P]
        lib.kda_chunk_fwd_from_host_pipelined.restype = ctypes.c_int
        lib.kda_chunk_fwd_pipelined_workspace_bytes.argtypes = [I32, I32, I32, I32, I32]
        lib.kda_chunk_fwd_pipelined_workspace_bytes.restype = ctypes.c_size_t
        lib.kda_chunk_fwd_pipeline_plan.argtypes = [P, I32, I64, I32, P, I32]
        lib.kda_chunk_fwd_pipeline_plan.restype = I32
        lib.kda_status_string.argtypes = [ctypes.c_int]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_last_error.argtypes = []
        lib.kda_last_error.restype = ctypes.c_char_p
        lib.kda_version.restype = ctypes.c_int
        lib.kda_kernel_launch_count.argtypes = []
        lib.kda_kernel_launch_count.restype = ctypes.c_uint64
        lib.kda_read_device_flags.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int, P]
        lib.kda_read_device_flags.restype = ctypes.c_int
        lib.kda_selftest_bounded_wait.argtypes = [I64, P, P]
        lib.kda_selftest_bounded_wait.restype = ctypes.c_int
        lib.kda_affine_combine.argtypes = [P, P, P, P, I32, I32, I32, P]
        lib.kda_affine_combine.restype = ctypes.c_int
        lib.kda_decode_step.argtypes = [P] * 7 + [I32, I32, I32, I32, ctypes.c_int, P]
        lib.kda_decode_step.restype = ctypes.c_int
        lib.kda_chunk_bwd_workspace_bytes.argtypes = [I64, I32, I32, I32, I32]
        lib.kda_chunk_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.kda_chunk_bwd.argtypes = [P] * 16 + [ctypes.c_size_t, I64, I32, I32, I32, I32,
                                                 ctypes.c_int, P]
        lib.kda_chunk_bwd.restype = ctypes.c_int
        lib.kda_chunk_bwd_static_scratch.argtypes = [P] * 15 + [I64, I32, I32, I32, I32,
                                                                ctypes.c_int, P]
        lib.kda_chunk_bwd_static_scratch.restype = ctypes.c_int
        lib.kda_bwd_timing_start.argtypes = [ctypes.c_int]
        lib.kda_bwd_timing_start.restype = ctypes.c_int
        lib.kda_bwd_timing_read.argtypes = [ctypes.POINTER(ctypes.c_float),
                                            ctypes.POINTER(ctypes.c_int)]
        lib.kda_bwd_timing_read.restype = ctypes.c_int
        lib.kda_validate_cu_seqlens.argtypes = [P, I32, I64, P, P]
        lib.kda_validate_cu_seqlens.restype = ctypes.c_int
        lib.kda_count_nonfinite.argtypes = [P, I64, ctypes.c_int, P, P]
        lib.kda_count_nonfinite.restype = ctypes.c_int
        lib.kda_check_outputs.argtypes = [P, I64, ctypes.c_int, P, I64, P,
                                          ctypes.POINTER(ctypes.c_uint64), P]
        lib.kda_check_outputs.restype = ctypes.c_int
        lib.kda_chunk_fwd_gated_workspace_bytes.argtypes = [I32, I32, I32, I32, I32]
        lib.kda_chunk_fwd_gated_workspace_bytes.restype = ctypes.c_size_t
        lib.kda_chunk_fwd_gated.argtypes = [P, P, P, I32] + [P] * 7 + [P, P, P, ctypes.c_size_t,
                                                                      I64, I32, I32, I32, I32, I32,
                                                                      ctypes.c_int, P]
        lib.kda_chunk_fwd_gated.restype = ctypes.c_int
        lib.kda_gate_projection_out.argtypes = [P, P, P, P, ctypes.c_int, I64, I32, I32, P]
        lib.kda_gate_projection_out.restype = ctypes.c_int
        _lib = lib
        return lib


def _check(lib, status: int):
    if status != 0:
        raise KDAError(status, lib.kda_last_error().decode() or
                       lib.kda_status_string(status).decode())


def _ptr(t):
    # an empty tensor has no meaningful address: pass NULL (the ABI needs none then)
    return None if t is None or t.numel() == 0 else ctypes.c_void_p(t.data_ptr())


def _dims(q, k, v, gate_logits, beta, h0, cu_seqlens, device_check=True):
    import torch
    if q.dim() != 3:
        raise ValueError("q must be [N, H, d_k] (packed, token-major)")
    N, H, dk = q.shape
    dv = v.shape[-1]
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("q/k/v must be bfloat16 or float32")
    for name, t, shape, dt in (("k", k, (N, H, dk), q.dtype), ("v", v, (N, H, dv), q.dtype),
                               ("gate_logits", gate_logits, (N, H, dk), torch.float32),
                               ("beta", beta, (N, H), torch.float32)):
        if tuple(t.shape) != shape or t.dtype != dt:
            raise ValueError(f"{name} must be {dt} with shape {shape}, got "
                             f"{t.dtype} {tuple(t.shape)}")
    n_seq = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise ValueError("cu_seqlens must be int32")
    if h0 is not None and (tuple(h0.shape) != (n_seq, H, dk, dv) or h0.dtype != torch.float32):
        raise ValueError(f"h0 must be float32 with shape {(n_seq, H, dk, dv)}")
    tensors = [q, k, v, gate_logits, beta, h0, cu_seqlens]
    for t in tensors:
        if t is not None and not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
        if device_check and t is not None and t.device != q.device:
            raise ValueError("all tensors must be on the same device")
    return N, H, dk, dv, n_seq


def _forward(symbol, q, k, v, gate_logits, beta, h0=None, cu_seqlens=None, *, out=None,
             h_final=None, output_final_state=True):
    import torch
    lib = load_library()
    if q.device.type != "cuda":
        raise ValueError("chunk_fwd runs on CUDA tensors only (there is no CPU path)")
    N, H, dk, dv, n_seq = _dims(q, k, v, gate_logits, beta, h0, cu_seqlens)
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, N], dtype=torch.int32, device=q.device)
    if out is None:
        out = torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    if h_final is None and output_final_state:
        h_final = torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device=q.device)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    st = getattr(lib, symbol)(_ptr(q), _ptr(k), _ptr(v), _ptr(gate_logits), _ptr(beta),
                              _ptr(h0), _ptr(cu_seqlens), _ptr(out), _ptr(h_final),
                              N, n_seq, H, dk, dv,
                              KDA_BF16 if q.dtype == torch.bfloat16 else KDA_F32,
                              ctypes.c_void_p(stream))
    _check(lib, st)
    return out, h_final


def chunk_fwd(q, k, v, gate_logits, beta, h0=None, cu_seqlens=None, *, out=None,
              h_final=None, output_final_state=True):
    """Chunked KDA forward through ``kda_chunk_fwd``. Returns ``(out, h_final)``;
    ``h_final`` is None when ``output_final_state`` is False."""
    return _forward("kda_chunk_fwd", q, k, v, gate_logits, beta, h0, cu_seqlens, out=out,
                    h_final=h_final, output_final_state=output_final_state)


def chunk_fwd_simt(q, k, v, gate_logits, beta, h0=None, cu_seqlens=None, *, out=None,
                   h_final=None, output_final_state=True):
    """Same operation on the fp32 SIMT kernel (``kda_chunk_fwd_simt``)."""
    return _forward("kda_chunk_fwd_simt", q, k, v, gate_logits, beta, h0, cu_seqlens,
                    out=out, h_final=h_final, output_final_state=output_final_state)


def gate_projection(x, weight, bias=None, *, out=None, out_dtype=None):
    """Gate logits ``a = x weight^T + bias`` through ``kda_gate_projection_out`` (tcgen05
    GEMM): ``x`` [N, d_model] bf16, ``weight`` [n_out, d_model] bf16, ``bias`` [n_out] fp32
    or None. Returns ``a`` [N, n_out] in ``out_dtype`` (fp32 by default -- view it as
    [N, H, d_k] for ``chunk_fwd`` -- or bf16: the fp32 result rounded to nearest even)."""
    import torch
    lib = load_library()
    if x.device.type != "cuda":
        raise ValueError("gate_projection runs on CUDA tensors only (there is no CPU path)")
    if x.dim() != 2 or weight.dim() != 2 or x.shape[1] != weight.shape[1]:
        raise ValueError("x must be [N, d_model] and weight [n_out, d_model]")
    if x.dtype != torch.bfloat16 or weight.dtype != torch.bfloat16:
        raise ValueError("x and weight must be bfloat16")
    N, D = x.shape
    n_out = weight.shape[0]
    if bias is not None and (bias.dtype != torch.float32 or tuple(bias.shape) != (n_out,)):
        raise ValueError(f"bias must be float32 with shape {(n_out,)}")
    for t in (x, weight, bias):
        if t is not None and (not t.is_contiguous() or t.device != x.device):
            raise ValueError("all tensors must be contiguous and on one device")
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else torch.float32
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("out_dtype must be float32 or bfloat16")
    if out is None:
        out = torch.empty((N, n_out), dtype=out_dtype, device=x.device)
    if out.dtype != out_dtype or tuple(out.shape) != (N, n_out) or not out.is_contiguous():
        raise ValueError(f"out must be contiguous {out_dtype} with shape {(N, n_out)}")
    stream = torch.cuda.current_stream(x.device).cuda_stream
    _check(lib, lib.kda_gate_projection_out(_ptr(x), _ptr(weight), _ptr(bias), _ptr(out),
                                            KDA_BF16 if out_dtype == torch.bfloat16 else KDA_F32,
                                            N, D, n_out, ctypes.c_void_p(stream)))
    return out


def chunk_fwd_gated(x, w_gate, b_gate, q, k, v, beta, h0=None, cu_seqlens=None, *,
                    segment_tokens=4096, out=None, h_final=None, output_final_state=True,
                    workspace=None):
    """The forward pass fed by the gate projection through ``kda_chunk_fwd_gated``: equal
    to ``chunk_fwd(q, k, v, gate_projection(x, w_gate, b_gate).view(N, H, d_k), ...)``, bit
    for bit, without the whole gate-logit tensor (per ``segment_tokens`` segment, the
    segment's logits go into one workspace slot and are consumed at once). ``x`` [N,
    d_model] bf16, ``w_gate`` [H * d_k, d_model] bf16, ``b_gate`` [H * d_k] fp32 or None;
    the rest as ``chunk_fwd`` (bf16). Returns ``(out, h_final)``."""
    import torch
    lib = load_library()
    if q.device.type != "cuda":
        raise ValueError("chunk_fwd_gated runs on CUDA tensors only (there is no CPU path)")
    if q.dim() != 3:
        raise ValueError("q must be [N, H, d_k] (packed, token-major)")
    # the gate logits the projection will produce have q's shape: check the rest against it
    gate_shape = torch.empty(q.shape, dtype=torch.float32, device="meta")
    N, H, dk, dv, n_seq = _dims(q, k, v, gate_shape, beta, h0, cu_seqlens, device_check=False)
    if x.dim() != 2 or x.shape[0] != N or x.dtype != torch.bfloat16:
        raise ValueError(f"x must be bfloat16 with shape ({N}, d_model)")
    D = x.shape[1]
    if tuple(w_gate.shape) != (H * dk, D) or w_gate.dtype != torch.bfloat16:
        raise ValueError(f"w_gate must be bfloat16 with shape {(H * dk, D)}")
    if b_gate is not None and (tuple(b_gate.shape) != (H * dk,) or b_gate.dtype != torch.float32):
        raise ValueError(f"b_gate must be float32 with shape {(H * dk,)}")
    for t in (x, w_gate, b_gate, q, k, v, beta, h0, cu_seqlens):
        if t is not None and (t.device != q.device or not t.is_contiguous()):
            raise ValueError("all tensors must be contiguous and on one device")
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, N], dtype=torch.int32, device=q.device)
    host_cu = cu_seqlens.to("cpu")
    if out is None:
        out = torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    if h_final is None and output_final_state:
        h_final = torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device=q.device)
    segment_tokens = max(64, min(int(segment_tokens), N))  # no larger slot than the call needs
    need = lib.kda_chunk_fwd_gated_workspace_bytes(n_seq, H, dk, dv, segment_tokens)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        stream = torch.cuda.current_stream(q.device).cuda_stream
        _check(lib, lib.kda_chunk_fwd_gated(
            _ptr(x), _ptr(w_gate), _ptr(b_gate), D, _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
            _ptr(h0), _ptr(cu_seqlens), ctypes.c_void_p(host_cu.data_ptr()), _ptr(out),
            _ptr(h_final), _ptr(workspace), workspace.numel(), N, n_seq, H, dk, dv,
            int(segment_tokens), KDA_BF16 if q.dtype == torch.bfloat16 else KDA_F32,
            ctypes.c_void_p(stream)))
    return out, (h_final if output_final_state else None)


GATES = {"bounded": 0, "softplus": 1}
DIAG_PATHS = {"dense": 0, "pairs": 1}


def chunk_fwd_variant(q, k, v, gate_logits, beta, h0=None, cu_seqlens=None, *,
                      gate="bounded", diag="dense", out=None, h_final=None):
    """Contrast variants through ``kda_chunk_fwd_variant`` (fp32 SIMT kernel): ``gate``
    "bounded" (-5 sigmoid(a), the method) or "softplus" (-softplus(a), unbounded);
    ``diag`` "dense" (the method's dense diagonal tile) or "pairs" (one exponential per
    position pair). softplus + dense overflows on strong decay, by design."""
    import torch
    lib = load_library()
    if q.device.type != "cuda":
        raise ValueError("chunk_fwd_variant runs on CUDA tensors only (there is no CPU path)")
    N, H, dk, dv, n_seq = _dims(q, k, v, gate_logits, beta, h0, cu_seqlens)
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, N], dtype=torch.int32, device=q.device)
    if out is None:
        out = torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    if h_final is None:
        h_final = torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device=q.device)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    _check(lib, lib.kda_chunk_fwd_variant(
        _ptr(q), _ptr(k), _ptr(v), _ptr(gate_logits), _ptr(beta), _ptr(h0), _ptr(cu_seqlens),
        _ptr(out), _ptr(h_final), N, n_seq, H, dk, dv,
        KDA_BF16 if q.dtype == torch.bfloat16 else KDA_F32, GATES[gate], DIAG_PATHS[diag],
        ctypes.c_void_p(stream)))
    return out, h_final


def chunk_fwd_from_host(q, k, v, gate_logits, beta, h0, cu_seqlens, out, h_final,
                        dev: dict, stream=None):
    """End-to-end call on host tensors through ``kda_chunk_fwd_from_host``.

    ``q ... cu_seqlens`` are CPU tensors (pinned for asynchronous copies); ``out`` and
    ``h_final`` are CPU tensors that receive the results (``h_final`` may be None).
    ``dev`` holds the caller's device buffers with keys q, k, v, gate_logits, beta, h0,
    cu_seqlens, out, h_final. The call only queues work on ``stream`` (default: the
    current stream); synchronise before reading ``out``.
    """
    import torch
    lib = load_library()
    N, H, dk, dv, n_seq = _dims(q, k, v, gate_logits, beta, h0, cu_seqlens,
                                device_check=False)
    if stream is None:
        stream = torch.cuda.current_stream(dev["q"].device)
    st = lib.kda_chunk_fwd_from_host(
        _ptr(q), _ptr(k), _ptr(v), _ptr(gate_logits), _ptr(beta), _ptr(h0),
        _ptr(cu_seqlens), _ptr(out), _ptr(h_final),
        _ptr(dev["q"]), _ptr(dev["k"]), _ptr(dev["v"]), _ptr(dev["gate_logits"]),
        _ptr(dev["beta"]), _ptr(dev.get("h0")), _ptr(dev["cu_seqlens"]),
        _ptr(dev["out"]), _ptr(dev.get("h_final")),
        N, n_seq, H, dk, dv, KDA_BF16 if q.dtype == torch.bfloat16 else KDA_F32,
        ctypes.c_void_p(stream.cuda_stream))
    _check(lib, st)
    return out, h_final


def fwd_pipelined_workspace_bytes(n_seq, n_heads, d_k, d_v, n_segments) -> int:
    """Bytes of device workspace ``chunk_fwd_from_host_pipelined`` needs."""
    return int(load_library().kda_chunk_fwd_pipelined_workspace_bytes(
        n_seq, n_heads, d_k, d_v, n_segments))


def fwd_pipeline_plan(cu_seqlens, n_segments):
    """The pieces ``chunk_fwd_from_host_pipelined`` runs for these sequence offsets (host
    only, ``kda_chunk_fwd_pipeline_plan``): a list of
    ``(t0, t1, n0, n1, h0_carried, hf_carried, segment)``."""
    lib = load_library()
    cu = (ctypes.c_int32 * len(cu_seqlens))(*[int(c) for c in cu_seqlens])
    n_seq, n_tok = len(cu_seqlens) - 1, int(cu_seqlens[-1]) if len(cu_seqlens) else 0
    count = lib.kda_chunk_fwd_pipeline_plan(ctypes.cast(cu, ctypes.c_void_p), n_seq, n_tok,
                                            n_segments, None, 0)
    if count < 0:
        raise KDAError(1, "invalid cu_seqlens or n_segments")
    buf = (ctypes.c_int64 * (7 * max(count, 1)))()
    got = lib.kda_chunk_fwd_pipeline_plan(ctypes.cast(cu, ctypes.c_void_p), n_seq, n_tok,
                                          n_segments, ctypes.cast(buf, ctypes.c_void_p), count)
    assert got == count
    return [tuple(int(buf[7 * j + i]) for i in range(7)) for j in range(count)]


PIPELINE_SEGMENT_BYTES = 32 << 20   # default: about this many input bytes per segment
PIPELINE_MAX_SEGMENTS = 16


def chunk_fwd_from_host_pipelined(q, k, v, gate_logits, beta, h0, cu_seqlens, out, h_final,
                                  dev: dict, stream=None, n_segments=None):
    """``chunk_fwd_from_host`` through ``kda_chunk_fwd_from_host_pipelined``: the copies in
    and out overlap the computation, segment by segment. ``dev`` as for
    ``chunk_fwd_from_host``, plus an optional ``workspace`` (a CUDA tensor of at least
    ``fwd_pipelined_workspace_bytes`` bytes; allocated here when absent). ``n_segments``
    defaults to one segment per ``PIPELINE_SEGMENT_BYTES`` of inputs, at most
    ``PIPELINE_MAX_SEGMENTS``: below that size the per-segment costs outweigh the overlap."""
    import torch
    lib = load_library()
    N, H, dk, dv, n_seq = _dims(q, k, v, gate_logits, beta, h0, cu_seqlens,
                                device_check=False)
    if n_segments is None:
        in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v, gate_logits, beta))
        n_segments = max(1, min(PIPELINE_MAX_SEGMENTS, in_bytes // PIPELINE_SEGMENT_BYTES))
    device = dev["q"].device
    if stream is None:
        stream = torch.cuda.current_stream(device)
    need = fwd_pipelined_workspace_bytes(n_seq, H, dk, dv, n_segments)
    if need == 0:
        raise KDAError(1, "invalid sizes or n_segments for the pipelined forward")
    ws = dev.get("workspace")
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=device)
        dev["workspace"] = ws
    st = lib.kda_chunk_fwd_from_host_pipelined(
        _ptr(q), _ptr(k), _ptr(v), _ptr(gate_logits), _ptr(beta), _ptr(h0),
        _ptr(cu_seqlens), _ptr(out), _ptr(h_final),
        _ptr(dev["q"]), _ptr(dev["k"]), _ptr(dev["v"]), _ptr(dev["gate_logits"]),
        _ptr(dev["beta"]), _ptr(dev.get("h0")), _ptr(dev["cu_seqlens"]),
        _ptr(dev["out"]), _ptr(dev.get("h_final")), _ptr(ws), ws.numel() * ws.element_size(),
        N, n_seq, H, dk, dv, n_segments, KDA_BF16 if q.dtype == torch.bfloat16 else KDA_F32,
        ctypes.c_void_p(stream.cuda_stream))
    _check(lib, st)
    return out, h_final


def kernel_launch_count() -> int:
    """Kernels the library has launched in this process (``kda_kernel_launch_count``)."""
    return int(load_library().kda_kernel_launch_count())


def validate_cu_seqlens(cu_seqlens, n_tok: int, stream=None):
    """Check the layout rules of ``cu_seqlens`` (int32, on the device) on the device:
    returns (bits, first offending index) -- bits 0 (first entry not 0), 1 (a decrease),
    2 (last entry not n_tok); (0, 2**31 - 1) when valid. Synchronises the stream."""
    import torch
    lib = load_library()
    if stream is None:
        stream = torch.cuda.current_stream()
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or cu_seqlens.dim() != 1:
        raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor")
    cu = cu_seqlens.contiguous()
    status = torch.empty(2, dtype=torch.int32, device=cu.device)
    _check(lib, lib.kda_validate_cu_seqlens(_ptr(cu), cu.numel() - 1, int(n_tok), _ptr(status),
                                            ctypes.c_void_p(stream.cuda_stream)))
    st = status.cpu().tolist()
    return int(st[0]), int(st[1])


def count_nonfinite(*tensors, stream=None) -> int:
    """Number of NaN / Inf elements over the given fp32 or bf16 CUDA tensors (None
    skipped), counted by the library's kernel. Synchronises the stream."""
    import torch
    lib = load_library()
    if stream is None:
        stream = torch.cuda.current_stream()
    ts = [t.contiguous() for t in tensors if t is not None]
    if not ts:
        return 0
    count = torch.zeros(1, dtype=torch.int64, device=ts[0].device)
    for t in ts:
        if t.dtype not in (torch.float32, torch.bfloat16):
            raise ValueError("count_nonfinite takes fp32 or bf16 tensors")
        _check(lib, lib.kda_count_nonfinite(_ptr(t), t.numel(),
                                            KDA_BF16 if t.dtype == torch.bfloat16 else KDA_F32,
                                            _ptr(count), ctypes.c_void_p(stream.cuda_stream)))
    return int(count.item())


def read_device_flags(reset: bool = True, stream=None) -> int:
    """Synchronise the stream and return the library's device status word (bit 0: a
    pipeline wait in the tensor-core kernel timed out). Clears it when ``reset``."""
    import torch
    lib = load_library()
    if stream is None:
        stream = torch.cuda.current_stream()
    v = ctypes.c_uint32(0)
    _check(lib, lib.kda_read_device_flags(ctypes.byref(v), int(reset),
                                          ctypes.c_void_p(stream.cuda_stream)))
    return int(v.value)


def selftest_bounded_wait(limit_cycles: int = 2_000_000):
    """Run the bounded-wait self-test; returns ``(returned_code, flags)`` where 1 and a
    set bit 0 mean the never-completing wait gave up as designed. Clears the flags."""
    import torch
    lib = load_library()
    read_device_flags(reset=True)
    d = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream()
    _check(lib, lib.kda_selftest_bounded_wait(int(limit_cycles), ctypes.c_void_p(d.data_ptr()),
                                              ctypes.c_void_p(st.cuda_stream)))
    flags = read_device_flags(reset=True)
    return int(d.item()), flags


def affine_combine(M, S, B, out=None):
    """``out = M S + B`` per head through ``kda_affine_combine`` (fp32 CUDA tensors;
    ``M`` [H, d_k, d_k], ``S`` and ``B`` [H, d_k, d_v]): the combine step of the segment
    scan -- a segment of tokens maps its start state S to M S + B."""
    import torch
    lib = load_library()
    if M.device.type != "cuda":
        raise ValueError("affine_combine runs on CUDA tensors only (there is no CPU path)")
    H, dk, dk2 = M.shape
    dv = S.shape[-1]
    if dk2 != dk or tuple(S.shape) != (H, dk, dv) or tuple(B.shape) != (H, dk, dv):
        raise ValueError("M must be [H, d_k, d_k], S and B [H, d_k, d_v]")
    for t in (M, S, B):
        if t.dtype != torch.float32 or not t.is_contiguous() or t.device != M.device:
            raise ValueError("M, S and B must be contiguous float32 on one device")
    if out is None:
        out = torch.empty_like(B)
    stream = torch.cuda.current_stream(M.device).cuda_stream
    _check(lib, lib.kda_affine_combine(_ptr(M), _ptr(S), _ptr(B), _ptr(out), H, dk, dv,
                                       ctypes.c_void_p(stream)))
    return out


def decode_step(q, k, v, gate_logits, beta, state, *, out=None):
    """One recurrent decode step through ``kda_decode_step``: every sequence advances by
    one token. ``q, k, gate_logits`` [B, H, d_k]; ``v`` [B, H, d_v]; ``beta`` [B, H];
    ``state`` [B, H, d_k, d_v] fp32, updated in place. Returns ``out`` [B, H, d_v]."""
    import torch
    lib = load_library()
    if q.device.type != "cuda":
        raise ValueError("decode_step runs on CUDA tensors only (there is no CPU path)")
    if q.dim() != 3:
        raise ValueError("q must be [B, H, d_k]")
    B, H, dk = q.shape
    dv = v.shape[-1]
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("q/k/v must be bfloat16 or float32")
    for name, t, shape, dt in (("k", k, (B, H, dk), q.dtype), ("v", v, (B, H, dv), q.dtype),
                               ("gate_logits", gate_logits, (B, H, dk), torch.float32),
                               ("beta", beta, (B, H), torch.float32),
                               ("state", state, (B, H, dk, dv), torch.float32)):
        if tuple(t.shape) != shape or t.dtype != dt:
            raise ValueError(f"{name} must be {dt} with shape {shape}, got "
                             f"{t.dtype} {tuple(t.shape)}")
    for t in (q, k, v, gate_logits, beta, state):
        if not t.is_contiguous() or t.device != q.device:
            raise ValueError("all tensors must be contiguous and on one device")
    if out is None:
        out = torch.empty((B, H, dv), dtype=q.dtype, device=q.device)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    _check(lib, lib.kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(gate_logits), _ptr(beta),
                                    _ptr(state), _ptr(out), B, H, dk, dv,
                                    KDA_BF16 if q.dtype == torch.bfloat16 else KDA_F32,
                                    ctypes.c_void_p(stream)))
    return out


def chunk_bwd(q, k, v, gate_logits, beta, h0, cu_seqlens, dout, dh_final=None, *,
              want_dh0=True, workspace=None):
    """Backward pass through ``kda_chunk_bwd``: the gradients of ``<dout, out> +
    <dh_final, h_final>`` for the forward ``chunk_fwd(q, k, v, gate_logits, beta, h0,
    cu_seqlens)``. Returns ``(dq, dk, dv, dgate_logits, dbeta, dh0)`` (``dh0`` None unless
    ``want_dh0``). ``workspace``: an optional uint8 CUDA tensor of at least
    ``kda_chunk_bwd_workspace_bytes`` bytes (allocated here when None)."""
    import torch
    lib = load_library()
    if q.device.type != "cuda":
        raise ValueError("chunk_bwd runs on CUDA tensors only (there is no CPU path)")
    N, H, dk, dv, n_seq = _dims(q, k, v, gate_logits, beta, h0, cu_seqlens)
    if tuple(dout.shape) != (N, H, dv) or dout.dtype != q.dtype or not dout.is_contiguous():
        raise ValueError(f"dout must be contiguous {q.dtype} with shape {(N, H, dv)}")
    if dh_final is not None and (tuple(dh_final.shape) != (n_seq, H, dk, dv) or
                                 dh_final.dtype != torch.float32 or
                                 not dh_final.is_contiguous()):
        raise ValueError(f"dh_final must be contiguous float32 {(n_seq, H, dk, dv)}")
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, N], dtype=torch.int32, device=q.device)
    need = int(lib.kda_chunk_bwd_workspace_bytes(N, n_seq, H, dk, dv))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    elif workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace needs {need} bytes")
    dq = torch.empty_like(q)
    dk_ = torch.empty_like(k)
    dv_ = torch.empty_like(v)
    da = torch.empty_like(gate_logits)
    db = torch.empty_like(beta)
    dh0 = torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device=q.device) if want_dh0 \
        else None
    stream = torch.cuda.current_stream(q.device).cuda_stream
    _check(lib, lib.kda_chunk_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(gate_logits), _ptr(beta), _ptr(h0), _ptr(cu_seqlens),
        _ptr(dout), _ptr(dh_final), _ptr(dq), _ptr(dk_), _ptr(dv_), _ptr(da), _ptr(db),
        _ptr(dh0), _ptr(workspace), workspace.numel() * workspace.element_size(),
        N, n_seq, H, dk, dv, KDA_BF16 if q.dtype == torch.bfloat16 else KDA_F32,
        ctypes.c_void_p(stream)))
    return dq, dk_, dv_, da, db, dh0


def bwd_timing_start(capacity: int) -> None:
    """Record the device time of each backward kernel for the next ``capacity`` calls."""
    lib = load_library()
    _check(lib, lib.kda_bwd_timing_start(int(capacity)))


def bwd_timing_read():
    """``([prep, forward pass, reverse pass, local] ms summed over the recorded calls),
    calls)``; stops recording."""
    ms = (ctypes.c_float * 4)()
    calls = ctypes.c_int(0)
    lib = load_library()
    _check(lib, lib.kda_bwd_timing_read(ms, ctypes.byref(calls)))
    return [float(x) for x in ms], int(calls.value)


def chunk_bwd_static_scratch(q, k, v, gate_logits, beta, h0, cu_seqlens, dout, dh_final=None,
                             *, want_dh0=True):
    """``chunk_bwd`` through ``kda_chunk_bwd_static_scratch``: no workspace is passed or
    allocated for the checkpoints (the library's fixed 64 MiB scratch holds them; calls
    must not overlap in time). Returns ``(dq, dk, dv, dgate_logits, dbeta, dh0)``."""
    import torch
    lib = load_library()
    if q.device.type != "cuda":
        raise ValueError("chunk_bwd_static_scratch runs on CUDA tensors only")
    N, H, dk, dv, n_seq = _dims(q, k, v, gate_logits, beta, h0, cu_seqlens)
    if tuple(dout.shape) != (N, H, dv) or dout.dtype != q.dtype or not dout.is_contiguous():
        raise ValueError(f"dout must be contiguous {q.dtype} with shape {(N, H, dv)}")
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, N], dtype=torch.int32, device=q.device)
    grads = [torch.empty_like(t) for t in (q, k, v, gate_logits, beta)]
    dh0 = torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device=q.device) if want_dh0 \
        else None
    # the library resolves the scratch array of the CURRENT device: make it q's
    with torch.cuda.device(q.device):
        stream = torch.cuda.current_stream(q.device).cuda_stream
        _check(lib, lib.kda_chunk_bwd_static_scratch(
            _ptr(q), _ptr(k), _ptr(v), _ptr(gate_logits), _ptr(beta), _ptr(h0),
            _ptr(cu_seqlens), _ptr(dout), _ptr(dh_final), *[_ptr(g) for g in grads], _ptr(dh0),
            N, n_seq, H, dk, dv, KDA_BF16 if q.dtype == torch.bfloat16 else KDA_F32,
            ctypes.c_void_p(stream)))
    return (*grads, dh0)


def segmented_fwd(q, k, v, gate_logits, beta, h0=None, cu_seqlens=None, *, segments: int,
                  output_final_state=True):
    """The forward pass of ONE sequence split into ``segments`` time segments that run
    side by side: for inputs whose heads alone leave most of the GPU idle.

    Scheduling only; every step runs in the library's kernels (three ``kda_chunk_fwd``
    calls and ``segments - 2`` ``kda_affine_combine`` calls):
      1. all segments from a zero start (the first from h0): the first segment's outputs
         and end state are final, every other segment gives its affine offset B_j;
      2. segments 1.. from h0 = I with v = 0 (and d_v = d_k): their transitions M_j;
      3. S_{j+1} = M_j S_j + B_j chains the true start states;
      4. segments 1.. replay from their start states, writing the final outputs.
    Costs about 3x the state-chain work of segments 1.. in exchange for a serial chain
    ``segments`` times shorter. Returns ``(out, h_final)`` like ``chunk_fwd``.
    """
    import torch
    from . import sharding
    N, H, dk, dv, n_seq = _dims(q, k, v, gate_logits, beta, h0, cu_seqlens)
    if n_seq != 1:
        raise ValueError("segmented_fwd takes a single sequence")
    if segments < 1:
        raise ValueError("segments must be >= 1")
    bounds = [(a, b) for a, b in sharding.segment_bounds(N, segments) if b > a]
    if len(bounds) <= 1:
        return chunk_fwd(q, k, v, gate_logits, beta, h0, cu_seqlens,
                         output_final_state=output_final_state)
    dev = q.device
    P = len(bounds)
    cu = torch.tensor([a for a, _ in bounds] + [N], dtype=torch.int32, device=dev)
    # 1. zero start everywhere except the first segment
    start = torch.zeros((P, H, dk, dv), dtype=torch.float32, device=dev)
    if h0 is not None:
        start[0].copy_(h0[0])
    out, ends = chunk_fwd(q, k, v, gate_logits, beta, start, cu)
    # 2. transitions of segments 1..P-1 (a contiguous token range)
    b1 = bounds[1][0]
    cu_t = (cu[1:] - b1).contiguous()
    eye = torch.eye(dk, dtype=torch.float32, device=dev).expand(P - 1, H, dk, dk).contiguous()
    v0 = torch.zeros((N - b1, H, dk), dtype=v.dtype, device=dev)
    _, trans = chunk_fwd(q[b1:], k[b1:], v0, gate_logits[b1:], beta[b1:], eye, cu_t)
    del v0
    # 3. true start states of segments 1..P-1
    starts = torch.empty((P - 1, H, dk, dv), dtype=torch.float32, device=dev)
    starts[0].copy_(ends[0])
    for j in range(1, P - 1):
        affine_combine(trans[j - 1], starts[j - 1], ends[j], out=starts[j])
    # 4. replay segments 1..P-1 into their slice of out
    _, h_last = chunk_fwd(q[b1:], k[b1:], v[b1:], gate_logits[b1:], beta[b1:], starts, cu_t,
                          out=out[b1:])
    h_final = h_last[P - 2:P - 1].clone() if output_final_state else None
    return out, h_final
