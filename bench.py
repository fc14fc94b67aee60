#!/usr/bin/env python3
"""Throughput of the chunked KDA forward pass on GB300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 3] [--impl ours|reference]

A step is one ``kda_chunk_fwd`` call over the whole workload (every row of the hot
path: gate prologue, diagonal tile, serial state recurrence, varlen front end), with
inputs resident in HBM. The default workload is the 64K-token context (B=1, H=32,
T=65536, d_k = d_v = 128, bf16 q/k/v/o, fp32 gates/beta/state); its 3.2 GB of inputs
are 25x the 129 MB L2, so no flush is needed between steps. Under torchrun with N > 1
every rank runs the same per-GPU workload on its own device with its own seed (weak
scaling, independent sequences: no collective on the data path; one max-reduction of
the elapsed time for the report).

Reported alongside the device-timed value:
  e2e          the same metric through ``kda_chunk_fwd_from_host_pipelined`` with pinned
               host buffers: H2D copies of the inputs, the kernels and D2H copies of the
               outputs inside the timed region, overlapped segment by segment; the
               median of event-timed calls (the mean beside it), the one-stream
               ``kda_chunk_fwd_from_host`` time and the inputs' copy alone reported too;
  roofline     algorithmic bytes per launch / CUDA-event launch time against the
               measured HBM copy bandwidth (MEASURED_PEAKS.json);
  cpu_baseline the fp64 oracle on the host cores on a bounded sample (rank 0, N = 1);
  parity       the timed run's outputs against the oracle on that sample, over the whole
               sample and for the worst (sequence, head) pair (final states too when
               the sample covers the whole sequence);
  diagnostics  non-finite outputs and states (the library's device counter) and the
               Frobenius norms of the final states;
  clocks       nvidia-smi samples taken during the timed region;
  workloads    with the default workload, the same timing, roofline, diagnostics and
               a prefix parity sample for the 256K-token context (B=1, H=32) and the
               packed variable-length workload (16 sequences of 4K-131K tokens plus one
               of 1M, H=16); the headline keys stay those of the 64K workload.
``--impl reference`` times the oracle alone (the reference arm of this build).

``--op decode`` measures the recurrent decode step instead (``kda_decode_step``: B = 256
sequences x H = 32 heads, d = 128, bf16, each step advances every sequence by one
token; the 512 MiB fp32 state, 4x the L2, is read and rewritten in place), with the
same timing rules and its own JSON line. ``--op backward`` measures the backward pass
(``kda_chunk_bwd``: every gradient of the forward) on the same workload as the forward.
``--op contrast`` times the contrast variants (``kda_chunk_fwd_variant``) on that workload:
the fp32 SIMT forward with the dense diagonal tile against the position-pair tile, with
the bounded and the unbounded softplus gate, beside the tensor-core kernel.
``--op projection`` measures the gate projection (``kda_gate_projection``, a tcgen05 GEMM:
a = x W^T + b for the 64K workload's tokens, d_model = 4096, 32 heads x 128 outputs).
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA chunked-forward tokens/s (1 GB300) and % of tensor-core/HBM roofline"
DECODE_METRIC = "KDA recurrent decode tokens/s (1 GB300) and % of HBM roofline"
DECODE_B, DECODE_H, DECODE_D = 256, 32, 128
UNIT = "tokens/s"
# the bench workload's kernel (bf16, d = 128 takes the 64-token tensor-core kernel)
KERNEL_SOURCES = ["chunked_linear_attention_kda_gb300/csrc/kda_fwd64.cu",
                  "chunked_linear_attention_kda_gb300/csrc/kda_ptx.h"]
# workloads timed after the headline one and reported under "workloads"
EXTRA_WORKLOADS = {5: 16384, 4: 4096}   # workload index -> oracle prefix tokens
DECODE_SOURCES = ["chunked_linear_attention_kda_gb300/csrc/kda_decode.cu"]
BACKWARD_SOURCES = ["chunked_linear_attention_kda_gb300/csrc/kda_bwd.cu"]
BACKWARD_METRIC = "KDA chunked-backward tokens/s (1 GB300) and % of HBM roofline (dominant kernel)"
BACKWARD_KERNELS = ["prep", "forward_pass", "reverse_pass", "local_gradients"]
# the tensor-core path runs both serial passes in one launch
BACKWARD_KERNELS_TC = ["prep", "serial_passes", "local_gradients"]
# fp32 lanes per SM on sm_100-class parts (4 sub-partitions x 32)
FP32_LANES_PER_SM = 128
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_dram_traffic.txt")


# ------------------------------------------------------------------ accounting

def bytes_per_token_head(d_k: int, d_v: int, io_bytes: int) -> int:
    """Algorithmic HBM bytes per token and head: q, k read and v read, o written in the
    I/O dtype; gate logits (d_k fp32) and beta (fp32) read."""
    return io_bytes * (2 * d_k + 2 * d_v) + 4 * d_k + 4


def flops_per_token_head(d_k: int, d_v: int, C: int = 16) -> int:
    """Algorithmic flops per token and head of the chunked form (a multiply-add is 2):
    W S, Q~ S and K'^T U (3 x 2 d_k d_v); K~ K^^T and Q~ K^^T (2 x 2 C d_k);
    TB K~ (2 C d_k); TB V and P U (2 x 2 C d_v)."""
    return 6 * d_k * d_v + 6 * C * d_k + 4 * C * d_v


def state_bytes(x) -> int:
    per = x.n_seq * x.n_heads * x.d_k * x.d_v * 4
    return per * (2 if x.h0 is not None else 1)   # h0 read (if given), h_final written


def bwd_kernel_bytes(x):
    """Bytes each kernel of the tensor-core backward (bf16, d = 128) must move per call
    in its design, summed over the (chunk, head) items: the prep record written (44352 B)
    from the q, k, v, gate-logit rows; each serial pass's bf16 state tiles written
    (34816 B) and the record parts it reads (once per item from DRAM); the local kernel's
    two state tiles and record read, its V, dO and gate-logit rows read and its gradients
    written. None for other configurations."""
    if not (str(x.dtype).endswith("bfloat16") and x.d_k == 128 and x.d_v == 128):
        return None
    rows = [max(0, b - a) for a, b in zip(x.cu_host[:-1], x.cu_host[1:])]
    tile, rec, ops, ut = 34816, 44352, 14336, 8192
    tot = [0, 0, 0]
    for n_rows in rows:
        for c0 in range(0, n_rows, 16):
            L = min(16, n_rows - c0)
            tot[0] += L * (3 * 256 + 512 + 4) + rec
            tot[1] += 2 * 4352 + 512 + ut + tile      # forward serial pass
            tot[1] += ops + L * 256 + tile            # reverse serial pass
            tot[2] += 2 * tile + rec + L * (2 * 256 + 512) + L * (3 * 256 + 512 + 4)
    return [t * x.n_heads for t in tot[:3]]


def algorithmic_bytes(x) -> int:
    io = 2 if str(x.dtype).endswith("bfloat16") else 4
    return x.n_tok * x.n_heads * bytes_per_token_head(x.d_k, x.d_v, io) + state_bytes(x)


def algorithmic_flops(x) -> int:
    return x.n_tok * x.n_heads * flops_per_token_head(x.d_k, x.d_v)


def kernel_source_digest(sources=None) -> str:
    """Digest of the kernel sources with comments and whitespace removed, so that the
    recorded ncu traffic stays valid across comment edits and is dropped on any code
    change."""
    h = hashlib.sha256()
    for rel in (sources or KERNEL_SOURCES) + ["chunked_linear_attention_kda_gb300/csrc/kda_internal.h"]:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, sources=None):
    """DRAM bytes per launch from the committed ncu summary, only if it was taken on
    the current kernel sources (the digest must match)."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    digest = kernel_source_digest(sources)
    for line in open(TRAFFIC_FILE):
        f = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
        if f.get("digest") == digest and f.get("workload") == workload:
            try:
                return int(float(f["dram_bytes_per_launch"]))
            except (KeyError, ValueError):
                return None
    return None


def fp32_alu_peak(dev, sm_max_mhz):
    """fp32 FMA peak of this device: SM count (queried) x 128 fp32 lanes x 2 flops x the
    maximum SM clock nvidia-smi reports during the run (2070 MHz if it reported none)."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = float(sm_max_mhz) if sm_max_mhz else 2070.0
    tf = sms * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12
    src = (f"derived: {sms} SMs (device query) x {FP32_LANES_PER_SM} fp32 lanes x 2 flops x "
           f"{mhz:.0f} MHz ({'nvidia-smi clocks.max.sm' if sm_max_mhz else 'nominal maximum'})")
    return tf, src


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="kda_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": rows[0][1],
                "power_w_max": max(r[2] for r in rows), "samples": len(rows),
                "reasons": reasons}


# ------------------------------------------------------------------ distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, local):
    import torch
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world > 1


def barrier(on):
    if on:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, on: bool, device) -> float:
    if not on:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ oracle timing

def oracle_sample(x, max_tokens: int, heads=None, threads=None, want_state=False):
    """The oracle on the first ``max_tokens`` tokens of every sequence (and the given
    heads), on ``threads`` host threads (default: all). Returns (seconds, token-heads
    processed, threads, the oracle's outputs of the sample); with ``want_state`` the
    oracle's final states are appended."""
    import kda_inputs as K
    from oracle import recurrence
    px = K.prefix(x, max_tokens)
    if heads is not None:
        px = K.slice_heads(px, heads)
    cpu = lambda t: None if t is None else t.detach().to("cpu")  # noqa: E731
    args = [cpu(px.q), cpu(px.k), cpu(px.v), cpu(px.a), cpu(px.beta), cpu(px.h0)]
    threads = threads or recurrence.default_threads()
    recurrence.build()
    t0 = time.perf_counter()
    o_ref, h_ref = recurrence.kda_forward(*args, px.cu_host, threads=threads,
                                          want_state=want_state)
    dt = time.perf_counter() - t0
    if want_state:
        return dt, px.n_tok * px.n_heads, threads, o_ref, h_ref
    return dt, px.n_tok * px.n_heads, threads, o_ref


def prefix_rel_l2(x, out, tokens: int, o_ref):
    """rel-L2 of the GPU output ``out`` (the whole workload) against the oracle's output
    ``o_ref`` on the first ``tokens`` tokens of every sequence (by causality those rows do
    not depend on anything after them): (over the whole sample, worst over (sequence,
    head) pairs with at least 16 tokens in the sample)."""
    import numpy as np
    num = den = 0.0
    worst = 0.0
    row = 0
    for i in range(x.n_seq):
        s0 = x.cu_host[i]
        n = min(x.cu_host[i + 1] - s0, tokens)
        hn = np.zeros(x.n_heads)
        hd = np.zeros(x.n_heads)
        for c in range(0, n, 8192):
            m = min(8192, n - c)
            g = out[s0 + c:s0 + c + m].detach().to("cpu", torch_float64()).numpy()
            r = o_ref[row + c:row + c + m]
            hn += ((g - r) ** 2).sum(axis=(0, 2))
            hd += (r ** 2).sum(axis=(0, 2))
        num += float(hn.sum())
        den += float(hd.sum())
        if n >= 16:
            worst = max(worst, float(np.max(np.sqrt(hn / np.maximum(hd, 1e-300)))))
        row += n
    return (num / den) ** 0.5 if den > 0 else num ** 0.5, worst


def state_rel_l2(hf, h_ref):
    """(whole-tensor, worst over (sequence, head)) rel-L2 of final states."""
    import numpy as np
    g = hf.detach().to("cpu", torch_float64()).numpy()
    r = np.asarray(h_ref, dtype=np.float64)
    num = ((g - r) ** 2).sum(axis=(2, 3))
    den = (r ** 2).sum(axis=(2, 3))
    whole = float(np.sqrt(num.sum() / max(den.sum(), 1e-300)))
    return whole, float(np.max(np.sqrt(num / np.maximum(den, 1e-300))))


def output_diagnostics(kda, out, hf):
    """Non-finite count over the outputs and final states (the library's counter) and the
    Frobenius norms of the final states, taken outside the timed region."""
    import torch
    nrm = torch.linalg.vector_norm(hf.float(), dim=(2, 3))
    return {"nonfinite": int(kda.count_nonfinite(out, hf)),
            "h_final_fro": round(float(torch.linalg.vector_norm(hf.float())), 4),
            "h_final_fro_max_per_head": round(float(nrm.max()), 4),
            "h_final_fro_min_per_head": round(float(nrm.min()), 4)}


def torch_float64():
    import torch
    return torch.float64


def cpu_baseline(x, budget_s: float = 15.0, out=None, hf=None):
    """Time the oracle on a bounded prefix sample, growing it until it takes a few
    seconds, scaled to the workload's tokens/s (a token counts all H heads). With the
    GPU's output ``out`` of the same inputs, also its rel-L2 against the oracle on that
    sample (key ``parity``), and with ``hf`` that of the final states when the sample
    covers every sequence whole."""
    tokens = 256
    while True:
        full = tokens >= max(x.lengths())
        dt, th, threads, o_ref, h_ref = oracle_sample(x, tokens, want_state=True)
        if dt > budget_s / 4 or full:
            break
        tokens = min(tokens * 4, max(x.lengths()))
    value = th / x.n_heads / dt
    # the same oracle once on one thread, on a smaller prefix (about budget_s / 8)
    t1 = 64
    while True:
        dt1, th1, _, _ = oracle_sample(x, t1, threads=1)
        if dt1 > budget_s / 16 or t1 >= max(x.lengths()):
            break
        t1 = min(t1 * 4, max(x.lengths()))
    parity = None
    if out is not None:
        import torch
        whole, worst = prefix_rel_l2(x, out, tokens, o_ref)
        parity = {"rel_l2_out": whole, "rel_l2_out_max_per_head": worst,
                  "bar": 1e-2 if x.dtype == torch.bfloat16 else 1e-4,
                  "sample": f"outputs of the first {tokens} tokens of every sequence, all "
                            f"{x.n_heads} heads, of the timed run against the fp64 oracle; "
                            "max_per_head is the worst (sequence, head) pair"}
        if full and hf is not None:
            parity["rel_l2_h_final"], parity["rel_l2_h_final_max_per_head"] = \
                state_rel_l2(hf, h_ref)
    del o_ref, h_ref
    return {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
            "seconds": dt, "parity": parity,
            "sample": f"fp64 token-by-token oracle on the first {tokens} tokens of every "
                      f"sequence, all {x.n_heads} heads ({th} token-heads), "
                      f"{threads} host threads",
            "single_thread": {"value": th1 / x.n_heads / dt1, "unit": UNIT, "cores": 1,
                              "seconds": dt1,
                              "sample": f"first {t1} tokens of every sequence, all "
                                        f"{x.n_heads} heads ({th1} token-heads)"}}


# ------------------------------------------------------------------ our arm

def timed_forward(kda, x, dev, stream, steps, warmup, on):
    """Warm up, then time ``steps`` forward calls over ``x`` (inputs resident) with CUDA
    events on the launching stream, bracketed by a barrier and a synchronise; nvidia-smi
    clocks sampled meanwhile. Returns (out, h_final, total ms (max over ranks), per-call
    ms, kernel launches, clocks)."""
    import torch
    out = torch.empty((x.n_tok, x.n_heads, x.d_v), dtype=x.dtype, device=dev)
    hf = torch.empty((x.n_seq, x.n_heads, x.d_k, x.d_v), dtype=torch.float32, device=dev)

    def step():
        kda.chunk_fwd(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_seqlens, out=out, h_final=hf)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    n0 = kda.kernel_launch_count()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    barrier(on)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        t_all0 = torch.cuda.Event(enable_timing=True)
        t_all1 = torch.cuda.Event(enable_timing=True)
        t_all0.record(stream)
        for i in range(steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        t_all1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(on)
    launches = kda.kernel_launch_count() - n0
    total_ms = max_over_ranks(t_all0.elapsed_time(t_all1), on, dev)
    per_launch_ms = [s_.elapsed_time(e) for s_, e in zip(starts, ends)]
    return out, hf, total_ms, per_launch_ms, launches, clk.summary()


def hbm_roofline(x, per_launch_ms, launches, steps, peaks):
    """The forward kernel's roofline entry: algorithmic bytes per launch over the mean
    event-timed launch duration, against the measured HBM copy bandwidth."""
    bytes_launch = algorithmic_bytes(x)
    flops_launch = algorithmic_flops(x)
    launches_per_step = max(1, launches // max(1, steps))
    mean_launch_s = statistics.mean(per_launch_ms) * 1e-3 / launches_per_step
    achieved_gbs = bytes_launch / launches_per_step / mean_launch_s / 1e9
    return {"bound": "hbm", "achieved": round(achieved_gbs, 1),
            "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved_gbs / peaks["hbm_gbs"], 4),
            "traffic": recorded_traffic(x.name),
            "peak_source": f"{peaks['source']} (HBM copy bandwidth, MEASURED_PEAKS.json)",
            "algorithmic_bytes_per_launch": bytes_launch,
            "tensor_tflops": round(flops_launch / mean_launch_s / 1e12, 1),
            "tensor_frac_of_bf16_peak": round(flops_launch / mean_launch_s / 1e12 /
                                              peaks["bf16_tflops"], 4)}


def extra_workload(kda, K, index, prefix, dev, stream, args, on, rank, world):
    """One of the workloads reported beside the headline: the same timing, roofline and
    output diagnostics, and (rank 0, one GPU) the oracle on the first ``prefix`` tokens of
    every sequence, all heads, with the worst (sequence, head) rel-L2."""
    import torch
    x = K.make_workload(index, dev, seed=K.SEED_BASE + index + 7919 * rank)
    out, hf, total_ms, per_ms, launches, clocks = timed_forward(
        kda, x, dev, stream, args.steps, args.warmup, on)
    peaks = measured_peaks()
    entry = {"value": round(x.n_tok * world * args.steps / (total_ms * 1e-3), 1), "unit": UNIT,
             "ms_per_step": round(total_ms / args.steps, 4), "steps": args.steps,
             "tokens_per_gpu": x.n_tok, "heads": x.n_heads, "n_seq": x.n_seq,
             "gpu_launches": int(launches),
             "roofline": hbm_roofline(x, per_ms, launches, args.steps, peaks),
             "clocks": clocks, "diagnostics": output_diagnostics(kda, out, hf)}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t0 = time.perf_counter()
        _, _, threads, o_ref = oracle_sample(x, prefix)
        whole, worst = prefix_rel_l2(x, out, prefix, o_ref)
        entry["parity"] = {"rel_l2_out": whole, "rel_l2_out_max_per_head": worst,
                           "bar": 1e-2 if x.dtype == torch.bfloat16 else 1e-4,
                           "oracle_seconds": round(time.perf_counter() - t0, 2),
                           "sample": f"outputs of the first {prefix} tokens of every sequence, "
                                     f"all {x.n_heads} heads, of the timed run against the "
                                     f"fp64 oracle ({threads} host threads); max_per_head is "
                                     "the worst (sequence, head) pair"}
        del o_ref
    del out, hf, x
    torch.cuda.empty_cache()
    return entry


def run_ours(args):
    import torch
    import chunked_linear_attention_kda_gb300 as kda
    import kda_inputs as K

    world, rank, local = dist_env()
    on = init_dist(world, local)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    kda.load_library(build_if_missing=True)

    x = K.make_workload(args.workload, dev, seed=K.SEED_BASE + args.workload + 7919 * rank)
    stream = torch.cuda.current_stream(dev)
    out, hf, total_ms, per_launch_ms, launches, clocks = timed_forward(
        kda, x, dev, stream, args.steps, args.warmup, on)
    ms_per_step = total_ms / args.steps
    tokens_all = x.n_tok * world
    value = tokens_all * args.steps / (total_ms * 1e-3)
    roofline = hbm_roofline(x, per_launch_ms, launches, args.steps, measured_peaks())
    diagnostics = output_diagnostics(kda, out, hf)

    # end-to-end through the host-buffer entry point
    e2e = measure_e2e(x, dev, stream, max(1, min(args.steps, 20)), kda)
    e2e["value"] = e2e["value"] * world

    line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if x.dtype == torch.bfloat16 else "f32",
            "data": "synthetic",
            "config": {"workload": x.name, "tokens_per_gpu": x.n_tok, "heads": x.n_heads,
                       "d_k": x.d_k, "d_v": x.d_v, "chunk": 16, "serial_step_tokens": 64,
                       "n_seq": x.n_seq, "global_batch_tokens": tokens_all,
                       "parallelism": f"independent replicas x{world}" if world > 1 else
                       "single GPU",
                       "l2": "inputs (%.2f GB) exceed the 129 MB L2; no flush between steps"
                             % (algorithmic_bytes(x) / 1e9)},
            "roofline": roofline, "e2e": e2e, "gpu_launches": int(launches),
            "clocks": clocks, "kernel_digest": kernel_source_digest(),
            "diagnostics": diagnostics}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline(x, out=out, hf=hf)
        line["parity"] = cb.pop("parity")
        line["cpu_baseline"] = cb
    del out, hf, x
    torch.cuda.empty_cache()
    if args.workload == 3 and not args.no_extra_workloads:
        line["workloads"] = {}
        for index, prefix in EXTRA_WORKLOADS.items():
            name = K.WORKLOADS[index]
            line["workloads"][name] = extra_workload(kda, K, index, prefix, dev, stream, args,
                                                     on, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if on:
        import torch.distributed as dist
        dist.destroy_process_group()


def measure_e2e(x, dev, stream, steps, kda):
    """Host inputs -> device -> kernel -> host outputs, timed with CUDA events."""
    import torch
    pin = lambda t: None if t is None else t.detach().to("cpu").pin_memory()  # noqa: E731
    host = {"q": pin(x.q), "k": pin(x.k), "v": pin(x.v), "gate_logits": pin(x.a),
            "beta": pin(x.beta), "h0": pin(x.h0), "cu_seqlens": pin(x.cu_seqlens)}
    h_out = torch.empty((x.n_tok, x.n_heads, x.d_v), dtype=x.dtype).pin_memory()
    h_hf = torch.empty((x.n_seq, x.n_heads, x.d_k, x.d_v), dtype=torch.float32).pin_memory()
    devb = {k: torch.empty_like(v, device=dev) if v is not None else None
            for k, v in host.items()}
    devb["out"] = torch.empty(h_out.shape, dtype=x.dtype, device=dev)
    devb["h_final"] = torch.empty(h_hf.shape, dtype=torch.float32, device=dev)

    args = (host["q"], host["k"], host["v"], host["gate_logits"], host["beta"], host["h0"],
            host["cu_seqlens"], h_out, h_hf, devb, stream)

    in_bytes = sum(host[n].numel() * host[n].element_size()
                   for n in ("q", "k", "v", "gate_logits", "beta"))
    segments = max(1, min(kda.PIPELINE_MAX_SEGMENTS, in_bytes // kda.PIPELINE_SEGMENT_BYTES))

    def pipelined():   # the binding's default segment count, stated in the report
        kda.chunk_fwd_from_host_pipelined(*args, n_segments=segments)

    def serial():
        kda.chunk_fwd_from_host(*args)

    def timed(call):
        """(median, mean, max) over ``steps`` back-to-back calls, each bracketed by CUDA
        events on the stream (every call ends with the stream waiting for its last copy),
        after three untimed calls."""
        for _ in range(3):
            call()
        torch.cuda.synchronize(dev)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        ev[0].record(stream)
        for i in range(steps):
            call()
            ev[i + 1].record(stream)
        torch.cuda.synchronize(dev)
        per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
        return statistics.median(per), ev[0].elapsed_time(ev[steps]) / steps, max(per)

    def inputs_only():  # the floor: the step's host-to-device bytes alone
        for name, t in host.items():
            if t is not None:
                devb[name].copy_(t, non_blocking=True)

    ms, ms_mean, ms_max = timed(pipelined)
    ms_serial, _, _ = timed(serial)
    with torch.cuda.stream(stream):
        ms_h2d, ms_h2d_mean, ms_h2d_max = timed(inputs_only)
    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    d2h = h_out.numel() * h_out.element_size() + h_hf.numel() * 4
    return {"value": round(x.n_tok / (ms * 1e-3), 1), "unit": UNIT,
            "ms_per_step": round(ms, 3), "mean_ms_per_step": round(ms_mean, 3),
            "max_ms_per_step": round(ms_max, 3),
            "statistic": f"median of {steps} event-timed calls",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "api": f"kda_chunk_fwd_from_host_pipelined (pinned host buffers, {segments} "
                   "segment(s): copies overlap the kernels)",
            "unpipelined_ms_per_step": round(ms_serial, 3),
            "h2d_only_ms_per_step": round(ms_h2d, 3),
            # the same spread for the inputs' copies alone: a slow call there as well points
            # at the host link, not at the library
            "h2d_only_mean_ms_per_step": round(ms_h2d_mean, 3),
            "h2d_only_max_ms_per_step": round(ms_h2d_max, 3)}


# ------------------------------------------------------------------ decode step

def decode_bytes_per_seq_head(d_k: int, d_v: int, io_bytes: int) -> int:
    """Algorithmic HBM bytes of one decode step per sequence and head: the fp32 state
    read and written, q, k, v read and o written in the I/O dtype, gate logits and beta
    read."""
    return 8 * d_k * d_v + io_bytes * (2 * d_k + 2 * d_v) + 4 * d_k + 4


def run_decode(args):
    import torch
    import chunked_linear_attention_kda_gb300 as kda
    import kda_inputs as K

    world, rank, local = dist_env()
    on = init_dist(world, local)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    kda.load_library(build_if_missing=True)
    B, H, d = DECODE_B, DECODE_H, DECODE_D
    x = K.make_inputs([1] * B, H, d, d, dtype=torch.bfloat16, device=dev,
                      seed=K.SEED_BASE + 99 + 7919 * rank, h0_std=0.5, name="decode")
    state = x.h0.clone()
    out = torch.empty((B, H, d), dtype=x.dtype, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kda.decode_step(x.q, x.k, x.v, x.a, x.beta, state, out=out)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    n0 = kda.kernel_launch_count()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(on)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(on)
    launches = kda.kernel_launch_count() - n0
    total_ms = max_over_ranks(t0.elapsed_time(t1), on, dev)
    value = B * world * args.steps / (total_ms * 1e-3)
    peaks = measured_peaks()
    bytes_launch = B * H * decode_bytes_per_seq_head(d, d, 2)
    mean_launch_s = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends)) * 1e-3
    achieved = bytes_launch / mean_launch_s / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": recorded_traffic("decode-B256-H32-d128", DECODE_SOURCES),
                "peak_source": f"{peaks['source']} (HBM copy bandwidth, MEASURED_PEAKS.json)",
                "algorithmic_bytes_per_launch": bytes_launch}

    # end to end through the public API: this step's inputs copied from pinned host
    # memory, the step, its outputs copied back; the state stays resident on the device
    host = [t.detach().to("cpu").pin_memory() for t in (x.q, x.k, x.v, x.a, x.beta)]
    devb = [torch.empty_like(t, device=dev) for t in host]
    h_out = torch.empty((B, H, d), dtype=x.dtype).pin_memory()
    e_steps = max(1, min(args.steps, 20))

    def e2e_step():
        for hb, db in zip(host, devb):
            db.copy_(hb, non_blocking=True)
        o = kda.decode_step(*devb, state)
        h_out.copy_(o, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e_ms = e0.elapsed_time(e1) / e_steps
    e2e = {"value": round(B * world / (e_ms * 1e-3), 1), "unit": "tokens/s",
           "ms_per_step": round(e_ms, 4),
           "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in host),
           "d2h_bytes_per_step": h_out.numel() * h_out.element_size(), "steps": e_steps,
           "api": "decode_step with pinned host inputs and outputs (state resident)"}
    line = {"metric": DECODE_METRIC, "value": round(value, 1), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "decode-B256-H32-d128", "sequences_per_gpu": B, "heads": H,
                       "d_k": d, "d_v": d, "state_bytes": B * H * d * d * 4,
                       "l2": "state (%.0f MiB) exceeds the 129 MB L2; no flush between steps"
                             % (B * H * d * d * 4 / 2**20)},
            "roofline": roofline, "e2e": e2e, "gpu_launches": int(launches),
            "clocks": clk.summary(), "kernel_digest": kernel_source_digest(DECODE_SOURCES)}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = decode_cpu_baseline(x)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if on:
        import torch.distributed as dist
        dist.destroy_process_group()


def decode_cpu_baseline(x, budget_s: float = 10.0):
    """The oracle's decode step on the host cores, on the first n sequences of the batch
    (all heads), n grown until a call takes a few seconds; scaled to tokens/s."""
    from oracle import recurrence
    cpu = lambda t: t.detach().to("cpu")  # noqa: E731
    threads = recurrence.default_threads()
    recurrence.build()
    n = 8
    while True:
        args = [cpu(t[:n]) for t in (x.q, x.k, x.v, x.a, x.beta, x.h0)]
        t0 = time.perf_counter()
        recurrence.decode_step(*args, threads=threads)
        dt = time.perf_counter() - t0
        if dt > budget_s / 4 or n >= x.q.shape[0]:
            break
        n = min(n * 4, x.q.shape[0])
    # repeat the step (each from the previous state) until the sample takes a few seconds
    reps, state = 0, args[5]
    t0 = time.perf_counter()
    while True:
        _, state = recurrence.decode_step(*args[:5], state, threads=threads)
        reps += 1
        if time.perf_counter() - t0 > budget_s / 4:
            break
    dt = time.perf_counter() - t0
    return {"value": n * reps / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "seconds": dt, "sample": f"{reps} fp64 oracle decode steps on {n} sequences x "
                                     f"{x.q.shape[1]} heads, {threads} host threads"}


# ------------------------------------------------------------------ backward pass

def run_backward(args):
    import torch
    import chunked_linear_attention_kda_gb300 as kda
    import kda_inputs as K

    world, rank, local = dist_env()
    on = init_dist(world, local)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib = kda.load_library(build_if_missing=True)
    x = K.make_workload(args.workload, dev, seed=K.SEED_BASE + args.workload + 7919 * rank)
    g = torch.Generator(device="cpu").manual_seed(1234 + rank)
    dout = torch.randn((x.n_tok, x.n_heads, x.d_v), generator=g).to(dev, x.dtype)
    ws = torch.empty(lib.kda_chunk_bwd_workspace_bytes(x.n_tok, x.n_seq, x.n_heads, x.d_k,
                                                       x.d_v), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        return kda.chunk_bwd(x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_seqlens, dout, None,
                             want_dh0=x.h0 is not None, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    n0 = kda.kernel_launch_count()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(on)
    torch.cuda.synchronize(dev)
    kda.bwd_timing_start(args.steps)  # events around each kernel of every timed call
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(on)
    kernel_ms, calls = kda.bwd_timing_read()
    kernel_ms = [t / max(1, calls) for t in kernel_ms]
    launches = kda.kernel_launch_count() - n0
    total_ms = max_over_ranks(t0.elapsed_time(t1), on, dev)
    value = x.n_tok * world * args.steps / (total_ms * 1e-3)
    mean_s = statistics.mean(s_.elapsed_time(e) for s_, e in zip(starts, ends)) * 1e-3
    peaks = measured_peaks()
    kbytes = bwd_kernel_bytes(x)
    names = BACKWARD_KERNELS
    if kbytes is not None:  # three launches: prep, both serial passes, local gradients
        names, kernel_ms = BACKWARD_KERNELS_TC, [kernel_ms[0], kernel_ms[1] + kernel_ms[2], kernel_ms[3]]
    kernels = {nm: {"ms": round(t, 4), "share": round(t / sum(kernel_ms), 4)}
               for nm, t in zip(names, kernel_ms)}
    if kbytes is not None:
        for nm, b, t in zip(names, kbytes, kernel_ms):
            kernels[nm].update(bytes=b, gbs=round(b / (t * 1e-3) / 1e9, 1))
        top = max(range(len(names)), key=lambda i: kernel_ms[i])
        achieved = kbytes[top] / (kernel_ms[top] * 1e-3) / 1e9
        roofline = {"bound": "hbm", "kernel": names[top], "achieved": round(achieved, 1),
                    "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": round(achieved / peaks["hbm_gbs"], 4),
                    "traffic": recorded_traffic(f"{x.name}:{names[top]}", BACKWARD_SOURCES),
                    "algorithmic_bytes_per_launch": kbytes[top],
                    "launch_ms": round(kernel_ms[top], 4),
                    "peak_source": f"{peaks['source']} (HBM copy bandwidth, MEASURED_PEAKS.json)"}
    else:  # the fp32 FMA kernels
        flops = 2 * algorithmic_flops(x)   # a gradient product for each operand of each product
        achieved = flops / mean_s / 1e12
        clk_sum = clk.summary()
        alu, alu_src = fp32_alu_peak(dev, clk_sum.get("sm_max_mhz"))
        roofline = {"bound": "alu", "achieved": round(achieved, 2), "peak": round(alu, 1),
                    "unit": "TFLOP/s", "frac": round(achieved / alu, 4), "traffic": None,
                    "peak_source": alu_src}

    # end to end through the public API: inputs and upstream gradients from pinned host
    # memory, the backward, the gradients back to pinned host memory
    host_in = [t.detach().to("cpu").pin_memory() for t in (x.q, x.k, x.v, x.a, x.beta, dout)]
    dev_in = [torch.empty_like(t, device=dev) for t in host_in]
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory()
                for t in (x.q, x.k, x.v, x.a, x.beta)]

    def e2e_step():
        for hb, db in zip(host_in, dev_in):
            db.copy_(hb, non_blocking=True)
        grads = kda.chunk_bwd(*dev_in[:5], x.h0, x.cu_seqlens, dev_in[5], None,
                              want_dh0=False, workspace=ws)
        for hb, gd in zip(host_out, grads[:5]):
            hb.copy_(gd, non_blocking=True)

    e_steps = max(1, min(args.steps, 3))
    e2e_step()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e_ms = e0.elapsed_time(e1) / e_steps
    e2e = {"value": round(x.n_tok * world / (e_ms * 1e-3), 1), "unit": UNIT,
           "ms_per_step": round(e_ms, 3),
           "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in host_in),
           "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in host_out),
           "steps": e_steps, "api": "chunk_bwd with pinned host inputs and gradients"}
    line = {"metric": BACKWARD_METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("bf16 tensor-core operands, f32 accumulation" if kbytes is not None
                      else "f32"),
            "data": "synthetic",
            "config": {"workload": x.name, "tokens_per_gpu": x.n_tok, "heads": x.n_heads,
                       "d_k": x.d_k, "d_v": x.d_v, "chunk": 16,
                       "workspace_bytes": int(ws.numel()),
                       "l2": "inputs and workspace exceed the 129 MB L2; no flush"},
            "roofline": roofline, "kernels": kernels, "e2e": e2e, "gpu_launches": int(launches),
            "clocks": clk_sum if kbytes is None else clk.summary(),
            "kernel_digest": kernel_source_digest(BACKWARD_SOURCES)}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = backward_cpu_baseline(x, dout)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if on:
        import torch.distributed as dist
        dist.destroy_process_group()


def backward_cpu_baseline(x, dout, budget_s: float = 10.0):
    """The reverse-mode oracle on the host cores on a prefix of the workload (all heads),
    grown until it takes a few seconds; scaled to tokens/s."""
    import torch
    from oracle import backward as B
    cpu = lambda t: None if t is None else t.detach().to("cpu")  # noqa: E731
    tokens = 8
    while True:
        sl = slice(0, tokens)
        t0 = time.perf_counter()
        B.kda_backward(cpu(x.q[sl]), cpu(x.k[sl]), cpu(x.v[sl]), cpu(x.a[sl]), cpu(x.beta[sl]),
                       cpu(x.h0[:1]) if x.h0 is not None else None, [0, tokens],
                       cpu(dout[sl]))
        dt = time.perf_counter() - t0
        if dt > budget_s / 4 or tokens >= 4096:
            break
        tokens *= 2
    return {"value": tokens / dt, "unit": UNIT, "cores": torch.get_num_threads(),
            "kind": "oracle", "seconds": dt,
            "sample": f"fp64 reverse-mode oracle on the first {tokens} tokens of the first "
                      f"sequence, all {x.n_heads} heads"}


# ------------------------------------------------------------------ gate projection

PROJ_M, PROJ_D, PROJ_N = 65536, 4096, 4096
PROJ_SOURCES = ["chunked_linear_attention_kda_gb300/csrc/kda_gemm.cu"]


def run_projection(args):
    import torch
    import chunked_linear_attention_kda_gb300 as kda
    dev = torch.device("cuda", 0)
    kda.load_library(build_if_missing=True)
    M, D, N = PROJ_M, PROJ_D, PROJ_N
    g = torch.Generator(device="cpu").manual_seed(77)
    x = torch.randn((M, D), generator=g).to(dev, torch.bfloat16)
    w = (torch.randn((N, D), generator=g) * D ** -0.5).to(dev, torch.bfloat16)
    b = torch.randn((N,), generator=g).to(dev)
    out = torch.empty((M, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kda.gate_projection(x, w, b, out=out)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    n0 = kda.kernel_launch_count()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(0) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
    launches = kda.kernel_launch_count() - n0
    total_ms = t0.elapsed_time(t1)
    mean_s = statistics.mean(s_.elapsed_time(e) for s_, e in zip(starts, ends)) * 1e-3
    flops = 2 * M * N * D
    peaks = measured_peaks()
    achieved = flops / mean_s / 1e12
    # the same GEMM with bf16 output (kda_gate_projection_out), timed the same way
    out16 = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    for _ in range(args.warmup):
        kda.gate_projection(x, w, b, out=out16)
    torch.cuda.synchronize(dev)
    b0 = torch.cuda.Event(enable_timing=True)
    b1 = torch.cuda.Event(enable_timing=True)
    b0.record(stream)
    for _ in range(args.steps):
        kda.gate_projection(x, w, b, out=out16)
    b1.record(stream)
    torch.cuda.synchronize(dev)
    bf16_ms = b0.elapsed_time(b1) / args.steps
    # context: the same product through cuBLAS (torch.mm, bf16 out), not on the product path
    for _ in range(3):
        torch.mm(x, w.t())
    torch.cuda.synchronize(dev)
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for _ in range(10):
        torch.mm(x, w.t())
    c1.record(stream)
    torch.cuda.synchronize(dev)
    cublas_ms = c0.elapsed_time(c1) / 10
    line = {"metric": "KDA gate projection tokens/s (a = x W^T + b, tcgen05 GEMM) and % of "
                      "bf16 tensor roofline",
            "value": round(M * args.steps / (total_ms * 1e-3), 1), "unit": "tokens/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 products, fp32 accumulate",
            "data": "synthetic",
            "config": {"workload": f"gate-projection-M{M}-K{D}-N{N}", "tokens": M,
                       "d_model": D, "n_out": N,
                       "l2": "x (512 MiB) and a (1 GiB) exceed the 129 MB L2; no flush"},
            "roofline": {"bound": "tensor", "achieved": round(achieved, 1),
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(achieved / peaks["bf16_tflops"], 4), "traffic": None,
                         "peak_source": f"{peaks['source']} (cuBLAS bf16 burst, "
                                        "MEASURED_PEAKS.json)",
                         "algorithmic_flops_per_launch": flops},
            "cublas_bf16_mm_ms_context": round(cublas_ms, 4),
            "bf16_output": {"ms_per_step": round(bf16_ms, 4),
                            "tflops": round(flops / (bf16_ms * 1e-3) / 1e12, 1),
                            "frac_of_bf16_peak": round(flops / (bf16_ms * 1e-3) / 1e12 /
                                                       peaks["bf16_tflops"], 4),
                            "api": "kda_gate_projection_out(..., KDA_BF16)"},
            "gpu_launches": int(launches), "clocks": clk.summary(),
            "kernel_digest": kernel_source_digest(PROJ_SOURCES)}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ gated forward

def run_gated(args):
    """The forward fed by the gate projection (``kda_chunk_fwd_gated``) on the 64K workload
    with d_model = 4096, against the projection GEMM and the forward run back to back."""
    import torch
    import chunked_linear_attention_kda_gb300 as kda
    import kda_inputs as K
    dev = torch.device("cuda", 0)
    lib = kda.load_library(build_if_missing=True)
    x = K.make_workload(3, dev)
    D, H = PROJ_D, x.n_heads
    g = torch.Generator(device="cpu").manual_seed(78)
    xx = torch.randn((x.n_tok, D), generator=g).to(dev, torch.bfloat16)
    w = (torch.randn((H * x.d_k, D), generator=g) * D ** -0.5).to(dev, torch.bfloat16)
    b = torch.randn((H * x.d_k,), generator=g).to(dev)
    a = torch.empty((x.n_tok, H, x.d_k), dtype=torch.float32, device=dev)
    out = torch.empty((x.n_tok, H, x.d_v), dtype=x.dtype, device=dev)
    hf = torch.empty((x.n_seq, H, x.d_k, x.d_v), dtype=torch.float32, device=dev)
    seg = args.segment_tokens
    ws = torch.empty(lib.kda_chunk_fwd_gated_workspace_bytes(x.n_seq, H, x.d_k, x.d_v, seg),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def separate():
        kda.gate_projection(xx, w, b, out=a.view(x.n_tok, H * x.d_k))
        kda.chunk_fwd(x.q, x.k, x.v, a, x.beta, x.h0, x.cu_seqlens, out=out, h_final=hf)

    def fused():
        kda.chunk_fwd_gated(xx, w, b, x.q, x.k, x.v, x.beta, x.h0, x.cu_seqlens, segment_tokens=seg,
                            out=out, h_final=hf, workspace=ws)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(dev)
        n0 = kda.kernel_launch_count()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with ClockSampler(0) as clk:
            e0.record(stream)
            for _ in range(args.steps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / args.steps, (kda.kernel_launch_count() - n0), clk.summary()

    ms_sep, l_sep, _ = timed(separate)
    o_sep = out.clone()
    ms_fused, l_fused, clocks = timed(fused)
    same = bool(torch.equal(out, o_sep))
    a_bytes = x.n_tok * H * x.d_k * 4
    fwd_bytes = algorithmic_bytes(x) - x.n_tok * H * (4 * x.d_k)   # the forward without a
    line = {"metric": "KDA forward with the gate projection fused (tokens/s)",
            "value": round(x.n_tok * args.steps / (ms_fused * args.steps * 1e-3), 1),
            "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_fused, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"gated-{x.name}-dmodel{D}", "tokens": x.n_tok, "heads": H,
                       "d_model": D, "segment_tokens": seg,
                       "workspace_bytes": int(ws.numel())},
            "separate_ms_per_step": round(ms_sep, 4),
            "separate": "kda_gate_projection (a written, 1 GiB fp32) then kda_chunk_fwd (a read)",
            "bitwise_equal_to_separate": same,
            "gate_logit_bytes_not_materialised": a_bytes,
            "hbm_bytes_algorithmic": {"separate": int(fwd_bytes + 2 * a_bytes + xx.numel() * 2 +
                                                      w.numel() * 2),
                                      "fused": int(fwd_bytes + xx.numel() * 2 + w.numel() * 2)},
            "gpu_launches": int(l_fused), "gpu_launches_separate": int(l_sep), "clocks": clocks}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ contrast variants

def run_contrast(args):
    import torch
    import chunked_linear_attention_kda_gb300 as kda
    import kda_inputs as K
    dev = torch.device("cuda", 0)
    kda.load_library(build_if_missing=True)
    x = K.make_workload(args.workload, dev)
    fargs = (x.q, x.k, x.v, x.a, x.beta, x.h0, x.cu_seqlens)
    steps = max(1, min(args.steps, 5))

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / steps

    with ClockSampler(0) as clk:
        ms = {"tensor_core_dense_bounded": timed(lambda: kda.chunk_fwd(*fargs))}
        for gate in ("bounded", "softplus"):
            for diag in ("dense", "pairs"):
                ms[f"simt_{diag}_{gate}"] = timed(
                    lambda g=gate, d=diag: kda.chunk_fwd_variant(*fargs, gate=g, diag=d))
    ratio = ms["simt_pairs_bounded"] / ms["simt_dense_bounded"]
    line = {"metric": "KDA forward time, position-pair / dense diagonal tile (same fp32 "
                      "SIMT kernel otherwise)",
            "value": round(ratio, 3), "unit": "x", "n_gpus": 1, "steps": steps,
            "warmup": args.warmup, "ms_per_step": round(ms["simt_pairs_bounded"], 3),
            "higher_is_better": True, "dtype": "f32 arithmetic", "data": "synthetic",
            "config": {"workload": x.name},
            "ms": {k: round(v, 3) for k, v in ms.items()},
            "note": "the softplus + dense variant is finite on this workload (gate logits "
                    "~ N(0, 2): its chunk decay stays inside fp32); tests reproduce its "
                    "overflow at -40 per token",
            "clocks": clk.summary(), "kernel_digest": kernel_source_digest()}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ reference arm

def run_reference(args):
    """The reference arm: the fp64 oracle on the host cores, each step a bounded
    prefix sample of the same workload, reported in the same unit."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import torch
    import kda_inputs as K
    # the same recipe, generated on the host only up to the longest prefix sampled
    x = K.make_workload(args.workload, "cpu", max_len=16384)
    tokens = 512
    # size one step to about a second of host work
    while True:
        dt, th, threads, _ = oracle_sample(x, tokens)
        if dt > 0.5 or tokens >= max(x.lengths()):
            break
        tokens = min(tokens * 2, max(x.lengths()))
    for _ in range(args.warmup):
        oracle_sample(x, tokens)
    t0 = time.perf_counter()
    total_th = 0
    for _ in range(args.steps):
        _, th, threads, _ = oracle_sample(x, tokens)
        total_th += th
    el = time.perf_counter() - t0
    value = total_th / x.n_heads / el
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": x.name, "heads": x.n_heads, "d_k": x.d_k, "d_v": x.d_v,
                       "chunk": 16},
            "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": threads,
                             "kind": "oracle",
                             "sample": f"first {tokens} tokens of every sequence, all "
                                       f"{x.n_heads} heads, per step"},
            "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    _ = torch


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", type=int, default=3, choices=[0, 1, 2, 3, 4, 5, 6])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-workloads", action="store_true",
                    help="with the default workload, skip the 256K and packed-1M lines "
                         "reported under 'workloads'")
    ap.add_argument("--op", default="forward",
                    choices=["forward", "decode", "backward", "contrast", "projection", "gated"],
                    help="forward: the chunked forward pass (default); decode: the "
                         "recurrent decode step; backward: the backward pass; contrast: "
                         "the unbounded-gate and position-pair variants; projection: "
                         "the gate projection GEMM; gated: the forward fed by the projection "
                         "(kda_chunk_fwd_gated) against the two run back to back")
    ap.add_argument("--segment-tokens", type=int, default=4096,
                    help="segment length of --op gated")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.op == "gated":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the gated line compares entry points of this library only"}),
                  flush=True)
        else:
            run_gated(args)
    elif args.op == "projection":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the projection line has no reference arm"}), flush=True)
        else:
            run_projection(args)
    elif args.op == "contrast":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the contrast line compares variants of this library only"}),
                  flush=True)
        else:
            run_contrast(args)
    elif args.op == "backward":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the backward line has no reference arm; its cpu_baseline is "
                              "the oracle"}), flush=True)
        else:
            run_backward(args)
    elif args.op == "decode":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the decode line has no reference arm; its cpu_baseline is "
                              "the oracle"}), flush=True)
        else:
            run_decode(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
