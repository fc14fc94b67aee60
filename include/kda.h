/*
 * kda.h -- C ABI of the GB300 (sm_103a) chunked forward pass of gated delta-rule
 * linear attention with the lower-bounded per-key-channel decay (Kimi Delta
 * Attention style).
 *
 * The operation, per sequence and head, with state S in R^{d_k x d_v}:
 *
 *   g_t  = g_min * sigmoid(a_t),  g_min = -5           (per key channel)
 *   S   <- Diag(exp g_t) S
 *   S   <- S + beta_t k_t (v_t - S^T k_t)^T
 *   o_t  = d_k^-1/2 S^T q_t                              (state after the write)
 *
 * Sources: the bounded gate g = g_min * sigmoid(.) with g_min = -5 and its range
 * [g_min, 0) -- "Demystifying Trillion-Parameter MoE Models", Breakthrough 1 §2,
 * and "From Numerical Stability to Load Balancing", §2.2. The state that forgets
 * through a cumulative decay and writes key-value outer products, computed with a
 * chunked strategy in which chunks run serially through the state recurrence while
 * the inside of a chunk is matrix products scaled by exp(G_i - G_j) -- the same
 * page, §2.1. Chunks of 16 tokens, whose worst-case log-decay span 16 x (-5) = -80
 * keeps exp(+-G) representable in BF16 so the diagonal tile stays a dense
 * tensor-core product with no per-position branch -- the same page, §2.2-2.3, and
 * "Architecting Long-Context LLMs: From Sparse Attention to Stable MoE in
 * Production", §2.2-2.3. The delta-rule form of the write is what those pages call
 * "Kimi Delta Attention" / "Delta networks"; g_min = -5 and the 16-token chunk are
 * compile-time constants of this library, not parameters.
 *
 * Memory layout (all buffers contiguous, row-major, token-major, owned by the
 * caller; the library allocates nothing and keeps no state between calls):
 *   q, k          [n_tok, n_heads, d_k]   dtype (KDA_BF16 or KDA_F32)
 *   v             [n_tok, n_heads, d_v]   dtype
 *   gate_logits   [n_tok, n_heads, d_k]   float32  (a; the gate is -5*sigmoid(a))
 *   beta          [n_tok, n_heads]        float32
 *   h0            [n_seq, n_heads, d_k, d_v] float32, or NULL for a zero state
 *   cu_seqlens    [n_seq + 1] int32, device memory: sequence n owns tokens
 *                 [cu_seqlens[n], cu_seqlens[n+1]); cu_seqlens[0] = 0,
 *                 non-decreasing, cu_seqlens[n_seq] = n_tok. Empty sequences are
 *                 allowed (their final state is h0). Sequences need not be
 *                 multiples of 16 tokens.
 *   out           [n_tok, n_heads, d_v]   dtype
 *   h_final       [n_seq, n_heads, d_k, d_v] float32, or NULL to skip writing it
 * q, k, v, gate_logits and out must be 16-byte aligned; beta, h0, cu_seqlens and
 * h_final 4-byte aligned. out and h_final must not overlap any input. The state and
 * all accumulation are float32.
 *
 * Execution: every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 * legacy default stream). The return value reports argument validation and launch
 * errors only; device-side faults surface at the next synchronising CUDA call.
 * Calls are thread-safe (the only mutable global is the launch counter below). cu_seqlens is read on the
 * device only, so the forward calls do not validate its contents; breaking the rules
 * above is undefined behaviour. kda_validate_cu_seqlens checks them on the device
 * without trapping, for callers who cannot vouch for their offsets.
 */
#ifndef KDA_GB300_H_
#define KDA_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1, /* null pointer, negative size, misalignment, bad layout */
    KDA_ERR_UNSUPPORTED = 2, /* valid but not built: dtype or head dimension */
    KDA_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
    KDA_ERR_NONFINITE = 4    /* kda_check_outputs found NaN or Inf in the outputs */
} kda_status;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

/* Library version as an integer MAJOR*10000 + MINOR*100 + PATCH. */
int kda_version(void);

/* Static description of a status code. Never NULL. */
const char *kda_status_string(kda_status status);

/* Human-readable detail of the last non-OK status returned on the calling host
 * thread (empty string if none). Valid until the next call on that thread. */
const char *kda_last_error(void);

/* Number of CUDA kernels this library has launched in the process so far (all
 * threads, all devices). A diagnostic counter for benchmarks and tests: the only
 * mutable global of the library, updated atomically, never read by a kernel. */
uint64_t kda_kernel_launch_count(void);

/*
 * kda_read_device_flags -- synchronise `stream`, then copy the library's device-side
 * status word into *flags (and clear it when `reset` is non-zero). A set bit means a
 * pipeline wait inside one of the library's kernels exceeded its time limit (about
 * two seconds); that kernel then stopped early and its outputs are unspecified:
 * bit 0 the 16-token-step tensor-core forward (and the self-test below), bit 1 the
 * gate-projection GEMM, bit 2 the backward's serial passes, bit 3 the 64-token-step
 * tensor-core forward. A healthy run leaves the word 0. Returns KDA_ERR_INVALID_ARG
 * for a NULL `flags`, KDA_ERR_CUDA if the copy or the synchronisation fails.
 */
kda_status kda_read_device_flags(uint32_t *flags, int reset, void *stream);

/*
 * kda_validate_cu_seqlens -- check on the device that `cu_seqlens` (device memory,
 * n_seq + 1 int32 entries) follows the layout rules above: cu_seqlens[0] = 0,
 * non-decreasing, cu_seqlens[n_seq] = n_tok. The forward kernels read cu_seqlens on
 * the device without checking it; a caller who cannot vouch for its offsets runs this
 * first and reads the result before calling them. Writes two int32 at the device
 * address `d_status`: d_status[0] is a bit set (bit 0: cu_seqlens[0] != 0; bit 1:
 * cu_seqlens[i + 1] < cu_seqlens[i] for some i; bit 2: cu_seqlens[n_seq] != n_tok;
 * 0 = valid) and d_status[1] the smallest offending index (i for a decrease between
 * i and i + 1, 0 or n_seq for the end points; INT32_MAX when valid). Only reads
 * cu_seqlens (n_seq + 1 entries must be readable); never traps. Asynchronous on
 * `stream`. Returns KDA_ERR_INVALID_ARG for NULL or misaligned (4 bytes) pointers or
 * negative sizes, KDA_ERR_CUDA if a launch fails.
 */
kda_status kda_validate_cu_seqlens(const int32_t *cu_seqlens, int32_t n_seq, int64_t n_tok,
                                   int32_t *d_status, void *stream);

/*
 * kda_count_nonfinite -- add to the uint64 at device address `d_count` the number of
 * NaN or +-Inf elements among the `n` elements of `x` (device memory, `dtype`
 * KDA_F32 or KDA_BF16). The bounded gate is what keeps the forward finite at the
 * decay bound ("Demystifying Trillion-Parameter MoE Models", Verification, monitors
 * the rate of such values); this counter measures it. The caller zeroes *d_count.
 * Asynchronous on `stream`. Returns KDA_ERR_INVALID_ARG (NULL pointers with n > 0,
 * n < 0, x not aligned to its element, d_count not 8-byte aligned),
 * KDA_ERR_UNSUPPORTED (dtype), KDA_ERR_CUDA.
 */
kda_status kda_count_nonfinite(const void *x, int64_t n, kda_dtype dtype,
                               unsigned long long *d_count, void *stream);

/*
 * kda_check_outputs -- the non-finite count over a forward call's outputs: `n_out`
 * elements of `out` (`dtype`) and `n_h_final` fp32 elements of `h_final` (either may
 * be NULL with a zero count), using the uint64 at device address `d_scratch`.
 * Synchronises `stream`; writes the count to *count (host memory) and returns
 * KDA_ERR_NONFINITE when it is non-zero (KDA_OK otherwise), or KDA_ERR_INVALID_ARG /
 * KDA_ERR_CUDA as above.
 */
kda_status kda_check_outputs(const void *out, int64_t n_out, kda_dtype dtype, const float *h_final,
                             int64_t n_h_final, unsigned long long *d_scratch, uint64_t *count,
                             void *stream);

/*
 * kda_selftest_bounded_wait -- failure-detection self-test; no counterpart in the
 * method. Launches one thread that waits on a pipeline barrier nothing will ever
 * complete, through the same bounded-wait routine the tensor-core kernel uses, with
 * a limit of `limit_cycles` SM cycles. The wait gives up, sets bit 0 of the device
 * status word (see kda_read_device_flags) and the kernel writes 1 to the int32 at
 * device address `d_returned` (2 would mean the wait wrongly completed). Nothing
 * faults, traps or hangs. Returns KDA_ERR_INVALID_ARG for a NULL `d_returned` or a
 * non-positive limit, KDA_ERR_CUDA if the launch fails.
 */
kda_status kda_selftest_bounded_wait(int64_t limit_cycles, int32_t *d_returned, void *stream);

/*
 * kda_chunk_fwd -- the chunked forward pass (all of the operation above).
 *
 * Kernel choice is made from the arguments, not from any global setting:
 *   dtype KDA_BF16 with d_k = d_v = 128: the tensor-core kernel (bf16 operands,
 *     fp32 accumulation and state) on thread-block clusters. It advances the state
 *     64 tokens (four bounded 16-token tiles) per serial step on tcgen05 tensor
 *     cores; the environment variable KDA_FWD_KERNEL=tc16 selects the earlier
 *     16-token-step mma.sync kernel instead (same results within rounding);
 *   any other supported case (KDA_F32, or 1 <= d_k, d_v <= 128): the fp32 SIMT
 *     kernel. Both compute the same chunked algebra.
 * Returns KDA_OK, KDA_ERR_INVALID_ARG (null required pointer, n_tok < 0,
 * n_seq < 0, n_heads <= 0, misaligned pointer), KDA_ERR_UNSUPPORTED (dtype or
 * d_k/d_v outside 1..128) or KDA_ERR_CUDA (launch failed; see kda_last_error).
 * n_seq = 0 or n_tok = 0 with all-empty sequences is valid (h_final = h0 is still
 * written when requested).
 */
kda_status kda_chunk_fwd(const void *q, const void *k, const void *v,
                         const float *gate_logits, const float *beta, const float *h0,
                         const int32_t *cu_seqlens, void *out, float *h_final,
                         int64_t n_tok, int32_t n_seq, int32_t n_heads, int32_t d_k,
                         int32_t d_v, kda_dtype dtype, void *stream);

/*
 * kda_chunk_fwd_simt -- the same operation forced onto the fp32 SIMT kernel
 * (fp32 FMA arithmetic throughout, bf16 or fp32 I/O). Same arguments, layout,
 * ownership and errors as kda_chunk_fwd. Used to cross-check the tensor-core
 * kernel and where bf16 operand rounding is not wanted.
 */
kda_status kda_chunk_fwd_simt(const void *q, const void *k, const void *v,
                              const float *gate_logits, const float *beta,
                              const float *h0, const int32_t *cu_seqlens, void *out,
                              float *h_final, int64_t n_tok, int32_t n_seq,
                              int32_t n_heads, int32_t d_k, int32_t d_v, kda_dtype dtype,
                              void *stream);

/*
 * kda_chunk_fwd_variant -- contrast variants of the forward pass, on the fp32 SIMT
 * kernel, for measuring what the bounded decay buys. They are not the method: the
 * pages replace the unbounded gate g = -softplus(a) with g = -5 sigmoid(a) precisely so
 * that the diagonal tile can be the dense products A = strict_lower(beta K~ K^^T),
 * P = lower(Q~ K^^T) with K^ = K e^-G, instead of a position-by-position computation
 * ("Architecture Analysis of Ultra-Long Context Sparse MoE Models", §2.1-2.2;
 * "Demystifying Trillion-Parameter MoE Models", Breakthrough 1 §1-2).
 *   gate_kind  KDA_GATE_BOUNDED: g = -5 sigmoid(a) (as kda_chunk_fwd);
 *              KDA_GATE_SOFTPLUS: g = -softplus(a) = -log(1 + e^a), unbounded below.
 *   diag_path  KDA_DIAG_DENSE: the dense tile above (as kda_chunk_fwd);
 *              KDA_DIAG_PAIRS: A_rj = beta_r sum_c k_rc k_jc e^{G_rc - G_jc} and
 *              P_rj = sum_c q_rc k_jc e^{G_rc - G_jc} for j <= r, one exponential per
 *              position pair and channel (finite for any decay).
 * With KDA_GATE_SOFTPLUS and KDA_DIAG_DENSE a chunk whose log-decay sums below about
 * -88 makes e^-G overflow fp32 and the outputs non-finite: the failure the bound
 * removes, reproduced on purpose. Other arguments, layout and errors as
 * kda_chunk_fwd, plus KDA_ERR_INVALID_ARG for an unknown gate_kind or diag_path.
 */
enum { KDA_GATE_BOUNDED = 0, KDA_GATE_SOFTPLUS = 1 };
enum { KDA_DIAG_DENSE = 0, KDA_DIAG_PAIRS = 1 };
kda_status kda_chunk_fwd_variant(const void *q, const void *k, const void *v,
                                 const float *gate_logits, const float *beta,
                                 const float *h0, const int32_t *cu_seqlens, void *out,
                                 float *h_final, int64_t n_tok, int32_t n_seq,
                                 int32_t n_heads, int32_t d_k, int32_t d_v, kda_dtype dtype,
                                 int32_t gate_kind, int32_t diag_path, void *stream);

/*
 * kda_gate_projection -- the gate logits from the layer input: a = x W^T + b, the
 * "projection(x)" inside the bounded gate g = -5 sigmoid(projection(x)) ("Architecture
 * Analysis of Ultra-Long Context Sparse MoE Models", §2.2; "From Numerical Stability to
 * Load Balancing", §2.2). Its output is kda_chunk_fwd's gate_logits.
 *   x            [n_tok, d_model] bf16, row-major
 *   weight       [n_out, d_model] bf16, row-major (a linear layer's weight; n_out is
 *                n_heads * d_k)
 *   bias         [n_out] float32, or NULL for none
 *   gate_logits  [n_tok, n_out] float32 (= [n_tok, n_heads, d_k]), fully overwritten
 * bf16 products accumulated in fp32 on the tensor cores (tcgen05). d_model must be a
 * multiple of 8; x, weight and gate_logits 16-byte aligned, bias 4-byte aligned;
 * gate_logits may not overlap an input. Asynchronous on `stream`; nothing is allocated.
 * Returns KDA_ERR_INVALID_ARG (NULL pointer, negative or zero size, misalignment,
 * overlap), KDA_ERR_UNSUPPORTED (d_model not a multiple of 8, n_tok >= 2^31) or
 * KDA_ERR_CUDA. A pipeline wait that gives up sets bit 1 of kda_read_device_flags.
 */
kda_status kda_gate_projection(const void *x, const void *weight, const float *bias,
                               float *gate_logits, int64_t n_tok, int32_t d_model,
                               int32_t n_out, void *stream);

/*
 * kda_gate_projection_out -- kda_gate_projection with the output type chosen: `out` is
 * [n_tok, n_out] of `out_dtype` (KDA_F32: as kda_gate_projection; KDA_BF16: the fp32 sum
 * plus bias rounded to the nearest bf16, ties to even -- half the output bytes, for
 * callers that keep activations in bf16; kda_chunk_fwd itself takes fp32 gate logits).
 * Same arguments, alignment and errors otherwise, plus KDA_ERR_UNSUPPORTED for another
 * out_dtype.
 */
kda_status kda_gate_projection_out(const void *x, const void *weight, const float *bias, void *out,
                                   kda_dtype out_dtype, int64_t n_tok, int32_t d_model,
                                   int32_t n_out, void *stream);

/*
 * kda_affine_combine -- combine step of the segment scan for one sequence split in
 * time (an addition of this library; the pages describe only the serial recurrence,
 * "From Numerical Stability to Load Balancing", §2.1, and this step follows from it).
 * Over any span of tokens the recurrence is affine in its start state, so a segment
 * maps S_start to S_end = M S_start + B, where M (d_k x d_k) is the segment's end state
 * when run (kda_chunk_fwd) from h0 = I with v = 0 and B (d_k x d_v) its end state from
 * h0 = 0. This call computes, per head, S_out = M S_in + B in fp32.
 * Layout: M [n_heads][d_k][d_k]; S_in, B, S_out [n_heads][d_k][d_v]; row-major fp32 in
 * device memory, 4-byte aligned, caller-owned; S_out may not alias an input. Queued on
 * `stream`. Returns KDA_ERR_INVALID_ARG (NULL or misaligned pointer, aliasing,
 * non-positive size), KDA_ERR_UNSUPPORTED (d_k or d_v above 128) or KDA_ERR_CUDA.
 */
kda_status kda_affine_combine(const float *M, const float *S_in, const float *B, float *S_out,
                              int32_t n_heads, int32_t d_k, int32_t d_v, void *stream);

/*
 * kda_decode_step -- one recurrent decode step: each of n_seq sequences advances by
 * one token, from its state to the next, per head:
 *   S' = Diag(exp g) S,  g = -5 sigmoid(a);  u = beta (v - S'^T k);
 *   S <- S' + k u^T;  o = d_k^-1/2 S^T q   (the state after the write)
 * -- the operation above for a single token ("From Numerical Stability to Load
 * Balancing", §2.1-2.2), i.e. what kda_chunk_fwd computes for a one-token sequence
 * started from `state`. Pairs with kda_chunk_fwd for generation: the prompt's h_final
 * is the first decode step's state.
 * Layout (contiguous, row-major, caller-owned device memory):
 *   q, k          [n_seq, n_heads, d_k]        dtype
 *   v             [n_seq, n_heads, d_v]        dtype
 *   gate_logits   [n_seq, n_heads, d_k]        float32
 *   beta          [n_seq, n_heads]             float32
 *   state         [n_seq, n_heads, d_k, d_v]   float32, read and overwritten in place
 *   out           [n_seq, n_heads, d_v]        dtype
 * q, k, v and out must be aligned to their element size, gate_logits, beta and state
 * to 4 bytes; state and out may not overlap each other or any input. Any 1 <= d_k,
 * d_v <= 128. Asynchronous on `stream`; nothing is allocated. Returns
 * KDA_ERR_INVALID_ARG (NULL pointer, negative or zero size, misalignment, overlap),
 * KDA_ERR_UNSUPPORTED (dtype, or d_k/d_v above 128) or KDA_ERR_CUDA; n_seq = 0 is a
 * valid no-op.
 */
kda_status kda_decode_step(const void *q, const void *k, const void *v,
                           const float *gate_logits, const float *beta, float *state,
                           void *out, int32_t n_seq, int32_t n_heads, int32_t d_k,
                           int32_t d_v, kda_dtype dtype, void *stream);

/*
 * kda_chunk_bwd -- backward pass of kda_chunk_fwd: the gradients of
 *   L = <dout, out> + <dh_final, h_final>
 * with respect to q, k, v, the gate logits, beta and h0 (the vector-Jacobian product of
 * the operation above; the pages define the forward only -- "From Numerical Stability
 * to Load Balancing", §2.1-2.2 -- and this is its derivative, taken through the same
 * 16-token chunked form).
 * Inputs: q, k, v, gate_logits, beta, h0 (NULL = zero start), cu_seqlens exactly as
 * for kda_chunk_fwd; dout [n_tok, n_heads, d_v] in dtype; dh_final [n_seq, n_heads,
 * d_k, d_v] float32 or NULL (zero).
 * Outputs (caller-owned, fully overwritten): dq, dk [n_tok, n_heads, d_k] and dv
 * [n_tok, n_heads, d_v] in dtype; dgate_logits [n_tok, n_heads, d_k] and dbeta
 * [n_tok, n_heads] float32; dh0 [n_seq, n_heads, d_k, d_v] float32, or NULL to skip.
 * workspace: caller-owned device memory of at least kda_chunk_bwd_workspace_bytes()
 * bytes, 4-byte aligned, contents ignored on entry (it receives the state at the start
 * and the state gradient at the end of every chunk). Arithmetic: fp32 accumulation
 * throughout; for KDA_BF16 with d_k = d_v = 128, and the workspace, q, k, v,
 * gate_logits and dout 16-byte aligned, the products take bf16 operands on the tensor
 * cores (the chunk products of the state-independent part as split bf16 high and low
 * parts), otherwise fp32 FMA. The result is deterministic: the same call gives the same
 * bits. Alignment as for kda_chunk_fwd for the inputs; outputs aligned to their element
 * size.
 * No output or the workspace may overlap an input or another output. Asynchronous on
 * `stream`; nothing is allocated. Errors as for kda_chunk_fwd, plus
 * KDA_ERR_INVALID_ARG for a missing gradient buffer, overlap, or a NULL or too small
 * workspace.
 */
size_t kda_chunk_bwd_workspace_bytes(int64_t n_tok, int32_t n_seq, int32_t n_heads,
                                     int32_t d_k, int32_t d_v);
kda_status kda_chunk_bwd(const void *q, const void *k, const void *v,
                         const float *gate_logits, const float *beta, const float *h0,
                         const int32_t *cu_seqlens, const void *dout, const float *dh_final,
                         void *dq, void *dk, void *dv, float *dgate_logits, float *dbeta,
                         float *dh0, void *workspace, size_t workspace_bytes,
                         int64_t n_tok, int32_t n_seq, int32_t n_heads, int32_t d_k,
                         int32_t d_v, kda_dtype dtype, void *stream);

/*
 * kda_bwd_timing_start / kda_bwd_timing_read -- device time of each kernel of the
 * backward pass, for measurement (an addition of this library: the pages have no
 * counterpart). After kda_bwd_timing_start(capacity) the next `capacity` calls of
 * kda_chunk_bwd or kda_chunk_bwd_static_scratch record CUDA events on their stream around
 * their kernels: ms[0] the state-independent chunk products, ms[1] the forward serial
 * pass, ms[2] the reverse serial pass, ms[3] the local gradients. The tensor-core path
 * runs both serial passes in one launch: its time is in ms[1] and ms[2] is about 0.
 * Recording adds no synchronisation. kda_bwd_timing_read waits for those events, writes the milliseconds of
 * each kernel summed over the recorded calls to ms[0..3] (host array of 4) and the number
 * of recorded calls to *calls (host), and stops recording. One recording at a time per
 * process; a new start discards the previous one. Errors: KDA_ERR_INVALID_ARG for
 * capacity outside [1, 1024] or a NULL pointer; KDA_ERR_CUDA when an event cannot be
 * created or waited for.
 */
kda_status kda_bwd_timing_start(int capacity);
kda_status kda_bwd_timing_read(float *ms, int *calls);

/*
 * kda_chunk_bwd_static_scratch -- kda_chunk_bwd without a caller workspace and without
 * any allocation: the checkpoints go to a fixed scratch array of
 * KDA_STATIC_SCRATCH_BYTES compiled into the library (static device memory of the
 * loaded module, one per device, its address looked up once per device). An addition
 * of this library: the pages have no counterpart.
 * Same arguments, layout, results and errors as kda_chunk_bwd minus the workspace;
 * problems with kda_chunk_bwd_workspace_bytes() > KDA_STATIC_SCRATCH_BYTES return
 * KDA_ERR_UNSUPPORTED before any device work. No part of the scratch has to start at
 * zero: every slot a call reads, that call has written first. The scratch is shared by
 * every call on the device: two calls that may run at the same time (different streams,
 * or host threads whose streams are not ordered) race on it and both results are
 * undefined -- order them on one stream. The scratch used is the one of the calling
 * thread's CURRENT device (cudaGetDevice): every pointer and `stream` must belong to that
 * device. The argument and size checks (those of kda_chunk_bwd, then the scratch size)
 * all run before any device work.
 */
#define KDA_STATIC_SCRATCH_BYTES ((size_t)64 << 20)
kda_status kda_chunk_bwd_static_scratch(const void *q, const void *k, const void *v,
                                        const float *gate_logits, const float *beta,
                                        const float *h0, const int32_t *cu_seqlens,
                                        const void *dout, const float *dh_final, void *dq,
                                        void *dk, void *dv, float *dgate_logits,
                                        float *dbeta, float *dh0, int64_t n_tok,
                                        int32_t n_seq, int32_t n_heads, int32_t d_k,
                                        int32_t d_v, kda_dtype dtype, void *stream);

/*
 * kda_chunk_fwd_gated -- the forward pass fed directly by the gate projection
 * ("Architecture Analysis of Ultra-Long Context Sparse MoE Models", §2.2: the gate is
 * sigmoid(projection(x)); "From Numerical Stability to Load Balancing", §2.2): the result of
 * kda_gate_projection(x, w_gate, b_gate) followed by kda_chunk_fwd, bit for bit, without
 * the whole gate-logit tensor ever existing. The tokens are cut into segments of about
 * `segment_tokens` (each cut a multiple of 64 tokens after the start of its sequence);
 * per segment, the segment's gate logits are computed into one workspace slot sized to
 * stay in L2 and consumed at once by the segment's forward pieces, and the state of a
 * sequence cut by a segment boundary is carried to its next piece in fp32 through the
 * workspace.
 *   x          [n_tok, d_model] bf16, device, 16-byte aligned; d_model % 8 == 0
 *   w_gate     [n_heads * d_k, d_model] bf16 (row h * d_k + c = head h, key channel c)
 *   b_gate     [n_heads * d_k] fp32 or NULL
 *   q .. h_final, cu_seqlens, n_tok .. d_v, stream: as kda_chunk_fwd (bf16 only)
 *   host_cu_seqlens  the same offsets in host memory (for the segment plan)
 *   workspace  device memory, 256-byte aligned, at least
 *              kda_chunk_fwd_gated_workspace_bytes(n_seq, n_heads, d_k, d_v, segment_tokens)
 *              bytes; owned by the caller, nothing in it has to be initialised
 *   segment_tokens  >= 64; 4096 keeps a slot at 64 MiB for n_heads * d_k = 4096
 * Runs on `stream` (current device must own every pointer and the stream); allocates no
 * memory; launches per segment one GEMM and one forward kernel per piece, plus one small
 * kernel per 64 segments. Errors: as kda_chunk_fwd and kda_gate_projection, plus
 * KDA_ERR_UNSUPPORTED for a dtype other than KDA_BF16, KDA_ERR_INVALID_ARG for
 * segment_tokens < 64, a missing or misaligned workspace or an invalid host_cu_seqlens.
 */
size_t kda_chunk_fwd_gated_workspace_bytes(int32_t n_seq, int32_t n_heads, int32_t d_k,
                                           int32_t d_v, int32_t segment_tokens);
kda_status kda_chunk_fwd_gated(const void *x, const void *w_gate, const float *b_gate,
                               int32_t d_model, const void *q, const void *k, const void *v,
                               const float *beta, const float *h0, const int32_t *cu_seqlens,
                               const int32_t *host_cu_seqlens, void *out, float *h_final,
                               void *workspace, size_t workspace_bytes, int64_t n_tok,
                               int32_t n_seq, int32_t n_heads, int32_t d_k, int32_t d_v,
                               int32_t segment_tokens, kda_dtype dtype, void *stream);

/*
 * kda_chunk_fwd_from_host -- end-to-end variant for callers whose inputs live in
 * host memory. Copies the inputs (host_*, preferably pinned) into the caller's
 * device buffers (dev_*) with one cudaMemcpyAsync each on `stream`, runs
 * kda_chunk_fwd on them, and copies out (and h_final when host_h_final is not
 * NULL) back to host memory on the same stream. cu_seqlens is given on the host
 * (host_cu_seqlens, int32 [n_seq + 1]) and copied to dev_cu_seqlens. host_h0 /
 * dev_h0 may both be NULL (zero start state); dev_h_final may be NULL only when
 * host_h_final is NULL. Nothing is allocated. The call returns after queuing; the
 * host buffers must stay valid until the stream reaches the last copy. Errors as
 * for kda_chunk_fwd, plus KDA_ERR_CUDA when a copy cannot be queued.
 */
kda_status kda_chunk_fwd_from_host(
    const void *host_q, const void *host_k, const void *host_v,
    const float *host_gate_logits, const float *host_beta, const float *host_h0,
    const int32_t *host_cu_seqlens, void *host_out, float *host_h_final,
    void *dev_q, void *dev_k, void *dev_v, float *dev_gate_logits, float *dev_beta,
    float *dev_h0, int32_t *dev_cu_seqlens, void *dev_out, float *dev_h_final,
    int64_t n_tok, int32_t n_seq, int32_t n_heads, int32_t d_k, int32_t d_v,
    kda_dtype dtype, void *stream);

/*
 * kda_chunk_fwd_from_host_pipelined -- kda_chunk_fwd_from_host with the copies overlapped
 * with the computation. The token range is cut into at most n_segments segments of about
 * n_tok / n_segments tokens (1 <= n_segments <= 64); segment i's inputs are copied in on
 * one stream while segment i-1 is computed on `stream` and segment i-2's outputs (and
 * the final states of the sequences that end in it) are copied out on another. Each cut
 * lies a multiple of 16 tokens after the start of the sequence that holds it, so every
 * piece keeps its sequence's 16-token chunk grid, and a cut sequence's state passes from
 * one piece to the next in fp32 (chunks run serially through the state recurrence, "From
 * Numerical Stability to Load Balancing", §2.1, so a sequence may be continued from any
 * chunk boundary given the state there, as kda_chunk_fwd's h0 already allows): out
 * and h_final equal those of kda_chunk_fwd on the whole input bit for bit (the same
 * kernels run on the same chunks). Cuts are made only when a token's q/k/v/gate rows are
 * whole multiples of 16 bytes (true for d_k = d_v = 128). When the plan has one segment
 * (n_segments = 1, too few tokens to cut, or rows that cannot be cut) the call is
 * kda_chunk_fwd_from_host: one stream, no overlap, the workspace unused.
 *   host_*, dev_*  as for kda_chunk_fwd_from_host (host buffers preferably pinned: a
 *                  pageable one makes its copy wait for the caller's earlier work);
 *                  dev_cu_seqlens receives host_cu_seqlens.
 *   dev_workspace  device memory, 256-byte aligned, at least
 *                  kda_chunk_fwd_pipelined_workspace_bytes(n_seq, n_heads, d_k, d_v,
 *                  n_segments) bytes: two carried states and the pieces' sequence
 *                  offsets. Owned by the caller; nothing in it has to be initialised.
 * The first call from a host thread on a device creates two streams and three events for
 * that (thread, device); later calls reuse them, and they are released with the CUDA
 * context. The current device (cudaGetDevice) must own every device pointer and
 * `stream`. The call allocates no device memory and launches one small kernel (the
 * pieces' offsets) besides the forward kernels. `stream` waits for the last copy before its next work. The host
 * buffers must stay valid until then. Errors as for kda_chunk_fwd_from_host, plus
 * KDA_ERR_INVALID_ARG for n_segments outside [1, 64], a too-small or misaligned
 * workspace, or a host_cu_seqlens that does not start at 0, decreases, or does not end
 * at n_tok.
 */
kda_status kda_chunk_fwd_from_host_pipelined(
    const void *host_q, const void *host_k, const void *host_v,
    const float *host_gate_logits, const float *host_beta, const float *host_h0,
    const int32_t *host_cu_seqlens, void *host_out, float *host_h_final,
    void *dev_q, void *dev_k, void *dev_v, float *dev_gate_logits, float *dev_beta,
    float *dev_h0, int32_t *dev_cu_seqlens, void *dev_out, float *dev_h_final,
    void *dev_workspace, size_t workspace_bytes, int64_t n_tok, int32_t n_seq,
    int32_t n_heads, int32_t d_k, int32_t d_v, int32_t n_segments, kda_dtype dtype,
    void *stream);

/* Workspace bytes of kda_chunk_fwd_from_host_pipelined; 0 for invalid arguments. */
size_t kda_chunk_fwd_pipelined_workspace_bytes(int32_t n_seq, int32_t n_heads, int32_t d_k,
                                               int32_t d_v, int32_t n_segments);

/*
 * kda_chunk_fwd_pipeline_plan -- the pieces kda_chunk_fwd_from_host_pipelined runs, on the
 * host only (no device work). Piece j is 7 int64 at pieces[7 j]: token range [t0, t1),
 * sequence range [n0, n1), h0_carried (1: starts from the state carried from the previous
 * piece of its sequence, 0: from h0), hf_carried (1: its final state is carried to the next
 * piece, 0: it is the sequence's h_final), segment index. Returns the number of pieces
 * (pieces may be NULL to count them), or -1 for an invalid host_cu_seqlens, n_segments
 * outside [1, 64], or a capacity below the count.
 */
int32_t kda_chunk_fwd_pipeline_plan(const int32_t *host_cu_seqlens, int32_t n_seq,
                                    int64_t n_tok, int32_t n_segments, int64_t *pieces,
                                    int32_t capacity);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_H_ */
