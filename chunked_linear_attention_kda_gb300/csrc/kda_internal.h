// Internal declarations shared by the CUDA translation units of the library.
// Not part of the C ABI (that is include/kda.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

// Tile length in tokens and the lower bound of the log-decay. Both are fixed by
// the method: a 16-token tile is co-designed with g_min = -5 so that every
// in-tile factor exp(+-G) stays within exp(+-80) ("From Numerical Stability to
// Load Balancing", §2.2-2.3).
constexpr int kChunk = 16;
constexpr float kGMin = -5.0f;

struct FwdArgs {
    const void *q, *k, *v;
    const float *a, *beta, *h0;
    const int32_t *cu_seqlens;
    void *out;
    float *h_final;
    int64_t n_tok;
    int32_t n_seq, n_heads, d_k, d_v;
    bool bf16;  // q/k/v/out element type: bf16 when true, fp32 otherwise
};

// Each returns cudaSuccess or the launch error; all work is queued on `stream`.
cudaError_t launch_simt(const FwdArgs &args, cudaStream_t stream);
// The SIMT kernel's contrast variants: gate 0 = -5 sigmoid(a), 1 = -softplus(a); pair =
// position-pair diagonal tile instead of the dense K~ K^^T, Q~ K^^T products.
cudaError_t launch_simt_variant(const FwdArgs &args, int gate, bool pair, cudaStream_t stream);
cudaError_t launch_tc(const FwdArgs &args, cudaStream_t stream);
// The 64-token-step tcgen05 kernel (kda_fwd64.cu) and its own status word (bit 3: a
// pipeline wait gave up; reading synchronises stream).
cudaError_t launch_fwd64(const FwdArgs &args, cudaStream_t stream);
bool fwd64_supported(const FwdArgs &args);
cudaError_t read_fwd64_flags(unsigned int *flags, bool reset, cudaStream_t stream);

// True when the tensor-core kernel handles this shape and dtype.
bool tc_supported(const FwdArgs &args);

// Launches a one-thread kernel whose pipeline wait can never complete; it gives up
// after limit_cycles, sets bit 0 of the status word and writes 1 to *d_returned.
cudaError_t bounded_wait_selftest(long long limit_cycles, int *d_returned, cudaStream_t stream);

// Per head, O = M S + B in fp32 (M: d_k x d_k; S, B, O: d_k x d_v; row-major, heads
// contiguous): the combine step of the segment scan.
cudaError_t launch_affine_combine(const float *M, const float *S, const float *B, float *O,
                                  int n_heads, int d_k, int d_v, cudaStream_t stream);

// One recurrent decode step: q, k, a [n_seq, H, d_k]; v, out [n_seq, H, d_v]; beta
// [n_seq, H]; state [n_seq, H, d_k, d_v] fp32, read and overwritten.
struct DecodeArgs {
    const void *q, *k, *v;
    const float *a, *beta;
    float *state;
    void *out;
    int32_t n_seq, n_heads, d_k, d_v;
    bool bf16;  // q/k/v/out element type: bf16 when true, fp32 otherwise
};
cudaError_t launch_decode_step(const DecodeArgs &args, cudaStream_t stream);

// Backward pass: inputs as FwdArgs plus dout [n_tok, H, d_v] (dtype) and dh_final
// (nullable); gradients dq, dk [n_tok, H, d_k], dv [n_tok, H, d_v] (dtype), da [n_tok,
// H, d_k], dbeta [n_tok, H] (fp32), dh0 (nullable); workspace of bwd_workspace_bytes().
struct BwdArgs {
    const void *q, *k, *v, *dout;
    const float *a, *beta, *h0, *dh_final;
    const int32_t *cu_seqlens;
    void *dq, *dk, *dv;
    float *da, *dbeta, *dh0, *workspace;
    int64_t n_tok;
    int32_t n_seq, n_heads, d_k, d_v;
    bool bf16;
};
size_t bwd_slots(int64_t n_tok, int32_t n_seq);
size_t bwd_workspace_bytes(int64_t n_tok, int32_t n_seq, int32_t n_heads, int32_t d_k,
                           int32_t d_v);
cudaError_t launch_bwd(const BwdArgs &args, cudaStream_t stream);

// Size of the library's fixed backward scratch array (kda_bwd_static.cu) and the lookup
// of its device address on the current device (cached per device).
constexpr size_t kStaticScratchBytes = (size_t)64 << 20;
cudaError_t static_scratch(void **ptr);

// Gate projection a[M, N] = x[M, K] W[N, K]^T (+ b[N]): bf16 x and W, fp32 a and b
// (tcgen05 GEMM, kda_gemm.cu). K % 8 == 0, x, W and a 16-byte aligned.
cudaError_t launch_gate_proj(const void *x, const void *w, const float *bias, float *out, int M,
                             int N, int K, cudaStream_t stream);
// the same with bf16 output (the fp32 sum + bias rounded to nearest even)
cudaError_t launch_gate_proj_bf16(const void *x, const void *w, const float *bias, void *out, int M,
                                  int N, int K, cudaStream_t stream);
// The GEMM's own status word (bit 1: a pipeline wait gave up); synchronises stream.
cudaError_t read_gemm_flags(unsigned int *flags, bool reset, cudaStream_t stream);
// The backward serial passes' status word (bit 2); synchronises stream.
cudaError_t read_bwd_flags(unsigned int *flags, bool reset, cudaStream_t stream);
// Per-kernel event timing of the next `capacity` backward calls; the read returns the
// summed milliseconds of the four kernels and the number of calls recorded, and stops.
cudaError_t bwd_timing_start(int capacity);
cudaError_t bwd_timing_read(float ms[4], int *calls);

// Layout checks of cu_seqlens on the device (status[0]: bit 0 cu[0] != 0, bit 1 a
// decrease, bit 2 cu[n_seq] != n_tok; status[1]: first offending index) and a count of
// non-finite elements added into *count (kda_check.cu).
cudaError_t launch_validate_cu(const int32_t *cu, int32_t n_seq, int64_t n_tok, int32_t *status,
                               cudaStream_t stream);
cudaError_t launch_count_nonfinite(const void *x, int64_t n, bool bf16, unsigned long long *count,
                                   cudaStream_t stream);

// Copies (and optionally clears) the device-side status word; synchronises stream.
cudaError_t read_device_flags(unsigned int *flags, bool reset, cudaStream_t stream);

// Adds n to the process-wide kernel launch counter (kda_kernel_launch_count).
void count_launches(uint64_t n);

}  // namespace kda
