// kda_scan.cu -- the combine step of the segment scan for a sequence split in time.
//
// Over any span of tokens the recurrence is affine in its start state: the decay
// Diag(exp g_t) and the delta write S + beta k (v - S^T k)^T = (I - beta k k^T) S +
// beta k v^T are both affine in S, and so is their composition. A segment therefore maps
// S_start to S_end = M S_start + B, where M (d_k x d_k) is the segment run from
// S_start = I with v = 0 and B (d_k x d_v) the segment run from S_start = 0 -- both
// ordinary forward passes. Chaining S_j = M_{j-1} S_{j-1} + B_{j-1} over the segments
// gives every segment's true start state, from which the segments replay in parallel.
// The serial state recurrence itself is the one of "From Numerical Stability to Load
// Balancing", §2.1.
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int T = 32;  // output tile edge; each thread computes 4 rows of one column

// O[h] = M[h] S[h] + B[h], fp32; grid (ceil(dv/T), ceil(dk/T), H), block (T, 8)
__global__ void __launch_bounds__(T * 8)
    affine_combine_kernel(const float *__restrict__ M, const float *__restrict__ S,
                          const float *__restrict__ B, float *__restrict__ O, int dk, int dv) {
    __shared__ float Ms[T][T + 1], Ss[T][T + 1];
    const int h = blockIdx.z;
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int col = blockIdx.x * T + tx, row0 = blockIdx.y * T;
    const float *Mh = M + (size_t)h * dk * dk;
    const float *Sh = S + (size_t)h * dk * dv;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k0 = 0; k0 < dk; k0 += T) {
        for (int i = ty; i < T; i += 8) {
            const int r = row0 + i, kk = k0 + tx;
            Ms[i][tx] = (r < dk && kk < dk) ? Mh[(size_t)r * dk + kk] : 0.f;
            const int kr = k0 + i;
            Ss[i][tx] = (kr < dk && col < dv) ? Sh[(size_t)kr * dv + col] : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < T; ++kk) {
            const float s = Ss[kk][tx];
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[j] = fmaf(Ms[ty + 8 * j][kk], s, acc[j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int r = row0 + ty + 8 * j;
        if (r < dk && col < dv) {
            const size_t o = (size_t)h * dk * dv + (size_t)r * dv + col;
            O[o] = acc[j] + B[o];
        }
    }
}

}  // namespace

cudaError_t launch_affine_combine(const float *M, const float *S, const float *B, float *O,
                                  int n_heads, int dk, int dv, cudaStream_t stream) {
    const dim3 grid((unsigned)((dv + T - 1) / T), (unsigned)((dk + T - 1) / T), (unsigned)n_heads);
    affine_combine_kernel<<<grid, dim3(T, 8), 0, stream>>>(M, S, B, O, dk, dv);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

}  // namespace kda
