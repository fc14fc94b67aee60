// kda_decode.cu -- one recurrent decode step: every sequence advances by one token.
//
// Per sequence and head, with the state S in R^{d_k x d_v} (fp32, updated in place):
//   gamma = exp(g), g = -5 sigmoid(a)                      (per key channel)
//   S'    = Diag(gamma) S
//   u     = beta (v - S'^T k)
//   S    <- S' + k u^T
//   o     = d_k^-1/2 S^T q = d_k^-1/2 (S'^T q + (q . k) u)
// This is the token-by-token form of the recurrence whose state forgets through the
// decay and writes key-value outer products ("From Numerical Stability to Load
// Balancing", §2.1), with the bounded gate of the same page, §2.2, and "Demystifying
// Trillion-Parameter MoE Models", Breakthrough 1 §2.
//
// Column j of S evolves on its own: before it is rewritten it contributes only the two
// dot products (k gamma)^T S[:, j] and (q gamma)^T S[:, j]. The state is therefore read
// once and written once, and the step is bound by HBM bandwidth: 8 d_k d_v bytes of state
// traffic per sequence and head against ~4 d_k d_v flops.
//
// One CTA of 256 threads per (sequence, head). Thread t owns column j = t mod 128 over
// rows [64 h, 64 h + 64), h = t / 128, and keeps those 64 values in registers between
// the read and the write; a warp reads or writes 32 consecutive floats of one row (one
// 128-byte line) per access, and each thread has its 64 loads in flight at once.
#include <cuda_bf16.h>

#include <cmath>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kCols = 128;        // columns (value channels) covered by a CTA
constexpr int kRows = 64;         // rows (key channels) per thread
constexpr int kHalves = kThreads / kCols;
static_assert(kHalves * kRows == 128, "two row halves cover d_k <= 128");

__device__ __forceinline__ float load_elem(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float load_elem(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void store_elem(float *p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void store_elem(__nv_bfloat16 *p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
    decode_step_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                       const float *__restrict__ a, const float *__restrict__ beta,
                       float *__restrict__ state, T *__restrict__ out, int dk, int dv,
                       float scale) {
    __shared__ float gam[kCols], kgam[kCols], qgam[kCols], kraw[kCols];
    __shared__ float part[kHalves][2][kCols];  // [row half][k-dot, q-dot][column]
    __shared__ float ucol[kCols];
    __shared__ float qk_warp[kCols / 32];
    const int sh = blockIdx.x;  // sequence * n_heads + head
    const int t = threadIdx.x, j = t % kCols, half = t / kCols;
    const size_t kv = (size_t)sh * dk;  // this (sequence, head)'s key-side vectors

    // per key channel c < d_k: gamma_c, k_c gamma_c, q_c gamma_c, k_c (zero past d_k),
    // and the warp partial sums of q . k
    if (t < kCols) {
        float kc = 0.f, qc = 0.f, g = 1.f;
        if (t < dk) {
            kc = load_elem(k, kv + t);
            qc = load_elem(q, kv + t);
            const float sig = 1.f / (1.f + expf(-a[kv + t]));
            g = expf(kGMin * sig);
        }
        gam[t] = g;
        kraw[t] = kc;
        kgam[t] = kc * g;
        qgam[t] = qc * g;
        float qk = qc * kc;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) qk += __shfl_xor_sync(0xffffffffu, qk, o);
        if ((t & 31) == 0) qk_warp[t >> 5] = qk;
    }
    __syncthreads();

    // read this thread's slice of column j once; its two partial dot products
    float *S = state + (size_t)sh * dk * dv;
    const int r0 = half * kRows;
    float s[kRows];
    float pk = 0.f, pq = 0.f;
    if (j < dv) {
#pragma unroll
        for (int i = 0; i < kRows; ++i) s[i] = r0 + i < dk ? S[(size_t)(r0 + i) * dv + j] : 0.f;
#pragma unroll
        for (int i = 0; i < kRows; ++i) {  // rows past d_k hold 0 and have zero weights
            pk = fmaf(kgam[r0 + i], s[i], pk);
            pq = fmaf(qgam[r0 + i], s[i], pq);
        }
    }
    part[half][0][j] = pk;
    part[half][1][j] = pq;
    __syncthreads();

    // u_j and o_j
    if (half == 0 && j < dv) {
        const float qk = qk_warp[0] + qk_warp[1] + qk_warp[2] + qk_warp[3];
        const size_t vo = (size_t)sh * dv + j;
        const float u = beta[sh] * (load_elem(v, vo) - (part[0][0][j] + part[1][0][j]));
        ucol[j] = u;
        store_elem(out, vo, scale * (part[0][1][j] + part[1][1][j] + qk * u));
    }
    __syncthreads();

    // write the column back: S = Diag(gamma) S + k u^T
    if (j < dv) {
        const float u = ucol[j];
#pragma unroll
        for (int i = 0; i < kRows; ++i)
            if (r0 + i < dk) S[(size_t)(r0 + i) * dv + j] = fmaf(gam[r0 + i], s[i], kraw[r0 + i] * u);
    }
}

// The same step with 16-byte state accesses (state 16-byte aligned, d_v a multiple of 4):
// thread t owns columns [4 (t mod 32), +4) over rows [16 (t / 32), +16) -- a warp reads or
// writes four whole 128-byte lines of one row block per access -- and the partial dot
// products of the 8 row blocks are added in shared memory.
template <typename T>
__global__ void __launch_bounds__(kThreads, 2)
    decode_step_v4_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                          const float *__restrict__ a, const float *__restrict__ beta,
                          float *__restrict__ state, T *__restrict__ out, int dk, int dv,
                          float scale) {
    constexpr int RB = kThreads / 32;  // row blocks of 16 rows
    __shared__ float gam[kCols], kgam[kCols], qgam[kCols], kraw[kCols];
    __shared__ __align__(16) float part[RB][2][kCols];  // [row block][k-dot, q-dot][column]
    __shared__ __align__(16) float ucol[kCols];
    __shared__ float qk_warp[kCols / 32];
    const int sh = blockIdx.x;
    const int t = threadIdx.x, c4 = 4 * (t & 31), rb = t >> 5, r0 = 16 * rb;
    const size_t kv = (size_t)sh * dk;
    const int dv4 = dv >> 2;
    // this thread's 16 x 4 block of the state (rows r0.., columns c4..), read once, before the
    // gate's loads; nrow rows of it exist
    float4 *S4 = reinterpret_cast<float4 *>(state + (size_t)sh * dk * dv) + (size_t)r0 * dv4 + (c4 >> 2);
    const int nrow = c4 < dv ? min(16, dk - r0) : 0;
    float4 s[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        s[i] = i < nrow ? S4[i * dv4] : make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < kCols) {
        float kc = 0.f, qc = 0.f, g = 1.f;
        if (t < dk) {
            kc = load_elem(k, kv + t);
            qc = load_elem(q, kv + t);
            const float sig = 1.f / (1.f + expf(-a[kv + t]));
            g = expf(kGMin * sig);
        }
        gam[t] = g;
        kraw[t] = kc;
        kgam[t] = kc * g;
        qgam[t] = qc * g;
        float qk = qc * kc;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) qk += __shfl_xor_sync(0xffffffffu, qk, o);
        if ((t & 31) == 0) qk_warp[t >> 5] = qk;
    }
    __syncthreads();
    {  // partial dot products of the 4 columns over this row block
        float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float kg = kgam[r0 + i], qg = qgam[r0 + i];  // 0 past d_k
            pk.x = fmaf(kg, s[i].x, pk.x); pk.y = fmaf(kg, s[i].y, pk.y);
            pk.z = fmaf(kg, s[i].z, pk.z); pk.w = fmaf(kg, s[i].w, pk.w);
            pq.x = fmaf(qg, s[i].x, pq.x); pq.y = fmaf(qg, s[i].y, pq.y);
            pq.z = fmaf(qg, s[i].z, pq.z); pq.w = fmaf(qg, s[i].w, pq.w);
        }
        *reinterpret_cast<float4 *>(&part[rb][0][c4]) = pk;
        *reinterpret_cast<float4 *>(&part[rb][1][c4]) = pq;
    }
    __syncthreads();
    if (t < kCols && t < dv) {  // u_j and o_j, column j = t
        float pk = 0.f, pq = 0.f;
#pragma unroll
        for (int b = 0; b < RB; ++b) {
            pk += part[b][0][t];
            pq += part[b][1][t];
        }
        const float qk = qk_warp[0] + qk_warp[1] + qk_warp[2] + qk_warp[3];
        const size_t vo = (size_t)sh * dv + t;
        const float u = beta[sh] * (load_elem(v, vo) - pk);
        ucol[t] = u;
        store_elem(out, vo, scale * (pq + qk * u));
    }
    __syncthreads();
    if (nrow > 0) {  // write the block back: S = Diag(gamma) S + k u^T
        const float4 u = *reinterpret_cast<const float4 *>(&ucol[c4]);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (i < nrow) {
                const float g = gam[r0 + i], kr = kraw[r0 + i];
                S4[i * dv4] = make_float4(fmaf(g, s[i].x, kr * u.x), fmaf(g, s[i].y, kr * u.y),
                                          fmaf(g, s[i].z, kr * u.z), fmaf(g, s[i].w, kr * u.w));
            }
        }
    }
}

}  // namespace

cudaError_t launch_decode_step(const DecodeArgs &p, cudaStream_t stream) {
    const unsigned grid = (unsigned)((int64_t)p.n_seq * p.n_heads);
    if (grid == 0) return cudaSuccess;
    const float scale = 1.0f / std::sqrt((float)p.d_k);
    const bool v4 = (p.d_v & 3) == 0 && (reinterpret_cast<uintptr_t>(p.state) & 15u) == 0;
    if (v4) {
        if (p.bf16) {
            using T = __nv_bfloat16;
            decode_step_v4_kernel<T><<<grid, kThreads, 0, stream>>>(
                static_cast<const T *>(p.q), static_cast<const T *>(p.k), static_cast<const T *>(p.v),
                p.a, p.beta, p.state, static_cast<T *>(p.out), p.d_k, p.d_v, scale);
        } else {
            decode_step_v4_kernel<float><<<grid, kThreads, 0, stream>>>(
                static_cast<const float *>(p.q), static_cast<const float *>(p.k),
                static_cast<const float *>(p.v), p.a, p.beta, p.state, static_cast<float *>(p.out),
                p.d_k, p.d_v, scale);
        }
    } else if (p.bf16) {
        using T = __nv_bfloat16;
        decode_step_kernel<T><<<grid, kThreads, 0, stream>>>(
            static_cast<const T *>(p.q), static_cast<const T *>(p.k), static_cast<const T *>(p.v),
            p.a, p.beta, p.state, static_cast<T *>(p.out), p.d_k, p.d_v, scale);
    } else {
        decode_step_kernel<float><<<grid, kThreads, 0, stream>>>(
            static_cast<const float *>(p.q), static_cast<const float *>(p.k),
            static_cast<const float *>(p.v), p.a, p.beta, p.state, static_cast<float *>(p.out),
            p.d_k, p.d_v, scale);
    }
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

}  // namespace kda
