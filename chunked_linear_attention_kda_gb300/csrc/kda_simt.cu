// kda_simt.cu -- fp32 SIMT kernel for the chunked KDA forward pass.
//
// One CTA per (sequence, head) walks its chunks of 16 tokens in order; the state
// S (d_k x d_v, fp32) lives in shared memory. Every product is an fp32 FMA loop,
// so this kernel is the precise path (fp32 workloads, any d_k, d_v <= 128) and a
// cross-check for the tensor-core kernel. Per chunk of L <= 16 tokens, with rows
// past L acting as q = k = v = 0, beta = 0, g = 0:
//
//   g = -5 sigmoid(a); G = in-chunk inclusive cumsum of g   (bounded gate:
//       "Demystifying Trillion-Parameter MoE Models", Breakthrough 1 §2)
//   Q~ = Q e^G, K~ = K e^G, K^ = K e^-G, K' = K e^(G_L - G)  (|G| <= 80:
//       "From Numerical Stability to Load Balancing", §2.2)
//   A = strict_lower(beta K~ K^^T), TB = (I + A)^-1 diag(beta)
//   W = TB K~, U~ = TB V, P = lower(Q~ K^^T)                (diagonal tile)
//   U = U~ - W S, O = d_k^-1/2 (Q~ S + P U)
//   S <- Diag(e^G_L) S + K'^T U       (serial state recurrence between chunks,
//       same page §2.1)
//
// The same kernel also builds the contrast variants (kda_chunk_fwd_variant): the
// unbounded gate g = -softplus(a) that the bound replaces, and the position-pair
// diagonal tile A_rj = beta_r sum_c k_rc k_jc e^{G_rc - G_jc}, P_rj = sum_c q_rc k_jc
// e^{G_rc - G_jc} (one exponential per pair and channel, no e^-G factor) that an
// unbounded decay forces ("Architecture Analysis of Ultra-Long Context Sparse MoE
// Models", §2.1-2.2; "Demystifying Trillion-Parameter MoE Models", Breakthrough 1 §1).
#include <cuda_bf16.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kSimtThreads = 256;

template <typename IO>
__device__ __forceinline__ float load_io(const IO *p);
template <>
__device__ __forceinline__ float load_io<float>(const float *p) { return *p; }
template <>
__device__ __forceinline__ float load_io<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}
template <typename IO>
__device__ __forceinline__ void store_io(IO *p, float x);
template <>
__device__ __forceinline__ void store_io<float>(float *p, float x) { *p = x; }
template <>
__device__ __forceinline__ void store_io<__nv_bfloat16>(__nv_bfloat16 *p, float x) {
    *p = __float2bfloat16_rn(x);
}

__host__ __device__ inline size_t simt_smem_floats(int dk, int dv, bool pair = false) {
    const int lk = dk + 1, lv = dv + 1;  // odd row pitch: column walks hit distinct banks
    return (size_t)dk * dv + (size_t)6 * kChunk * lk + (size_t)3 * kChunk * lv +
           3 * kChunk * kChunk + dk + kChunk + (pair ? (size_t)kChunk * lk : 0);
}

enum Gate { kBounded = 0, kSoftplus = 1 };

// log-decay of one channel from its gate logit
template <int GATE>
__device__ __forceinline__ float log_decay(float a) {
    if (GATE == kBounded) return kGMin / (1.f + expf(-a));          // -5 sigmoid(a)
    return -(fmaxf(a, 0.f) + log1pf(expf(-fabsf(a))));              // -softplus(a)
}

template <typename IO, int GATE, bool PAIR>
__global__ void __launch_bounds__(kSimtThreads)
    kda_simt_kernel(const IO *__restrict__ q, const IO *__restrict__ k,
                    const IO *__restrict__ v, const float *__restrict__ a,
                    const float *__restrict__ beta, const float *__restrict__ h0,
                    const int32_t *__restrict__ cu_seqlens, IO *__restrict__ out,
                    float *__restrict__ h_final, int H, int dk, int dv) {
    extern __shared__ float sm[];
    const int lk = dk + 1, lv = dv + 1;
    float *S = sm;                        // [dk][dv]
    float *Qt = S + (size_t)dk * dv;      // [16][lk]  q, then q e^G
    float *Kt = Qt + kChunk * lk;         // [16][lk]  k, then k e^G
    float *Kh = Kt + kChunk * lk;         // [16][lk]  k e^-G
    float *Kp = Kh + kChunk * lk;         // [16][lk]  k e^(G_L - G)
    float *Gs = Kp + kChunk * lk;         // [16][lk]  g, then G
    float *W = Gs + kChunk * lk;          // [16][lk]
    float *V = W + kChunk * lk;           // [16][lv]  v
    float *U = V + kChunk * lv;           // [16][lv]  U~, then U
    float *Ob = U + kChunk * lv;          // [16][lv]  Q~ S, then O
    float *A = Ob + kChunk * lv;          // [16][16]
    float *TB = A + kChunk * kChunk;      // [16][16]
    float *P = TB + kChunk * kChunk;      // [16][16]
    float *gl = P + kChunk * kChunk;      // [dk]  e^{G_L}
    float *bt = gl + dk;                  // [16]
    float *Qr = bt + kChunk;              // [16][lk]  q, position-pair tile only

    const int tid = threadIdx.x;
    const int item = blockIdx.x;
    const int n = item / H, h = item % H;
    const int64_t t0 = cu_seqlens[n], t1 = cu_seqlens[n + 1];
    const float scale = rsqrtf((float)dk);
    const size_t sidx = ((size_t)n * H + h) * dk * dv;

    for (int i = tid; i < dk * dv; i += kSimtThreads) S[i] = h0 ? h0[sidx + i] : 0.f;

    for (int64_t c0 = t0; c0 < t1; c0 += kChunk) {
        const int L = (int)(t1 - c0 < kChunk ? t1 - c0 : kChunk);
        __syncthreads();  // previous chunk finished with every buffer
        // 1. load the chunk; padded rows are zero with g = 0
        for (int i = tid; i < kChunk * dk; i += kSimtThreads) {
            const int r = i / dk, c = i % dk;
            float qv = 0.f, kv = 0.f, g = 0.f;
            if (r < L) {
                const size_t o = ((size_t)(c0 + r) * H + h) * dk + c;
                qv = load_io(q + o);
                kv = load_io(k + o);
                g = log_decay<GATE>(a[o]);
            }
            Qt[r * lk + c] = qv;
            Kt[r * lk + c] = kv;
            Gs[r * lk + c] = g;
            if (PAIR) Qr[r * lk + c] = qv;
        }
        for (int i = tid; i < kChunk * dv; i += kSimtThreads) {
            const int r = i / dv, c = i % dv;
            V[r * lv + c] = r < L ? load_io(v + ((size_t)(c0 + r) * H + h) * dv + c) : 0.f;
        }
        if (tid < kChunk) bt[tid] = tid < L ? beta[(size_t)(c0 + tid) * H + h] : 0.f;
        __syncthreads();
        // 2. cumulative log-decay per key channel and the scaled operands
        for (int c = tid; c < dk; c += kSimtThreads) {
            float G = 0.f;
            for (int r = 0; r < kChunk; ++r) {
                G += Gs[r * lk + c];
                Gs[r * lk + c] = G;
            }
            const float GL = G;
            gl[c] = expf(GL);
            for (int r = 0; r < kChunk; ++r) {
                const float Gr = Gs[r * lk + c];
                const float eg = expf(Gr), emg = expf(-Gr);
                const float kv = Kt[r * lk + c];
                Qt[r * lk + c] *= eg;
                Kt[r * lk + c] = kv * eg;
                Kh[r * lk + c] = PAIR ? kv : kv * emg;  // the pair tile keeps k itself
                Kp[r * lk + c] = kv * expf(GL - Gr);
            }
        }
        __syncthreads();
        // 3. A = strict_lower(beta K~ K^^T), P = lower(Q~ K^^T): one (r, j) per thread
        {
            const int r = tid / kChunk, j = tid % kChunk;
            float dkk = 0.f, dqk = 0.f;
            if (!PAIR) {
                for (int c = 0; c < dk; ++c) {
                    const float kh = Kh[j * lk + c];
                    dkk = fmaf(Kt[r * lk + c], kh, dkk);
                    dqk = fmaf(Qt[r * lk + c], kh, dqk);
                }
            } else if (j <= r) {  // position pairs: e^{G_r - G_j} <= 1 for j <= r
                for (int c = 0; c < dk; ++c) {
                    const float e = expf(Gs[r * lk + c] - Gs[j * lk + c]);
                    const float kj = Kh[j * lk + c] * e;
                    dkk = fmaf(Kh[r * lk + c], kj, dkk);
                    dqk = fmaf(Qr[r * lk + c], kj, dqk);
                }
            }
            A[r * kChunk + j] = j < r ? bt[r] * dkk : 0.f;
            P[r * kChunk + j] = j <= r ? dqk : 0.f;
        }
        __syncthreads();
        // 4. TB = (I + A)^-1 diag(beta): forward substitution, one column per thread
        if (tid < kChunk) {
            const int j = tid;
            float col[kChunk];
#pragma unroll
            for (int r = 0; r < kChunk; ++r) {
                float x = r == j ? 1.f : 0.f;
#pragma unroll
                for (int i = 0; i < r; ++i) x = fmaf(-A[r * kChunk + i], col[i], x);
                col[r] = x;
            }
#pragma unroll
            for (int r = 0; r < kChunk; ++r) TB[r * kChunk + j] = col[r] * bt[j];
        }
        __syncthreads();
        // 5. W = TB K~, U~ = TB V
        for (int i = tid; i < kChunk * dk; i += kSimtThreads) {
            const int r = i / dk, c = i % dk;
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < kChunk; ++j) acc = fmaf(TB[r * kChunk + j], Kt[j * lk + c], acc);
            W[r * lk + c] = acc;
        }
        for (int i = tid; i < kChunk * dv; i += kSimtThreads) {
            const int r = i / dv, c = i % dv;
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < kChunk; ++j) acc = fmaf(TB[r * kChunk + j], V[j * lv + c], acc);
            U[r * lv + c] = acc;
        }
        __syncthreads();
        // 6. U = U~ - W S and Q~ S (old state)
        for (int i = tid; i < kChunk * dv; i += kSimtThreads) {
            const int r = i / dv, c = i % dv;
            float ws = 0.f, qs = 0.f;
            for (int x = 0; x < dk; ++x) {
                const float s = S[x * dv + c];
                ws = fmaf(W[r * lk + x], s, ws);
                qs = fmaf(Qt[r * lk + x], s, qs);
            }
            U[r * lv + c] -= ws;
            Ob[r * lv + c] = qs;
        }
        __syncthreads();
        // 7. O = scale (Q~ S + P U); S <- Diag(e^G_L) S + K'^T U
        for (int i = tid; i < kChunk * dv; i += kSimtThreads) {
            const int r = i / dv, c = i % dv;
            float acc = Ob[r * lv + c];
            for (int j = 0; j <= r; ++j) acc = fmaf(P[r * kChunk + j], U[j * lv + c], acc);
            if (r < L) store_io(out + ((size_t)(c0 + r) * H + h) * dv + c, scale * acc);
        }
        for (int i = tid; i < dk * dv; i += kSimtThreads) {
            const int x = i / dv, c = i % dv;
            float acc = gl[x] * S[i];
#pragma unroll
            for (int r = 0; r < kChunk; ++r) acc = fmaf(Kp[r * lk + x], U[r * lv + c], acc);
            S[i] = acc;
        }
    }
    if (h_final) {
        __syncthreads();
        for (int i = tid; i < dk * dv; i += kSimtThreads) h_final[sidx + i] = S[i];
    }
}

template <typename IO, int GATE = kBounded, bool PAIR = false>
cudaError_t launch_simt_t(const FwdArgs &p, cudaStream_t stream) {
    const size_t smem = simt_smem_floats(p.d_k, p.d_v, PAIR) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(kda_simt_kernel<IO, GATE, PAIR>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)p.n_seq * (unsigned)p.n_heads;
    kda_simt_kernel<IO, GATE, PAIR><<<grid, kSimtThreads, smem, stream>>>(
        (const IO *)p.q, (const IO *)p.k, (const IO *)p.v, p.a, p.beta, p.h0,
        p.cu_seqlens, (IO *)p.out, p.h_final, p.n_heads, p.d_k, p.d_v);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

}  // namespace

cudaError_t launch_simt(const FwdArgs &p, cudaStream_t stream) {
    if (p.n_seq == 0) return cudaSuccess;
    return p.bf16 ? launch_simt_t<__nv_bfloat16>(p, stream) : launch_simt_t<float>(p, stream);
}

namespace {
template <typename IO>
cudaError_t launch_variant_t(const FwdArgs &p, int gate, bool pair, cudaStream_t stream) {
    if (gate == kBounded)
        return pair ? launch_simt_t<IO, kBounded, true>(p, stream)
                    : launch_simt_t<IO, kBounded, false>(p, stream);
    return pair ? launch_simt_t<IO, kSoftplus, true>(p, stream)
                : launch_simt_t<IO, kSoftplus, false>(p, stream);
}
}  // namespace

cudaError_t launch_simt_variant(const FwdArgs &p, int gate, bool pair, cudaStream_t stream) {
    if (p.n_seq == 0) return cudaSuccess;
    return p.bf16 ? launch_variant_t<__nv_bfloat16>(p, gate, pair, stream)
                  : launch_variant_t<float>(p, gate, pair, stream);
}

}  // namespace kda
