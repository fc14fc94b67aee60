// kda_bwd.cu -- backward pass of the chunked forward: the gradients of
//   L = <dout, out> + <dh_final, h_final>
// with respect to q, k, v, the gate logits a, beta and h0 (its vector-Jacobian product).
// The pages give the forward only ("From Numerical Stability to Load Balancing", §2.1-2.2);
// this is the derivative of the chunked form of it that kda_simt.cu computes. Chunk-local
// notation (L <= 16 tokens, rows past L acting as q = k = v = 0, beta = 0, g = 0):
//
//   G = inclusive cumsum of g = -5 sigmoid(a), Gamma = e^G, gamma_L = e^{G_15}
//   Q~ = Q Gamma, K~ = K Gamma, K^ = K / Gamma, K' = K gamma_L / Gamma
//   Z = K~ K^^T, A = strict_lower(diag(beta) Z), T = (I + A)^-1, M = T diag(beta)
//   W = M K~, U~ = M V, P = lower(Q~ K^^T), U = U~ - W S
//   O = s (Q~ S + P U),  S_end = Diag(gamma_L) S + K'^T U          (s = d_k^-1/2)
//
// The workspace holds, per (chunk slot, head), the state at the start of the chunk and the
// gradient with respect to its end state, and the chunk's state-independent products:
//   0. chunk products, all chunks in parallel (the record: K', W, Q~, P, U~, ...);
//   1. forward serial pass per (sequence, head): the state at the start of every chunk;
//   2. reverse serial pass per (sequence, head), last chunk first. dS, the gradient with
//      respect to the current chunk's end state, is stored, then carried to its start:
//        X = K' dS + s P^T dO,   dS <- Diag(gamma_L) dS + s Q~^T dO - W^T X
//      (the transpose of the chunk's affine state map: S_end = (Diag(gamma_L) - K'^T W)
//      S + K'^T U~ and O = s (Q~ - P W) S + s P U~); dh0 is the dS left at the first chunk;
//      passes 1 and 2 are independent of each other;
//   3. local gradients, all (sequence, head, chunk) independent given S and dS_end:
//        dU = s P^T dO + K' dS_end            dP = lower(s dO U^T)
//        dQ~ = s dO S^T + dP K^                dK' = U dS_end^T
//        dW = -dU S^T                          dgamma_L = rowsum(dS_end . S)
//        dM = dW K~^T + dU V^T                 dV = M^T dU,  dK~ = M^T dW + dZ K^
//        dbeta_j = sum_i dM_ij T_ij + sum_i dA_ji Z_ji,  dA = strict_lower(-T^T dM diag(beta) T^T)
//        dZ = diag(beta) dA,                   dK^ = dP^T Q~ + dZ^T K~
//        dQ = dQ~ Gamma,  dK = dK~ Gamma + dK^ / Gamma + dK' gamma_L / Gamma
//        dG = dQ~ Q~ + dK~ K~ - dK^ K^ - dK' K'  (+ gamma_L dgamma_L + colsum(dK' K') at row 15)
//        dg = reverse cumsum of dG,  da = dg (-5) sigmoid(a) (1 - sigmoid(a))
// Two implementations: for bf16 I/O at d_k = d_v = 128 (16-byte aligned buffers) the
// tensor-core kernels (prep_tc_kernel, chains_tc_kernel with both serial passes in one
// launch, local_tc_kernel: mma.sync with bf16 operands and fp32 accumulation, bf16 state
// tiles, TMA tensor and bulk copies); otherwise fp32 FMA kernels (prep_kernel, ckpt_kernel,
// chain_kernel, local_kernel: fp32 states, S and dS_end read 32 columns at a time).
// The chunk of token start t in sequence n has the workspace slot (cu[n] >> 4) + c + n:
// strictly increasing over all chunks, below (n_tok >> 4) + n_seq + 1.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <climits>
#include <mutex>
#include <vector>

#include "kda_internal.h"

namespace kda {

__device__ unsigned int g_bwd_flags;  // bit 2: a serial-pass wait exceeded its limit

namespace {

constexpr int C = kChunk;
constexpr int kThreads = 256;
constexpr int JB = 32;  // value columns of S / dS_end per block in the local-gradient kernel

__device__ __forceinline__ float ld_io(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld_io(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void st_io(float *p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st_io(__nv_bfloat16 *p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

__device__ __forceinline__ size_t slot_of(const int32_t *cu, int n, int c) {
    return (size_t)(cu[n] >> 4) + (size_t)c + (size_t)n;
}

// Shared-memory views of one chunk's prologue products (pitches lk = d_k + 1, lv = d_v + 1).
struct Chunk {
    float *Qt, *Kt, *Kh, *Kp, *Gs, *W;  // [16][lk]: Q~, K~, K^, K', G, W
    float *V, *Ut;                      // [16][lv]: V, U~
    float *Z, *T, *M, *P;               // [16][16]: K~ K^^T, (I + A)^-1, T diag(beta), P
    float *gl, *bt;                     // [d_k] gamma_L, [16] beta
};

__host__ __device__ constexpr size_t chunk_floats(int dk, int dv) {
    return (size_t)6 * C * (dk + 1) + (size_t)2 * C * (dv + 1) + 4 * C * C + dk + C;
}

__device__ Chunk carve_chunk(float *p, int dk, int dv) {
    const int lk = dk + 1, lv = dv + 1;
    Chunk b;
    b.Qt = p; p += C * lk;
    b.Kt = p; p += C * lk;
    b.Kh = p; p += C * lk;
    b.Kp = p; p += C * lk;
    b.Gs = p; p += C * lk;
    b.W = p; p += C * lk;
    b.V = p; p += C * lv;
    b.Ut = p; p += C * lv;
    b.Z = p; p += C * C;
    b.T = p; p += C * C;
    b.M = p; p += C * C;
    b.P = p; p += C * C;
    b.gl = p; p += dk;
    b.bt = p;
    return b;
}

// The chunk prologue of tokens [c0, c0 + L) of head h: every product above that does not
// involve the state. want_q: also Q~ and P. Ends with a barrier.
template <typename IO>
__device__ void prologue(const Chunk &b, const IO *q, const IO *k, const IO *v, const float *a,
                         const float *beta, int64_t c0, int L, int H, int h, int dk, int dv,
                         bool want_q) {
    const int tid = threadIdx.x, lk = dk + 1, lv = dv + 1;
    __syncthreads();  // the previous user of the buffers is done
    for (int i = tid; i < C * dk; i += kThreads) {
        const int r = i / dk, c = i % dk;
        float qv = 0.f, kv = 0.f, g = 0.f;
        if (r < L) {
            const size_t o = ((size_t)(c0 + r) * H + h) * dk + c;
            if (want_q) qv = ld_io(q, o);
            kv = ld_io(k, o);
            g = kGMin / (1.f + expf(-a[o]));
        }
        b.Qt[r * lk + c] = qv;
        b.Kt[r * lk + c] = kv;
        b.Gs[r * lk + c] = g;
    }
    for (int i = tid; i < C * dv; i += kThreads) {
        const int r = i / dv, c = i % dv;
        b.V[r * lv + c] = r < L ? ld_io(v, ((size_t)(c0 + r) * H + h) * dv + c) : 0.f;
    }
    if (tid < C) b.bt[tid] = tid < L ? beta[(size_t)(c0 + tid) * H + h] : 0.f;
    __syncthreads();
    for (int c = tid; c < dk; c += kThreads) {  // cumulative log-decay, scaled operands
        float G = 0.f;
        for (int r = 0; r < C; ++r) {
            G += b.Gs[r * lk + c];
            b.Gs[r * lk + c] = G;
        }
        const float GL = G;
        b.gl[c] = expf(GL);
        for (int r = 0; r < C; ++r) {
            const float Gr = b.Gs[r * lk + c], kv = b.Kt[r * lk + c];
            b.Qt[r * lk + c] *= expf(Gr);
            b.Kt[r * lk + c] = kv * expf(Gr);
            b.Kh[r * lk + c] = kv * expf(-Gr);
            b.Kp[r * lk + c] = kv * expf(GL - Gr);
        }
    }
    __syncthreads();
    {  // Z = K~ K^^T, A = strict_lower(beta Z) (kept in M for the solve), P = lower(Q~ K^^T)
        const int r = tid / C, j = tid % C;
        float z = 0.f, pq = 0.f;
        for (int c = 0; c < dk; ++c) {
            const float kh = b.Kh[j * lk + c];
            z = fmaf(b.Kt[r * lk + c], kh, z);
            if (want_q) pq = fmaf(b.Qt[r * lk + c], kh, pq);
        }
        b.Z[r * C + j] = z;
        b.M[r * C + j] = j < r ? b.bt[r] * z : 0.f;
        b.P[r * C + j] = (want_q && j <= r) ? pq : 0.f;
    }
    __syncthreads();
    if (tid < C) {  // T = (I + A)^-1 by forward substitution, one column per thread
        const int j = tid;
        float col[C];
#pragma unroll
        for (int r = 0; r < C; ++r) {
            float x = r == j ? 1.f : 0.f;
#pragma unroll
            for (int i = 0; i < r; ++i) x = fmaf(-b.M[r * C + i], col[i], x);
            col[r] = x;
        }
#pragma unroll
        for (int r = 0; r < C; ++r) b.T[r * C + j] = col[r];
    }
    __syncthreads();
    {  // M = T diag(beta)
        const int r = tid / C, j = tid % C;
        b.M[r * C + j] = b.T[r * C + j] * b.bt[j];
    }
    __syncthreads();
    for (int i = tid; i < C * dk; i += kThreads) {  // W = M K~
        const int r = i / dk, c = i % dk;
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < C; ++j) acc = fmaf(b.M[r * C + j], b.Kt[j * lk + c], acc);
        b.W[r * lk + c] = acc;
    }
    for (int i = tid; i < C * dv; i += kThreads) {  // U~ = M V
        const int r = i / dv, c = i % dv;
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < C; ++j) acc = fmaf(b.M[r * C + j], b.V[j * lv + c], acc);
        b.Ut[r * lv + c] = acc;
    }
    __syncthreads();
}

// bulk prefetch of [p, p + bytes) into L2 (16-byte aligned, size a multiple of 16)
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---- tensor-core fragments (mma.sync m16n8k16, bf16 operands, fp32 accumulation)
__device__ __forceinline__ void ldsm4(uint32_t a, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}
__device__ __forceinline__ void ldsm4t(uint32_t a, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}
__device__ __forceinline__ void stsm4(uint32_t a, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};"
                 ::"r"(a), "r"(r0), "r"(r1), "r"(r2), "r"(r3) : "memory");
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// A fragment: rows [0, 16), columns [k0, k0 + 16) of a row-major bf16 tile
__device__ __forceinline__ void ld_a(uint32_t base, int pitch, int k0, uint32_t (&a)[4]) {
    const int l = threadIdx.x & 31;
    ldsm4(base + (uint32_t)(((l & 15) * pitch + k0 + (l >> 4) * 8) * 2), a);
}
// B fragments of the two n8 tiles [n0, n0 + 16) x k16 [k0, k0 + 16): from [n][k] storage
// (b[0], b[1] the first tile, b[2], b[3] the second), or from [k][n] storage (transposed read)
__device__ __forceinline__ void ld_b_nk(uint32_t base, int pitch, int n0, int k0, uint32_t (&b)[4]) {
    const int l = threadIdx.x & 31;
    ldsm4(base + (uint32_t)(((n0 + (l & 7) + ((l >> 4) << 3)) * pitch + k0 + ((l >> 3) & 1) * 8) * 2), b);
}
__device__ __forceinline__ void ld_b_kn(uint32_t base, int pitch, int k0, int n0, uint32_t (&b)[4]) {
    const int l = threadIdx.x & 31;
    ldsm4t(base + (uint32_t)(((k0 + (l & 7) + (((l >> 3) & 1) << 3)) * pitch + n0 + (l >> 4) * 8) * 2), b);
}
// A fragment of X^T (16 x 16) from X stored row-major [k][m]: rows [k0, k0 + 16), columns
// [m0, m0 + 16) of the storage
__device__ __forceinline__ void ld_a_t(uint32_t base, int pitch, int k0, int m0, uint32_t (&a)[4]) {
    const int l = threadIdx.x & 31, j = l >> 3;
    ldsm4t(base + (uint32_t)(((k0 + ((j >> 1) << 3) + (l & 7)) * pitch + m0 + ((j & 1) << 3)) * 2), a);
}
// A [16][128] bf16 tile stored as two [16][64] halves, each written by a tensor copy with
// 128-byte swizzle: the 16-byte chunk k of row r of a half sits at chunk k ^ (r & 7).
// Address of the 8 elements starting at (r, c0), c0 a multiple of 8:
__device__ __forceinline__ uint32_t sw128(uint32_t base, int r, int c0) {
    return base + (uint32_t)((c0 >> 6) * (C * 128) + r * 128 + ((((c0 & 63) >> 3) ^ (r & 7)) << 4));
}
// the fragment loaders above, for such tiles
__device__ __forceinline__ void ld_a_sw(uint32_t base, int k0, uint32_t (&a)[4]) {
    const int l = threadIdx.x & 31;
    ldsm4(sw128(base, l & 15, k0 + (l >> 4) * 8), a);
}
__device__ __forceinline__ void ld_b_nk_sw(uint32_t base, int n0, int k0, uint32_t (&b)[4]) {
    const int l = threadIdx.x & 31;
    ldsm4(sw128(base, n0 + (l & 7) + ((l >> 4) << 3), k0 + ((l >> 3) & 1) * 8), b);
}
__device__ __forceinline__ void ld_b_kn_sw(uint32_t base, int k0, int n0, uint32_t (&b)[4]) {
    const int l = threadIdx.x & 31;
    ldsm4t(sw128(base, k0 + (l & 7) + (((l >> 3) & 1) << 3), n0 + (l >> 4) * 8), b);
}
// the accumulator tile (16 rows x columns [n0, n0 + 16)) into bf16 row-major storage
__device__ __forceinline__ void store_c16(__nv_bfloat16 *dst, int pitch, int n0,
                                          const float (&acc)[2][4]) {
    const int l = threadIdx.x & 31, g4 = l >> 2, l4 = l & 3;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int col = n0 + 8 * t + 2 * l4;
        *reinterpret_cast<__nv_bfloat162 *>(dst + g4 * pitch + col) = __floats2bfloat162_rn(acc[t][0], acc[t][1]);
        *reinterpret_cast<__nv_bfloat162 *>(dst + (g4 + 8) * pitch + col) =
            __floats2bfloat162_rn(acc[t][2], acc[t][3]);
    }
}
constexpr int PB = 136;  // bf16 pitch of 128-wide operand tiles: 272-byte rows, conflict-free
constexpr int PS = 24;   // bf16 pitch of 16-wide operand tiles

// ---- 0. the state-independent products of every chunk, all chunks in parallel
// Record per (chunk slot, head): K', W, Q~ [16][d_k], U~ [16][d_v], P [16][16], gamma_L
// [d_k], fp32, unpadded.
__host__ __device__ constexpr size_t prep_floats(int dk, int dv) {
    return (size_t)3 * C * dk + (size_t)C * dv + C * C + dk;
}
__host__ __device__ constexpr size_t P_KP(int) { return 0; }
__host__ __device__ constexpr size_t P_W(int dk) { return (size_t)C * dk; }
__host__ __device__ constexpr size_t P_QT(int dk) { return (size_t)2 * C * dk; }
__host__ __device__ constexpr size_t P_UT(int dk) { return (size_t)3 * C * dk; }
__host__ __device__ constexpr size_t P_P(int dk, int dv) { return (size_t)3 * C * dk + (size_t)C * dv; }
__host__ __device__ constexpr size_t P_GL(int dk, int dv) { return P_P(dk, dv) + C * C; }

// Tensor-core path (bf16 I/O, d_k = d_v = 128): the workspace holds, per (chunk slot, head),
// REC_TC bytes -- the chunk's start state S and end-state gradient dS_end as bf16 S^T
// tiles [128 v][136] (written by the two serial passes in the row layout shared memory
// uses), then the prep kernel's record of the chunk's state-independent products:
//   K', -W, Q~ bf16 [16][136]; P bf16 [16][24]; gamma_L fp32 in the serial passes' float4
//   order (the part [0, TR_OPS) is what the serial passes copy); U~^T fp32 [128 v][16 t];
//   K~, K^ bf16 [16][136]; M bf16 [16][24]; T, T^T, Z fp32 [16][16]; beta fp32 [16];
//   G fp32 [16][136]; gamma_L fp32 [128].
constexpr int T128 = C * 136 * 2;        // a [16][PB] bf16 tile
constexpr int TR_K = 0, TR_W = T128, TR_Q = 2 * T128, TR_P = 3 * T128;
constexpr int TR_G = TR_P + C * 24 * 2;
constexpr int TR_OPS = TR_G + 128 * 4;   // bytes the serial passes' copies start from
constexpr int TR_UT = TR_OPS;            // + 2048 r: value block r's U~^T [32][16]
constexpr int TR_KT = TR_UT + 128 * C * 4, TR_KH = TR_KT + T128;
constexpr int TR_M = TR_KH + T128;
constexpr int TR_T = TR_M + C * 24 * 2, TR_TT = TR_T + C * C * 4, TR_Z = TR_TT + C * C * 4;
constexpr int TR_B = TR_Z + C * C * 4;
constexpr int GP = 136;                  // pitch (floats) of the record's G rows
constexpr int TR_GS = TR_B + C * 4, TR_GL = TR_GS + C * GP * 4;
constexpr int RECB = TR_GL + 128 * 4;    // record bytes
constexpr int ST16 = 128 * 136 * 2;      // a bf16 state tile
constexpr size_t TC_S = 0, TC_DS = ST16, TC_REC = 2 * ST16;
constexpr size_t REC_TC = TC_REC + RECB; // workspace bytes per (chunk slot, head)
static_assert(TR_G % 16 == 0 && TR_OPS % 16 == 0 && TR_KT % 16 == 0 && TR_M % 16 == 0 &&
                  TR_T % 16 == 0 && TR_GS % 16 == 0 && RECB % 16 == 0 && REC_TC % 16 == 0,
              "16-byte record parts");
static_assert(REC_TC <= ((size_t)2 * 128 * 128 + prep_floats(128, 128)) * 4,
              "the tensor-core layout fits the workspace the fp32 layout sizes");
// gamma_L[c], c = 16 np + 8 hh + 2 l4 + e, stored at 16 np + 4 l4 + 2 hh + e: the lane holding
// S^T columns 2 l4 (+1, +8, +9) of 16-column group np reads its four factors as one float4
__device__ __forceinline__ int gperm_tc(int c) {
    return ((c >> 4) * 4 + ((c >> 1) & 3)) * 4 + ((c >> 3) & 1) * 2 + (c & 1);
}

template <typename IO>
__global__ void __launch_bounds__(kThreads)
    prep_kernel(const IO *__restrict__ q, const IO *__restrict__ k, const IO *__restrict__ v,
                const float *__restrict__ a, const float *__restrict__ beta,
                const int32_t *__restrict__ cu, float *__restrict__ prep,
                int H, int dk, int dv) {
    extern __shared__ float sm[];
    const int tid = threadIdx.x, lk = dk + 1, lv = dv + 1;
    const int n = blockIdx.x / H, h = blockIdx.x % H;
    const Chunk b = carve_chunk(sm, dk, dv);
    const size_t rec = prep_floats(dk, dv);
    const int64_t t0 = cu[n], t1 = cu[n + 1];
    const int nc = (int)((t1 - t0 + C - 1) / C);
    for (int c = blockIdx.y; c < nc; c += gridDim.y) {
        const int64_t c0 = t0 + (int64_t)c * C;
        const int L = (int)(t1 - c0 < C ? t1 - c0 : C);
        prologue(b, q, k, v, a, beta, c0, L, H, h, dk, dv, true);
        {
            float *o = prep + (slot_of(cu, n, c) * H + h) * rec;
            for (int i = tid; i < C * dk; i += kThreads) {
                const int r = i / dk, x = i % dk;
                o[P_KP(dk) + i] = b.Kp[r * lk + x];
                o[P_W(dk) + i] = b.W[r * lk + x];
                o[P_QT(dk) + i] = b.Qt[r * lk + x];
            }
            for (int i = tid; i < C * dv; i += kThreads)
                o[P_UT(dk) + i] = b.Ut[(i / dv) * lv + i % dv];
            o[P_P(dk, dv) + tid] = b.P[tid];  // kThreads == C * C
            for (int x = tid; x < dk; x += kThreads) o[P_GL(dk, dv) + x] = b.gl[x];
        }
    }
}

// The serial passes split the value columns: column j of S (and of dS) evolves on its own
// given the chunk products, so CTA (sequence, head, block) carries JS columns of one
// chain, thread t holding rows [RPT (t / JS), RPT (t / JS) + RPT) of column t mod JS in
// registers. The chunk's products are staged into shared memory with 4-byte cp.async one
// chunk ahead (any d_k, d_v).
constexpr int JS = 16;                 // value columns per CTA
constexpr int RG = kThreads / JS;      // row groups (16)
constexpr int RPT = 128 / RG;          // rows per thread (8): d_k <= 128

__device__ __forceinline__ void cp_async4(float *dst, const float *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void cp_async16(float *dst, const float *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}

// Stage one chunk's products for value columns [j0, j0 + JS): K' and W (and Q~, P when
// chain) whole, U~ only for those columns, gamma_L. 16-byte copies when every piece is a
// multiple of 4 floats (d_k, d_v multiples of 4) and the record starts on a 16-byte
// boundary (the workspace need only be 4-byte aligned), 4-byte copies otherwise.
__device__ void stage(float *dst, const float *rec, int dk, int dv, int j0, bool chain) {
    const int tid = threadIdx.x;
    const bool v4 = (dk & 3) == 0 && (dv & 3) == 0 && (reinterpret_cast<uintptr_t>(rec) & 15) == 0;
    if (v4) {
        for (int i = tid; i < C * dk / 4; i += kThreads) {
            cp_async16(dst + 4 * i, rec + P_KP(dk) + 4 * i);
            cp_async16(dst + C * dk + 4 * i, rec + P_W(dk) + 4 * i);
            if (chain) cp_async16(dst + 2 * C * dk + 4 * i, rec + P_QT(dk) + 4 * i);
        }
    } else {
        for (int i = tid; i < C * dk; i += kThreads) {
            cp_async4(dst + i, rec + P_KP(dk) + i);
            cp_async4(dst + C * dk + i, rec + P_W(dk) + i);
            if (chain) cp_async4(dst + 2 * C * dk + i, rec + P_QT(dk) + i);
        }
    }
    float *d2 = dst + 3 * C * dk;
    if (!chain) {
        if (v4 && j0 + JS <= dv) {
            for (int i = tid; i < C * JS / 4; i += kThreads) {
                const int r = i / (JS / 4), q4 = i % (JS / 4);
                cp_async16(d2 + 4 * i, rec + P_UT(dk) + (size_t)r * dv + j0 + 4 * q4);
            }
        } else {
            for (int i = tid; i < C * JS; i += kThreads) {
                const int r = i / JS, jj = i % JS;
                if (j0 + jj < dv) cp_async4(d2 + i, rec + P_UT(dk) + (size_t)r * dv + j0 + jj);
            }
        }
    }
    if (chain) cp_async4(d2 + C * JS + tid, rec + P_P(dk, dv) + tid);
    for (int x = tid; x < dk; x += kThreads) cp_async4(d2 + C * JS + C * C + x, rec + P_GL(dk, dv) + x);
    cp_async_commit();
}
__host__ __device__ constexpr int stage_floats(int dk) { return 3 * C * dk + C * JS + C * C + dk; }

// ---- 1. forward recurrence with a checkpoint at every chunk start (column blocks)
__global__ void __launch_bounds__(kThreads)
    ckpt_kernel(const float *__restrict__ h0, const int32_t *__restrict__ cu,
                const float *__restrict__ prep, float *__restrict__ ck, int H, int dk, int dv) {
    extern __shared__ float sm[];
    const int tid = threadIdx.x, jj = tid % JS, rg = tid / JS;
    const int n = blockIdx.x / H, h = blockIdx.x % H, j0 = blockIdx.y * JS, j = j0 + jj;
    const bool col = j < dv;
    const int sf = stage_floats(dk);
    auto buf = [&](int i) { return sm + (i & 1) * sf; };  // two staging buffers
    float *part = sm + 2 * sf;          // [RG][16][JS] partial sums of W S
    float *U = part + RG * C * JS;      // [16][JS]
    const size_t st = (size_t)dk * dv, rec = prep_floats(dk, dv);
    float s[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int x = rg * RPT + i;
        s[i] = (h0 && col && x < dk) ? h0[((size_t)n * H + h) * st + (size_t)x * dv + j] : 0.f;
    }
    const int64_t t0 = cu[n], t1 = cu[n + 1];
    const int nc = (int)((t1 - t0 + C - 1) / C);
    if (nc > 0) stage(buf(0), prep + (slot_of(cu, n, 0) * H + h) * rec, dk, dv, j0, false);
    for (int c = 0; c < nc; ++c) {
        cp_async_wait_all();
        __syncthreads();  // chunk c staged; every reader of the other buffer is done
        if (c + 1 < nc) stage(buf(c + 1), prep + (slot_of(cu, n, c + 1) * H + h) * rec, dk, dv, j0, false);
        const float *Kp = buf(c), *W = Kp + C * dk, *Ut = Kp + 3 * C * dk;
        const float *gl = Ut + C * JS + C * C;
        float *dst = ck + (slot_of(cu, n, c) * H + h) * st;
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const int x = rg * RPT + i;
            if (col && x < dk) dst[(size_t)x * dv + j] = s[i];
        }
        if (dk == RG * RPT) {  // full height: this thread's rows as float4 per product row
#pragma unroll
            for (int r = 0; r < C; ++r) {
                float acc = 0.f;
#pragma unroll
                for (int i = 0; i < RPT; i += 4) {
                    const float4 w = *reinterpret_cast<const float4 *>(W + r * dk + rg * RPT + i);
                    acc = fmaf(w.x, s[i], acc); acc = fmaf(w.y, s[i + 1], acc);
                    acc = fmaf(w.z, s[i + 2], acc); acc = fmaf(w.w, s[i + 3], acc);
                }
                part[(rg * C + r) * JS + jj] = acc;
            }
        } else {
#pragma unroll
        for (int r = 0; r < C; ++r) {  // this thread's rows of (W S)[r][j]
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const int x = rg * RPT + i;
                if (x < dk) acc = fmaf(W[r * dk + x], s[i], acc);
            }
            part[(rg * C + r) * JS + jj] = acc;
        }
        }
        __syncthreads();
        if (tid < C * JS) {  // U = U~ - W S, one (r, column) per thread
            const int r = tid / JS;
            float acc = Ut[r * JS + jj];
#pragma unroll
            for (int g = 0; g < RG; ++g) acc -= part[(g * C + r) * JS + jj];
            U[r * JS + jj] = acc;
        }
        __syncthreads();
        if (dk == RG * RPT) {  // S <- Diag(gamma_L) S + K'^T U, float4 rows
            float u[C];
#pragma unroll
            for (int r = 0; r < C; ++r) u[r] = U[r * JS + jj];
#pragma unroll
            for (int i = 0; i < RPT; i += 4) {
                const float4 g = *reinterpret_cast<const float4 *>(gl + rg * RPT + i);
                float a0 = g.x * s[i], a1 = g.y * s[i + 1], a2 = g.z * s[i + 2], a3 = g.w * s[i + 3];
#pragma unroll
                for (int r = 0; r < C; ++r) {
                    const float4 kp = *reinterpret_cast<const float4 *>(Kp + r * dk + rg * RPT + i);
                    a0 = fmaf(kp.x, u[r], a0); a1 = fmaf(kp.y, u[r], a1);
                    a2 = fmaf(kp.z, u[r], a2); a3 = fmaf(kp.w, u[r], a3);
                }
                s[i] = a0; s[i + 1] = a1; s[i + 2] = a2; s[i + 3] = a3;
            }
        } else {
#pragma unroll
        for (int i = 0; i < RPT; ++i) {  // S <- Diag(gamma_L) S + K'^T U
            const int x = rg * RPT + i;
            if (x < dk) {
                float acc = gl[x] * s[i];
#pragma unroll
                for (int r = 0; r < C; ++r) acc = fmaf(Kp[r * dk + x], U[r * JS + jj], acc);
                s[i] = acc;
            }
        }
        }
    }
}

// ---- 2. reverse chain of the state gradient (column blocks)
template <typename IO>
__global__ void __launch_bounds__(kThreads)
    chain_kernel(const int32_t *__restrict__ cu, const IO *__restrict__ dout,
                 const float *__restrict__ dh_final, const float *__restrict__ prep,
                 float *__restrict__ dck, float *__restrict__ dh0, int H, int dk, int dv,
                 float scale) {
    extern __shared__ float sm[];
    const int tid = threadIdx.x, jj = tid % JS, rg = tid / JS;
    const int n = blockIdx.x / H, h = blockIdx.x % H, j0 = blockIdx.y * JS, j = j0 + jj;
    const bool col = j < dv;
    const int sf = stage_floats(dk);
    auto buf = [&](int i) { return sm + (i & 1) * sf; };  // two staging buffers
    float *part = sm + 2 * sf;          // [RG][16][JS] partial sums of K' dS
    float *X = part + RG * C * JS;      // [16][JS]
    float *dO = X + C * JS;             // [16][JS]
    const size_t st = (size_t)dk * dv, rec = prep_floats(dk, dv);
    float ds[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int x = rg * RPT + i;
        ds[i] = (dh_final && col && x < dk)
                    ? dh_final[((size_t)n * H + h) * st + (size_t)x * dv + j] : 0.f;
    }
    const int64_t t0 = cu[n], t1 = cu[n + 1];
    const int nc = (int)((t1 - t0 + C - 1) / C);
    if (nc > 0) stage(buf(nc - 1), prep + (slot_of(cu, n, nc - 1) * H + h) * rec, dk, dv, j0, true);
    for (int c = nc - 1; c >= 0; --c) {
        const int64_t c0 = t0 + (int64_t)c * C;
        const int L = (int)(t1 - c0 < C ? t1 - c0 : C);
        cp_async_wait_all();
        __syncthreads();
        if (c > 0) stage(buf(c - 1), prep + (slot_of(cu, n, c - 1) * H + h) * rec, dk, dv, j0, true);
        const float *Kp = buf(c), *W = Kp + C * dk, *Qt = Kp + 2 * C * dk;
        const float *P = Qt + C * dk + C * JS, *gl = P + C * C;
        if (tid < C * JS) {
            const int r = tid / JS;
            dO[r * JS + jj] = (r < L && col) ? ld_io(dout, ((size_t)(c0 + r) * H + h) * dv + j) : 0.f;
        }
        float *dst = dck + (slot_of(cu, n, c) * H + h) * st;
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const int x = rg * RPT + i;
            if (col && x < dk) dst[(size_t)x * dv + j] = ds[i];
        }
        if (dk == RG * RPT) {  // full height: this thread's rows as float4 per product row
#pragma unroll
            for (int r = 0; r < C; ++r) {
                float acc = 0.f;
#pragma unroll
                for (int i = 0; i < RPT; i += 4) {
                    const float4 k4 = *reinterpret_cast<const float4 *>(Kp + r * dk + rg * RPT + i);
                    acc = fmaf(k4.x, ds[i], acc); acc = fmaf(k4.y, ds[i + 1], acc);
                    acc = fmaf(k4.z, ds[i + 2], acc); acc = fmaf(k4.w, ds[i + 3], acc);
                }
                part[(rg * C + r) * JS + jj] = acc;
            }
        } else {
#pragma unroll
        for (int r = 0; r < C; ++r) {  // this thread's rows of (K' dS)[r][j]
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const int x = rg * RPT + i;
                if (x < dk) acc = fmaf(Kp[r * dk + x], ds[i], acc);
            }
            part[(rg * C + r) * JS + jj] = acc;
        }
        }
        __syncthreads();
        if (tid < C * JS) {  // X = K' dS + s P^T dO
            const int r = tid / JS;
            float acc = 0.f;
#pragma unroll
            for (int g = 0; g < RG; ++g) acc += part[(g * C + r) * JS + jj];
            float pd = 0.f;
            for (int i2 = r; i2 < C; ++i2) pd = fmaf(P[i2 * C + r], dO[i2 * JS + jj], pd);
            X[r * JS + jj] = fmaf(scale, pd, acc);
        }
        __syncthreads();
        if (dk == RG * RPT) {  // dS <- Diag(gamma_L) dS + s Q~^T dO - W^T X, float4 rows
            float od[C], xr[C];
#pragma unroll
            for (int r = 0; r < C; ++r) {
                od[r] = scale * dO[r * JS + jj];
                xr[r] = X[r * JS + jj];
            }
#pragma unroll
            for (int i = 0; i < RPT; i += 4) {
                const float4 g = *reinterpret_cast<const float4 *>(gl + rg * RPT + i);
                float a0 = g.x * ds[i], a1 = g.y * ds[i + 1], a2 = g.z * ds[i + 2], a3 = g.w * ds[i + 3];
#pragma unroll
                for (int r = 0; r < C; ++r) {
                    const float4 qt = *reinterpret_cast<const float4 *>(Qt + r * dk + rg * RPT + i);
                    const float4 w = *reinterpret_cast<const float4 *>(W + r * dk + rg * RPT + i);
                    a0 = fmaf(qt.x, od[r], fmaf(-w.x, xr[r], a0));
                    a1 = fmaf(qt.y, od[r], fmaf(-w.y, xr[r], a1));
                    a2 = fmaf(qt.z, od[r], fmaf(-w.z, xr[r], a2));
                    a3 = fmaf(qt.w, od[r], fmaf(-w.w, xr[r], a3));
                }
                ds[i] = a0; ds[i + 1] = a1; ds[i + 2] = a2; ds[i + 3] = a3;
            }
        } else {
#pragma unroll
        for (int i = 0; i < RPT; ++i) {  // dS <- Diag(gamma_L) dS + s Q~^T dO - W^T X
            const int x = rg * RPT + i;
            if (x < dk) {
                float qd = 0.f, wx = 0.f;
#pragma unroll
                for (int r = 0; r < C; ++r) {
                    qd = fmaf(Qt[r * dk + x], dO[r * JS + jj], qd);
                    wx = fmaf(W[r * dk + x], X[r * JS + jj], wx);
                }
                ds[i] = gl[x] * ds[i] + scale * qd - wx;
            }
        }
        }
    }
    if (dh0) {
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const int x = rg * RPT + i;
            if (col && x < dk) dh0[((size_t)n * H + h) * st + (size_t)x * dv + j] = ds[i];
        }
    }
}

// ---- 1b/2b. the two serial passes on the tensor cores (bf16 I/O, d_k = d_v = 128)
// CTA (sequence, head, r) carries value columns [32 r, 32 r + 32) of one chain: two chain
// warps hold 16 rows each of S^T (or dS^T, d_v x d_k) as fp32 mma fragments in registers
// for the whole sequence, and two loader warps convert each chunk's products from its prep
// record into bf16 operand tiles a few chunks ahead (a ring of NS slots). Per chunk, with
// a warp's rows of the state A = S^T as bf16 A fragments (mma.sync m16n8k16):
//   forward:  write S^T (the chunk's start state); U^T = U~^T + S^T (-W)^T;
//             S^T <- S^T Diag(gamma_L) + U^T K'
//   reverse:  write dS^T (the gradient at the chunk's end); X^T = dS^T K'^T + (s dO)^T P;
//             dS^T <- dS^T Diag(gamma_L) + (s dO)^T Q~ + X^T (-W)
// the transposed forms of the two chains above, the state an fp32 accumulator throughout.
constexpr int NS = 4;                    // ring slots
constexpr int PO = 32;                   // bf16 pitch of the [16][32] dO slice (a dense TMA box)
// slot layout (bytes): the record's operand part [0, TR_OPS) (K', -W, Q~, P, gamma_L), then
// U~^T [32][16] fp32 (forward) or dO [16][PO] bf16 (reverse)
constexpr int SL_K = TR_K, SL_W = TR_W, SL_Q = TR_Q, SL_P = TR_P, SL_G = TR_G, SL_X = TR_OPS;
constexpr int SLOT = SL_X + 32 * C * 4;
constexpr int CT_ROWS = 16 * 136 * 2;    // a chain warp's 16 rows of a bf16 state tile
static_assert(SL_X % 16 == 0 && SLOT % 16 == 0, "16-byte aligned slot parts");

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(mbar) : "memory");
}
__device__ __forceinline__ void bar_arrive_tx(uint32_t a, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes)
                 : "memory");
}
// a box of a 3-D tensor map (x innermost) into shared memory, completing on mbar
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            int z, uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(map), "r"(x), "r"(y), "r"(z), "r"(mbar) : "memory");
}
// a box of a 3-D tensor map into L2
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
                 ::"l"(map), "r"(x), "r"(y), "r"(z) : "memory");
}
__device__ __forceinline__ void bar_init(uint32_t a, uint32_t c) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(c));
}
__device__ __forceinline__ void bar_arrive(uint32_t a) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}
__device__ __forceinline__ bool bar_try(uint32_t a, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok) : "r"(a), "r"(parity) : "memory");
    return ok != 0;
}
// bounded wait; false when this or another wait of the grid gave up
__device__ bool bar_wait(uint32_t a, uint32_t parity) {
    if (bar_try(a, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (bar_try(a, parity)) return true;
        if ((it & 63u) == 0) {
            if (*(volatile unsigned int *)&g_bwd_flags != 0u) return false;
            if (clock64() - t0 > 4000000000LL) {
                atomicOr(&g_bwd_flags, 4u);
                return false;
            }
        }
    }
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ void mul2(float &a, float &b, float ga, float gb) {
    asm("{ .reg .b64 x, y; mov.b64 x, {%0, %1}; mov.b64 y, {%2, %3}; mul.rn.f32x2 x, x, y; "
        "mov.b64 {%0, %1}, x; }"
        : "+f"(a), "+f"(b) : "f"(ga), "f"(gb));
}

template <bool REVERSE>
__device__ __forceinline__ void chain_body(int blk, unsigned char *smc, unsigned long long *bars,
                                           const int32_t *__restrict__ cu,
                                           unsigned char *__restrict__ ws,
                                           const CUtensorMap *tm_dout,
                                           const float *__restrict__ init,
                                           float *__restrict__ final_state, int H, float scale) {
    constexpr int D = 128;
    // roles by warp: chain warps 0, 1 and loader warp 2 (forward); the reverse pass takes
    // warps 2, 3 as chain warps and 0 as loader, so that a forward and a reverse CTA on
    // one SM put their four chain warps on four different schedulers
    const int lane = threadIdx.x & 31, warp = (threadIdx.x >> 5) ^ (REVERSE ? 2 : 0);
    const int item = blk / 4, r4 = blk % 4;
    const int n = item / H, h = item % H;
    const int v0 = 32 * r4;  // first value column of this CTA
    const int64_t t0 = cu[n], t1 = cu[n + 1];
    const int nc = (int)((t1 - t0 + C - 1) / C);
    const size_t st = (size_t)D * D;
    // workspace record of chunk c: rec0 + c * REC_TC * H (the slot of chunk 0, read once)
    unsigned char *const rec0 = ws + (((size_t)(t0 >> 4) + (size_t)n) * H + h) * REC_TC;
    const size_t rstride = (size_t)H * REC_TC;
    auto full = [&](int s) { return static_cast<uint32_t>(__cvta_generic_to_shared(&bars[s])); };
    auto empty = [&](int s) { return static_cast<uint32_t>(__cvta_generic_to_shared(&bars[NS + s])); };
    // state-tile hand-off to the writer warp: staged[w][b] (chain warp w filled staging buffer
    // b), freed[w][b] (the writer's bulk copy has read it)
    auto staged = [&](int w, int b) { return static_cast<uint32_t>(__cvta_generic_to_shared(&bars[2 * NS + 2 * w + b])); };
    auto freed = [&](int w, int b) { return static_cast<uint32_t>(__cvta_generic_to_shared(&bars[2 * NS + 4 + 2 * w + b])); };
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            bar_init(full(s), 1);   // the copies' issue
            bar_init(empty(s), 2);  // one arrival per chain warp
        }
        for (int i = 0; i < 4; ++i) {
            bar_init(staged(i >> 1, i & 1), 1);
            bar_init(freed(i >> 1, i & 1), 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const uint32_t sbase0 = static_cast<uint32_t>(__cvta_generic_to_shared(smc));
    if (warp == 3) {
        // ---------------------------------------------------------------- writer warp
        // each chunk's two staged state tiles (16 rows per chain warp) to the workspace
        if (lane == 0) {
            for (int c = REVERSE ? nc - 1 : 0, m = 0; REVERSE ? c >= 0 : c < nc; c += REVERSE ? -1 : 1, ++m) {
                unsigned char *dst = rec0 + (size_t)c * rstride + (REVERSE ? TC_DS : TC_S);
                bool ok = true;
                for (int w = 0; w < 2 && ok; ++w) {
                    ok = bar_wait(staged(w, m & 1), (uint32_t)((m >> 1) & 1));
                    if (!ok) break;
                    const uint32_t src = sbase0 + NS * SLOT + (2 * w + (m & 1)) * CT_ROWS;
                    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                                 ::"l"(dst + (size_t)(v0 + 16 * w) * 272), "r"(src), "r"((uint32_t)CT_ROWS)
                                 : "memory");
                    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                    bar_arrive(freed(w, m & 1));
                }
                if (!ok) break;
            }
            asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        }
        return;
    }
    if (warp == 2) {
        // ---------------------------------------------------------------- loader warp
        for (int c = REVERSE ? nc - 1 : 0, m = 0; REVERSE ? c >= 0 : c < nc; c += REVERSE ? -1 : 1, ++m) {
            const int s = m % NS;
            bool ok = true;
            if (m >= NS) ok = bar_wait(empty(s), ((m / NS) & 1) ^ 1);
            if (!__all_sync(0xffffffffu, ok)) break;
            const uint32_t sl = static_cast<uint32_t>(__cvta_generic_to_shared(smc + s * SLOT));
            const unsigned char *tr = rec0 + (size_t)c * rstride + TC_REC;
            if (REVERSE) {  // K', -W, Q~, P, gamma_L; the chunk's dO rows, this CTA's 32 columns
                if (((sl + SL_X) & 127u) != 0) {  // a tensor copy needs 128-byte alignment:
                    if (lane == 0) atomicOr(&g_bwd_flags, 4u);  // report it (warp-uniform
                    break;                                      // exit; the waits give up)
                }
                if (lane == 0) {  // (rows past the sequence's end are masked where used)
                    bar_arrive_tx(full(s), TR_OPS + C * 32 * 2);
                    bulk_g2s(sl, tr, TR_OPS, full(s));
                    tma_load_3d(sl + SL_X, tm_dout, v0, h, (int)(t0 + (int64_t)c * C), full(s));
                }
            } else if (lane == 0) {  // K', -W; gamma_L; this CTA's block of U~^T
                bar_arrive_tx(full(s), 2 * T128 + 128 * 4 + 32 * C * 4);
                bulk_g2s(sl + SL_K, tr + TR_K, 2 * T128, full(s));
                bulk_g2s(sl + SL_G, tr + TR_G, 128 * 4, full(s));
                bulk_g2s(sl + SL_X, tr + TR_UT + r4 * 32 * C * 4, 32 * C * 4, full(s));
            }
        }
        return;
    }
    // -------------------------------------------------------------------- chain warps
    const int sw = warp, vr = v0 + 16 * sw;  // this warp's first value row of S^T
    const int g4 = lane >> 2, l4 = lane & 3, i8 = lane >> 3, r8 = lane & 7;
    const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(smc));
    float S[16][4];  // S^T (or dS^T) fragments: n-tile j = key channels 8j .. 8j + 7
    const size_t hidx = ((size_t)n * H + h) * st;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int kc = 8 * j + 2 * l4, v = vr + g4;
        if (init) {
            S[j][0] = init[hidx + (size_t)kc * D + v];
            S[j][1] = init[hidx + (size_t)(kc + 1) * D + v];
            S[j][2] = init[hidx + (size_t)kc * D + v + 8];
            S[j][3] = init[hidx + (size_t)(kc + 1) * D + v + 8];
        } else {
            S[j][0] = S[j][1] = S[j][2] = S[j][3] = 0.f;
        }
    }
    auto write_state = [&](float *dst) {  // fp32 [key][v] (the final state)
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int kc = 8 * j + 2 * l4, v = vr + g4;
            dst[(size_t)kc * D + v] = S[j][0];
            dst[(size_t)(kc + 1) * D + v] = S[j][1];
            dst[(size_t)kc * D + v + 8] = S[j][2];
            dst[(size_t)(kc + 1) * D + v + 8] = S[j][3];
        }
    };
    // this warp's 16 rows of the bf16 S^T tile [v][136]: staged in shared memory by
    // stmatrix (a double buffer per warp) and handed to the writer warp, which copies the
    // 4352 contiguous bytes to the workspace
    const uint32_t stage = sbase + NS * SLOT + sw * 2 * CT_ROWS;
    auto write_tile = [&](int m) {  // returns false when a wait gave up
        const int buf = m & 1;
        bool ok = true;
        if (m >= 2) ok = bar_wait(freed(sw, buf), (uint32_t)(((m >> 1) - 1) & 1));
        if (!__all_sync(0xffffffffu, ok)) return false;
        const uint32_t sb2 = stage + buf * CT_ROWS;
        const int mi = lane >> 3, r = lane & 7;
#pragma unroll
        for (int j = 0; j < 16; j += 2)
            stsm4(sb2 + (uint32_t)((((mi & 1) * 8 + r) * 136 + 8 * (j + (mi >> 1))) * 2),
                  pack2(S[j][0], S[j][1]), pack2(S[j][2], S[j][3]), pack2(S[j + 1][0], S[j + 1][1]),
                  pack2(S[j + 1][2], S[j + 1][3]));
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) bar_arrive(staged(sw, buf));  // release: the staging is written
        return true;
    };
    for (int c = REVERSE ? nc - 1 : 0, m = 0; REVERSE ? c >= 0 : c < nc; c += REVERSE ? -1 : 1, ++m) {
        const int s = m % NS;
        const bool ok = bar_wait(full(s), (m / NS) & 1);
        if (!__all_sync(0xffffffffu, ok)) break;
        const uint32_t sl = sbase + s * SLOT;
        const float4 *G4 = reinterpret_cast<const float4 *>(smc + s * SLOT + SL_G);
        if (!write_tile(m)) break;
        float acc[2][4];  // U^T (forward) or X^T (reverse): 16 value rows x 16 tokens
        if (!REVERSE) {
            const float *tu = reinterpret_cast<const float *>(smc + s * SLOT + SL_X);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int col = 8 * t + 2 * l4, row = 16 * sw + g4;
                acc[t][0] = tu[row * C + col];
                acc[t][1] = tu[row * C + col + 1];
                acc[t][2] = tu[(row + 8) * C + col];
                acc[t][3] = tu[(row + 8) * C + col + 1];
            }
        } else {
#pragma unroll
            for (int t = 0; t < 2; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
        }
        // (s dO)^T as the A fragment (reverse): 16 value rows x 16 tokens, read transposed
        uint32_t oa[4] = {0u, 0u, 0u, 0u};
        if (REVERSE) {
            ldsm4t(sl + SL_X + (uint32_t)((((i8 >> 1) * 8 + r8) + 0) * PO * 2 + (16 * sw + (i8 & 1) * 8) * 2), oa);
            const int64_t left = t1 - (t0 + (int64_t)c * C);  // valid token rows of the chunk
#pragma unroll
            for (int i = 0; i < 4; ++i) {  // s dO; tokens past the sequence's end to zero
                const int tk = (i >> 1) * 8 + 2 * l4;
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&oa[i]));
                oa[i] = pack2(tk < left ? scale * f.x : 0.f, tk + 1 < left ? scale * f.y : 0.f);
            }
        }
        // two independent accumulator chains (even / odd state tiles) halve the dependent
        // mma sequence of this product, the serial step's critical path
        float acc2[2][4] = {};
#pragma unroll
        for (int kt = 0; kt < 8; ++kt) {  // state tile kt against the chunk's 16 tokens
            uint32_t a[4];
            a[0] = pack2(S[2 * kt][0], S[2 * kt][1]);
            a[1] = pack2(S[2 * kt][2], S[2 * kt][3]);
            a[2] = pack2(S[2 * kt + 1][0], S[2 * kt + 1][1]);
            a[3] = pack2(S[2 * kt + 1][2], S[2 * kt + 1][3]);
            uint32_t bfr[4];
            // forward: B[k = channel][n = token] = -W[t][c]; reverse: = K'[t][c]; [n][k] storage
            ld_b_nk(sl + (REVERSE ? SL_K : SL_W), PB, 0, 16 * kt, bfr);
            float (&ac)[2][4] = (kt & 1) ? acc2 : acc;
            mma16816(ac[0], a, bfr[0], bfr[1]);
            mma16816(ac[1], a, bfr[2], bfr[3]);
        }
        if (REVERSE) {  // + (s dO)^T P: B[k = token i][n = token r] = P[i][r], [k][n] storage
            uint32_t bfr[4];
            ld_b_kn(sl + SL_P, PS, 0, 0, bfr);
            mma16816(acc2[0], oa, bfr[0], bfr[1]);
            mma16816(acc2[1], oa, bfr[2], bfr[3]);
        }
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[t][i] += acc2[t][i];
        uint32_t ua[4];  // U^T / X^T as the A fragment of the update
        ua[0] = pack2(acc[0][0], acc[0][1]);
        ua[1] = pack2(acc[0][2], acc[0][3]);
        ua[2] = pack2(acc[1][0], acc[1][1]);
        ua[3] = pack2(acc[1][2], acc[1][3]);
#pragma unroll
        for (int np = 0; np < 8; ++np) {  // key tile np: decay, then the chunk's write
            const float4 g = G4[np * 4 + l4];
            mul2(S[2 * np][0], S[2 * np][1], g.x, g.y);
            mul2(S[2 * np][2], S[2 * np][3], g.x, g.y);
            mul2(S[2 * np + 1][0], S[2 * np + 1][1], g.z, g.w);
            mul2(S[2 * np + 1][2], S[2 * np + 1][3], g.z, g.w);
            uint32_t bfr[4];
            // forward: U^T K' (B[k = token][n = channel] = K'[t][c]); reverse: X^T (-W)
            ld_b_kn(sl + (REVERSE ? SL_W : SL_K), PB, 0, 16 * np, bfr);
            mma16816(S[2 * np], ua, bfr[0], bfr[1]);
            mma16816(S[2 * np + 1], ua, bfr[2], bfr[3]);
            if (REVERSE) {  // + (s dO)^T Q~
                ld_b_kn(sl + SL_Q, PB, 0, 16 * np, bfr);
                mma16816(S[2 * np], oa, bfr[0], bfr[1]);
                mma16816(S[2 * np + 1], oa, bfr[2], bfr[3]);
            }
        }
        __syncwarp();
        if (lane == 0) bar_arrive(empty(s));  // this warp's reads of the slot are done
    }
    if (final_state) write_state(final_state + hidx);
}

// Both serial passes in one launch: they are independent (the reverse pass reads only the
// records and dO), and each leaves most of an SM idle. Blocks [0, nfwd) run the forward
// pass, the rest the reverse pass; two CTAs fit on an SM.
__global__ void __launch_bounds__(128, 2)
    chains_tc_kernel(const int32_t *__restrict__ cu, unsigned char *__restrict__ ws,
                     const __grid_constant__ CUtensorMap tm_dout, const float *__restrict__ h0,
                     const float *__restrict__ dh_final, float *__restrict__ dh0, int H,
                     float scale, int nfwd) {
    extern __shared__ __align__(128) unsigned char smc[];  // tensor copies land 128-byte aligned
    __shared__ __align__(8) unsigned long long bars[2 * NS + 8];
    if ((int)blockIdx.x < nfwd)
        chain_body<false>(blockIdx.x, smc, bars, cu, ws, &tm_dout, h0, nullptr, H, scale);
    else
        chain_body<true>(blockIdx.x - nfwd, smc, bars, cu, ws, &tm_dout, dh_final, dh0, H, scale);
}

// ---- 3. local gradients of every chunk
__host__ __device__ constexpr size_t local_mid_floats(int dk, int dv) {
    return (size_t)C * (dv + 1)                   // dO
           + (size_t)2 * dk * (JB + 1)            // S, dS_end column blocks
           + (size_t)2 * C * (JB + 1);            // U, dU column blocks
}
__host__ __device__ constexpr size_t local_floats(int dk, int dv) {
    return chunk_floats(dk, dv) + local_mid_floats(dk, dv)
           + (size_t)5 * C * (dk + 1)                   // dQ~, dW, dK', dK~, dK^
           + (size_t)4 * C * C                          // dP, dM, dT / Y, dA
           + dk + C;                                    // dgamma_L, dbeta
}

// fp32 FMA loops, the sums over value columns accumulated over 32-column blocks (any
// d_k, d_v <= 128; the tensor-core kernel below takes bf16 I/O at d_k = d_v = 128).
template <typename IO>
__global__ void __launch_bounds__(kThreads)
    local_kernel(const IO *__restrict__ q, const IO *__restrict__ k, const IO *__restrict__ v,
                 const float *__restrict__ a, const float *__restrict__ beta,
                 const int32_t *__restrict__ cu, const IO *__restrict__ dout,
                 const float *__restrict__ ck, const float *__restrict__ dck,
                 IO *__restrict__ dq, IO *__restrict__ dk_out, IO *__restrict__ dv_out,
                 float *__restrict__ da, float *__restrict__ dbeta, int H, int dk, int dv,
                 float scale) {
    extern __shared__ float sm[];
    const int tid = threadIdx.x, lk = dk + 1, lv = dv + 1, lj = JB + 1;
    const int n = blockIdx.x / H, h = blockIdx.x % H;
    const Chunk b = carve_chunk(sm, dk, dv);
    float *p = sm + chunk_floats(dk, dv);
    float *mid = p;
    p += local_mid_floats(dk, dv);
    float *dO = mid;
    float *Sb = dO + C * lv;
    float *dSb = Sb + dk * lj;
    float *Ub = dSb + dk * lj;
    float *dUb = Ub + C * lj;
    float *dQt = p; p += C * lk;
    float *dW = p; p += C * lk;
    float *dKp = p; p += C * lk;
    float *dKt = p; p += C * lk;
    float *dKh = p; p += C * lk;
    float *dP = p; p += C * C;
    float *dM = p; p += C * C;
    float *dT = p; p += C * C;
    float *dA = p; p += C * C;
    float *dgl = p; p += dk;
    float *db = p;
    const size_t st = (size_t)dk * dv;
    const int64_t t0 = cu[n], t1 = cu[n + 1];
    const int nc = (int)((t1 - t0 + C - 1) / C);
    for (int c = blockIdx.y; c < nc; c += gridDim.y) {
        const int64_t c0 = t0 + (int64_t)c * C;
        const int L = (int)(t1 - c0 < C ? t1 - c0 : C);
        prologue(b, q, k, v, a, beta, c0, L, H, h, dk, dv, true);
        const float *S = ck + (slot_of(cu, n, c) * H + h) * st;
        const float *dSe = dck + (slot_of(cu, n, c) * H + h) * st;
        for (int i = tid; i < C * dv; i += kThreads) {
            const int r = i / dv, j = i % dv;
            dO[r * lv + j] = r < L ? ld_io(dout, ((size_t)(c0 + r) * H + h) * dv + j) : 0.f;
        }
        for (int i = tid; i < C * dk; i += kThreads) {
            const int r = i / dk, x = i % dk;
            dQt[r * lk + x] = dW[r * lk + x] = dKp[r * lk + x] = 0.f;
        }
        for (int i = tid; i < dk; i += kThreads) dgl[i] = 0.f;
        float dp_acc = 0.f, dm_acc = 0.f;  // element tid of s dO U^T and dU V^T
        for (int j0 = 0; j0 < dv; j0 += JB) {
            const int w = dv - j0 < JB ? dv - j0 : JB;
            __syncthreads();  // previous block's readers are done
            for (int i = tid; i < dk * JB; i += kThreads) {
                const int x = i / JB, jj = i % JB;
                const bool in = jj < w;
                Sb[x * lj + jj] = in ? S[(size_t)x * dv + j0 + jj] : 0.f;
                dSb[x * lj + jj] = in ? dSe[(size_t)x * dv + j0 + jj] : 0.f;
            }
            __syncthreads();
            for (int i = tid; i < C * JB; i += kThreads) {  // U and dU of this block
                const int r = i / JB, jj = i % JB;
                float u = 0.f, du = 0.f;
                if (jj < w) {
                    const int j = j0 + jj;
                    u = b.Ut[r * lv + j];
                    for (int x = 0; x < dk; ++x) {
                        u = fmaf(-b.W[r * lk + x], Sb[x * lj + jj], u);
                        du = fmaf(b.Kp[r * lk + x], dSb[x * lj + jj], du);
                    }
                    float pd = 0.f;
                    for (int i2 = r; i2 < C; ++i2) pd = fmaf(b.P[i2 * C + r], dO[i2 * lv + j], pd);
                    du = fmaf(scale, pd, du);
                }
                Ub[r * lj + jj] = u;
                dUb[r * lj + jj] = du;
            }
            __syncthreads();
            for (int i = tid; i < C * JB; i += kThreads) {  // dV = M^T dU
                const int r = i / JB, jj = i % JB;
                if (r < L && jj < w) {
                    float acc = 0.f;
#pragma unroll
                    for (int i2 = 0; i2 < C; ++i2) acc = fmaf(b.M[i2 * C + r], dUb[i2 * lj + jj], acc);
                    st_io(dv_out, ((size_t)(c0 + r) * H + h) * dv + j0 + jj, acc);
                }
            }
            for (int i = tid; i < C * dk; i += kThreads) {  // sums over this block's columns
                const int r = i / dk, x = i % dk;
                float qs = 0.f, ws = 0.f, kp = 0.f;
                for (int jj = 0; jj < w; ++jj) {
                    const float s = Sb[x * lj + jj];
                    qs = fmaf(dO[r * lv + j0 + jj], s, qs);
                    ws = fmaf(dUb[r * lj + jj], s, ws);
                    kp = fmaf(Ub[r * lj + jj], dSb[x * lj + jj], kp);
                }
                dQt[r * lk + x] += scale * qs;
                dW[r * lk + x] -= ws;
                dKp[r * lk + x] += kp;
            }
            for (int x = tid; x < dk; x += kThreads) {
                float acc = 0.f;
                for (int jj = 0; jj < w; ++jj) acc = fmaf(dSb[x * lj + jj], Sb[x * lj + jj], acc);
                dgl[x] += acc;
            }
            {
                const int r = tid / C, i2 = tid % C;
                float pa = 0.f, ma = 0.f;
                for (int jj = 0; jj < w; ++jj) {
                    pa = fmaf(dO[r * lv + j0 + jj], Ub[i2 * lj + jj], pa);
                    ma = fmaf(dUb[r * lj + jj], b.V[i2 * lv + j0 + jj], ma);
                }
                dp_acc = fmaf(scale, pa, dp_acc);
                dm_acc += ma;
            }
        }
        {
            const int r = tid / C, i2 = tid % C;
            dP[r * C + i2] = i2 <= r ? dp_acc : 0.f;
            dM[r * C + i2] = dm_acc;
        }
        __syncthreads();
        for (int i = tid; i < C * dk; i += kThreads) {  // dQ~ += dP K^
            const int r = i / dk, x = i % dk;
            float acc = 0.f;
            for (int i2 = 0; i2 <= r; ++i2) acc = fmaf(dP[r * C + i2], b.Kh[i2 * lk + x], acc);
            dQt[r * lk + x] += acc;
        }
        {  // dM += dW K~^T
            const int r = tid / C, j = tid % C;
            float acc = 0.f;
            for (int x = 0; x < dk; ++x) acc = fmaf(dW[r * lk + x], b.Kt[j * lk + x], acc);
            dM[r * C + j] += acc;
        }
        __syncthreads();
        {  // dT = dM diag(beta)
            const int r = tid / C, j = tid % C;
            dT[r * C + j] = dM[r * C + j] * b.bt[j];
        }
        if (tid < C) {  // dbeta from M = T diag(beta)
            float acc = 0.f;
            for (int i2 = 0; i2 < C; ++i2) acc = fmaf(dM[i2 * C + tid], b.T[i2 * C + tid], acc);
            db[tid] = acc;
        }
        __syncthreads();
        {  // Y = dT T^T (into dA)
            const int r = tid / C, j = tid % C;
            float acc = 0.f;
#pragma unroll
            for (int l = 0; l < C; ++l) acc = fmaf(dT[r * C + l], b.T[j * C + l], acc);
            dA[r * C + j] = acc;
        }
        __syncthreads();
        {  // dA = strict_lower(-T^T Y), then dZ = diag(beta) dA (into dT)
            const int r = tid / C, j = tid % C;
            float acc = 0.f;
#pragma unroll
            for (int l = 0; l < C; ++l) acc = fmaf(b.T[l * C + r], dA[l * C + j], acc);
            const float d = j < r ? -acc : 0.f;
            __syncthreads();
            dA[r * C + j] = d;
            dT[r * C + j] = b.bt[r] * d;
        }
        __syncthreads();
        if (tid < C) {  // dbeta from A = strict_lower(diag(beta) Z)
            float acc = 0.f;
            for (int j = 0; j < tid; ++j) acc = fmaf(dA[tid * C + j], b.Z[tid * C + j], acc);
            db[tid] += acc;
        }
        for (int i = tid; i < C * dk; i += kThreads) {  // dK~ and dK^
            const int r = i / dk, x = i % dk;
            float kt = 0.f, kh = 0.f;
#pragma unroll
            for (int i2 = 0; i2 < C; ++i2) {
                kt = fmaf(b.M[i2 * C + r], dW[i2 * lk + x], kt);
                kt = fmaf(dT[r * C + i2], b.Kh[i2 * lk + x], kt);
                kh = fmaf(dP[i2 * C + r], b.Qt[i2 * lk + x], kh);
                kh = fmaf(dT[i2 * C + r], b.Kt[i2 * lk + x], kh);
            }
            dKt[r * lk + x] = kt;
            dKh[r * lk + x] = kh;
        }
        __syncthreads();
        if (tid < L) dbeta[(size_t)(c0 + tid) * H + h] = db[tid];
        for (int x = tid; x < dk; x += kThreads) {  // per key channel: dq, dk, the log-decay
            float dG[C];
            float kpsum = 0.f;
            const float GL = b.Gs[(C - 1) * lk + x];
#pragma unroll
            for (int r = 0; r < C; ++r) {
                const float Gr = b.Gs[r * lk + x];
                const float qt = dQt[r * lk + x], kt = dKt[r * lk + x], kh = dKh[r * lk + x],
                            kp = dKp[r * lk + x];
                const float kpk = kp * b.Kp[r * lk + x];
                dG[r] = qt * b.Qt[r * lk + x] + kt * b.Kt[r * lk + x] - kh * b.Kh[r * lk + x] - kpk;
                kpsum += kpk;
                if (r < L) {
                    const size_t o = ((size_t)(c0 + r) * H + h) * dk + x;
                    st_io(dq, o, qt * expf(Gr));
                    st_io(dk_out, o, kt * expf(Gr) + kh * expf(-Gr) + kp * expf(GL - Gr));
                }
            }
            dG[C - 1] += b.gl[x] * dgl[x] + kpsum;
            float acc = 0.f;
#pragma unroll
            for (int r = C - 1; r >= 0; --r) {
                acc += dG[r];
                if (r < L) {
                    const size_t o = ((size_t)(c0 + r) * H + h) * dk + x;
                    const float sg = 1.f / (1.f + expf(-a[o]));
                    da[o] = acc * (kGMin * sg * (1.f - sg));
                }
            }
        }
    }
}

// ---- 3b. local gradients on the tensor cores (bf16 I/O, d_k = d_v = 128)
// One CTA per SM walks a contiguous range of items (chunk slot, head), flat index slot H + h.
// Per item it bulk-copies the two bf16 state tiles and the prep record into shared memory:
// the record, with the item's V and dO rows, one item ahead into a second buffer; the
// states as soon as the previous item's last reader of them is done (prefetched into L2 an
// item ahead). Every product runs on mma.sync (bf16 operands, fp32 accumulation). Warp w
// owns value columns [16 w, 16 w + 16) in phase 1 (U, dU, dV) and key channels [16 w,
// 16 w + 16) in phases 2 and 4 (dQ~, dK', dW, dgamma_L, dK~, dK^ and the per-channel
// gradients dq, dk, da, computed on the accumulator fragments); the 16 x 16 adjoint of the
// solve (phase 3) is one element per thread.
// Phase stamps of the local-gradient kernel (CTA 0, thread 0, first 64 items), compiled
// only with -DKDA_BWD_TRACE.
#ifdef KDA_BWD_TRACE
__device__ long long g_local_trace[64][9];
#define LOCAL_TRACE(i) \
    do { \
        if (blockIdx.x == 0 && tid == 0 && m < 64) g_local_trace[m][i] = clock64(); \
    } while (0)
#else
#define LOCAL_TRACE(i) \
    do { \
    } while (0)
#endif
constexpr int LT_THREADS = 256;
// record buffer: V and dO rows as two 128-byte-swizzled [16][64] halves each (tensor
// copies, 1024-byte aligned), then the record
constexpr int SWT = C * 128 * 2;        // a swizzled [16][128] bf16 tile
constexpr int RBUF = ((2 * SWT + RECB) + 1023) / 1024 * 1024;
constexpr int LS_S = 0, LS_DS = ST16, LS_R = 2 * ST16;
constexpr int LS_U = LS_R + 2 * RBUF, LS_DU = LS_U + T128, LS_DW = LS_DU + T128;
constexpr int LS_DP = LS_DW + T128, LS_DZ = LS_DP + C * PS * 2;
constexpr int LS_PART = LS_DZ + C * PS * 2;  // per warp: dM, dP partial sums [2][16][16]
constexpr int LS_DT = LS_PART + 8 * 2 * C * C * 4, LS_DMS = LS_DT + C * C * 4, LS_Y = LS_DMS + C * C * 4;
constexpr int LS_DB = LS_Y + C * C * 4;
constexpr int LS_BYTES = LS_DB + C * 4;
static_assert(RBUF % 1024 == 0 && LS_R % 1024 == 0 && LS_U % 16 == 0 && LS_DP % 16 == 0 &&
                  LS_BYTES <= 227 * 1024,
              "local tensor-core kernel shared memory");
static_assert(LT_THREADS == C * C, "one thread per element of a 16 x 16 product");

struct Item {
    int n, h, c;
    int L;           // the chunk's token rows (<= 16)
    int64_t c0;      // its first token
    long long slot;  // its workspace slot
};
// item idx = slot H + h; false when the slot holds no chunk (the gap after a sequence)
__device__ bool decode_item(const int32_t *cu, int n_seq, int H, long long idx, Item &it) {
    const long long slot = idx / H;
    it.h = (int)(idx - slot * H);
    int lo = 0, hi = n_seq - 1;  // the last sequence whose first slot is <= slot
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((long long)(cu[mid] >> 4) + mid <= slot) lo = mid;
        else hi = mid - 1;
    }
    it.n = lo;
    it.c = (int)(slot - ((long long)(cu[lo] >> 4) + lo));
    return it.c < (cu[lo + 1] - cu[lo] + C - 1) / C;
}
// Walks items idx = slot H + h in increasing order: one division and binary search at the
// start, then a step per item (the next sequence's slots looked up as they are reached);
// items of slots that hold no chunk are skipped.
struct ItemCursor {
    const int32_t *cu;
    int n_seq, H, h, n, nc;
    long long idx, end, slot, b0, b1;  // b0, b1: the first slots of sequences n and n + 1
    int64_t tok0, tok1;                // sequence n's tokens [tok0, tok1)
    __device__ void load_seq() {
        tok0 = cu[n];
        tok1 = cu[n + 1];
        b0 = (long long)(tok0 >> 4) + n;
        b1 = n + 1 < n_seq ? (long long)(tok1 >> 4) + n + 1 : LLONG_MAX;
        nc = (int)((tok1 - tok0 + C - 1) / C);
    }
    __device__ void start(const int32_t *cu_, int n_seq_, int H_, long long beg, long long end_) {
        cu = cu_;
        n_seq = n_seq_;
        H = H_;
        end = end_;
        idx = beg;
        slot = beg / H;
        h = (int)(beg - slot * H);
        Item it;
        decode_item(cu, n_seq, H, beg, it);
        n = it.n;
        load_seq();
        skip();
    }
    __device__ void step() {
        ++idx;
        if (++h == H) {
            h = 0;
            ++slot;
            while (slot >= b1) {
                ++n;
                load_seq();
            }
        }
    }
    __device__ void skip() {
        while (idx < end && slot - b0 >= nc) step();
    }
    __device__ void advance() {
        step();
        skip();
    }
    // the current item, with its rows, first token and slot (no memory access)
    __device__ Item item() const {
        Item it;
        it.n = n;
        it.h = h;
        it.c = (int)(slot - b0);
        it.c0 = tok0 + (int64_t)it.c * C;
        const int64_t left = tok1 - it.c0;
        it.L = (int)(left < C ? left : C);
        it.slot = slot;
        return it;
    }
};

__global__ void __launch_bounds__(LT_THREADS, 1)
    local_tc_kernel(const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_a,
                    const float *__restrict__ a,
                    const int32_t *__restrict__ cu, const __grid_constant__ CUtensorMap tm_dout,
                    const unsigned char *__restrict__ ws, __nv_bfloat16 *__restrict__ dq,
                    __nv_bfloat16 *__restrict__ dk_out, __nv_bfloat16 *__restrict__ dv_out,
                    float *__restrict__ da, float *__restrict__ dbeta, int H, int n_seq,
                    long long n_items, float scale) {
    constexpr int D = 128;
    extern __shared__ __align__(1024) unsigned char sl[];  // 128-byte-swizzled tensor copies
    __shared__ __align__(8) unsigned long long bars[3];  // states; record buffers 0, 1
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g4 = lane >> 2, l4 = lane & 3, n0 = 16 * warp;
    const long long beg = (long long)blockIdx.x * n_items / gridDim.x;
    const long long end = (long long)(blockIdx.x + 1) * n_items / gridDim.x;
    const uint32_t sb = static_cast<uint32_t>(__cvta_generic_to_shared(sl));
    auto bar = [&](int i) { return static_cast<uint32_t>(__cvta_generic_to_shared(&bars[i])); };
    float *part = reinterpret_cast<float *>(sl + LS_PART);
    float *dTs = reinterpret_cast<float *>(sl + LS_DT), *dMs = reinterpret_cast<float *>(sl + LS_DMS);
    float *Ys = reinterpret_cast<float *>(sl + LS_Y), *dbs = reinterpret_cast<float *>(sl + LS_DB);
    __nv_bfloat16 *dP16 = reinterpret_cast<__nv_bfloat16 *>(sl + LS_DP);
    __nv_bfloat16 *dZ16 = reinterpret_cast<__nv_bfloat16 *>(sl + LS_DZ);
    if (tid == 0) {
        for (int i = 0; i < 3; ++i) bar_init(bar(i), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    auto rec_of = [&](const Item &it) { return ws + ((size_t)it.slot * H + it.h) * REC_TC; };
    // one thread: the V and dO rows of item it (four tensor copies: two 64-column halves
    // each) and its record into record buffer rb
    auto issue_rec = [&](const Item &it, int rb) {
        const int64_t c0 = it.c0;
        const uint32_t bb = sb + LS_R + rb * RBUF;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        bar_arrive_tx(bar(1 + rb), (uint32_t)(2 * SWT + RECB));
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            tma_load_3d(bb + x * (SWT / 2), &tm_v, 64 * x, it.h, (int)c0, bar(1 + rb));
            tma_load_3d(bb + SWT + x * (SWT / 2), &tm_dout, 64 * x, it.h, (int)c0, bar(1 + rb));
        }
        bulk_g2s(bb + 2 * SWT, rec_of(it) + TC_REC, RECB, bar(1 + rb));
    };
    auto issue_states = [&](const Item &it) {  // one thread: S and dS_end, adjacent both sides
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        bar_arrive_tx(bar(0), 2 * ST16);
        bulk_g2s(sb + LS_S, rec_of(it) + TC_S, 2 * ST16, bar(0));
    };
    // one thread: the next item's states and gate-logit rows into L2
    auto prefetch_next = [&](const Item &it) {
        prefetch_l2(rec_of(it) + TC_S, 2 * ST16);
        tma_prefetch_3d(&tm_a, 0, it.h, (int)it.c0);
    };

    ItemCursor ic;
    ic.start(cu, n_seq, H, beg, end);
    Item cur = ic.item(), nxt;
    long long idx = ic.idx;
    if (idx < end && tid == 0) {
        issue_rec(cur, 0);
        issue_states(cur);
    }

    for (int m = 0; idx < end; ++m) {
        ic.advance();
        const long long nidx = ic.idx;
        nxt = ic.item();
        const bool more = nidx < end;
        __syncthreads();  // the other record buffer's readers (the previous item) are done
        if (more) {
            if (tid == 0) issue_rec(nxt, (m + 1) & 1);
            else if (tid == 32) prefetch_next(nxt);
        }
        const int rb = m & 1;
        LOCAL_TRACE(0);
        const bool ok = bar_wait(bar(1 + rb), (uint32_t)((m >> 1) & 1)) && bar_wait(bar(0), (uint32_t)(m & 1));
        if (__syncthreads_or(!ok)) break;
        LOCAL_TRACE(1);
        const int64_t c0 = cur.c0;
        const int L = cur.L;
        const int h = cur.h;
        const unsigned char *R = sl + LS_R + rb * RBUF + 2 * SWT;  // the record
        const uint32_t rbase = sb + LS_R + rb * RBUF + 2 * SWT;
        if (L < C) {  // V, dO rows past the sequence's end (other tokens, or zeros) to zero
            unsigned char *t2 = sl + LS_R + rb * RBUF;
            for (int i = tid; i < 2 * 2 * (C - L) * 8; i += LT_THREADS) {  // [tile][half][row][chunk]
                const int chunk = i & 7, row = L + (i >> 3) % (C - L), hv = (i >> 3) / (C - L);
                *reinterpret_cast<uint4 *>(t2 + hv * (SWT / 2) + row * 128 + chunk * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // before its next copy
            __syncthreads();
        }
        const uint32_t SB = sb + LS_S, DSB = sb + LS_DS;
        const uint32_t KP = rbase + TR_K, WN = rbase + TR_W, QT = rbase + TR_Q, P16 = rbase + TR_P;
        const uint32_t KT = rbase + TR_KT, KH = rbase + TR_KH, M16 = rbase + TR_M;
        const uint32_t V16 = sb + LS_R + rb * RBUF, DO = V16 + SWT;  // swizzled tiles
        const uint32_t U16 = sb + LS_U, DU16 = sb + LS_DU, DW16 = sb + LS_DW;
        const uint32_t DP = sb + LS_DP, DZ = sb + LS_DZ;

        // the gate logits phase 4 needs (prefetched into L2 an item ahead): issued now, so
        // that their latency passes under phases 1-3
        float2 av[2][2];
#pragma unroll
        for (int tt = 0; tt < 2; ++tt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int t = g4 + 8 * hh;
                av[tt][hh] = make_float2(0.f, 0.f);
                if (t < L)
                    av[tt][hh] = *reinterpret_cast<const float2 *>(
                        a + ((size_t)(c0 + t) * H + h) * D + n0 + 8 * tt + 2 * l4);
            }

        LOCAL_TRACE(2);
        // ---- phase 1 (value columns [n0, n0 + 16)): U = U~ - W S, dU = K' dS_end + s P^T dO,
        // dV = M^T dU; partial sums of dO U^T and dU V^T over these columns
        float u[2][4], du[2][4] = {}, dpp[2][4] = {}, dmp[2][4] = {};
        {
            const float *Ut = reinterpret_cast<const float *>(R + TR_UT);  // [v][16 t]
#pragma unroll
            for (int tt = 0; tt < 2; ++tt) {
                const int vc = n0 + 8 * tt + 2 * l4;
                u[tt][0] = Ut[vc * C + g4];
                u[tt][1] = Ut[(vc + 1) * C + g4];
                u[tt][2] = Ut[vc * C + g4 + 8];
                u[tt][3] = Ut[(vc + 1) * C + g4 + 8];
            }
#pragma unroll
            for (int k0 = 0; k0 < D; k0 += 16) {  // k = key channel
                uint32_t aw[4], ak[4], bs[4], bd[4];
                ld_a(WN, PB, k0, aw);
                ld_a(KP, PB, k0, ak);
                ld_b_nk(SB, PB, n0, k0, bs);   // B[key][v] = S^T tile [v][key]
                ld_b_nk(DSB, PB, n0, k0, bd);
                mma16816(u[0], aw, bs[0], bs[1]);
                mma16816(u[1], aw, bs[2], bs[3]);
                mma16816(du[0], ak, bd[0], bd[1]);
                mma16816(du[1], ak, bd[2], bd[3]);
            }
            uint32_t ap[4], bo[4];
            float pd[2][4] = {};
            ld_a_t(P16, PS, 0, 0, ap);         // P^T
            ld_b_kn_sw(DO, 0, n0, bo);         // B[i][v] = dO[i][v]
            mma16816(pd[0], ap, bo[0], bo[1]);
            mma16816(pd[1], ap, bo[2], bo[3]);
#pragma unroll
            for (int tt = 0; tt < 2; ++tt)
#pragma unroll
                for (int i = 0; i < 4; ++i) du[tt][i] = fmaf(scale, pd[tt][i], du[tt][i]);
            store_c16(reinterpret_cast<__nv_bfloat16 *>(sl + LS_U), PB, n0, u);
            store_c16(reinterpret_cast<__nv_bfloat16 *>(sl + LS_DU), PB, n0, du);
            // dO[:, cols] U[:, cols]^T: U's accumulator fragments are the B operand as they are
            uint32_t ao[4];
            ld_a_sw(DO, n0, ao);
            mma16816(dpp[0], ao, pack2(u[0][0], u[0][1]), pack2(u[1][0], u[1][1]));
            mma16816(dpp[1], ao, pack2(u[0][2], u[0][3]), pack2(u[1][2], u[1][3]));
            // dU[:, cols] V[:, cols]^T: dU's fragments are the A operand as they are
            const uint32_t adu[4] = {pack2(du[0][0], du[0][1]), pack2(du[0][2], du[0][3]),
                                     pack2(du[1][0], du[1][1]), pack2(du[1][2], du[1][3])};
            uint32_t bv[4];
            ld_b_nk_sw(V16, 0, n0, bv);        // B[v][t'] = V[t'][v]
            mma16816(dmp[0], adu, bv[0], bv[1]);
            mma16816(dmp[1], adu, bv[2], bv[3]);
            __syncwarp();  // this warp's dU columns are in shared memory
            uint32_t am[4], bu[4];
            float dvf[2][4] = {};
            ld_a_t(M16, PS, 0, 0, am);         // M^T
            ld_b_kn(DU16, PB, 0, n0, bu);
            mma16816(dvf[0], am, bu[0], bu[1]);
            mma16816(dvf[1], am, bu[2], bu[3]);
#pragma unroll
            for (int tt = 0; tt < 2; ++tt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int t = g4 + 8 * hh;
                    if (t < L)
                        *reinterpret_cast<uint32_t *>(
                            dv_out + ((size_t)(c0 + t) * H + h) * D + n0 + 8 * tt + 2 * l4) =
                            pack2(dvf[tt][2 * hh], dvf[tt][2 * hh + 1]);
                }
        }
        LOCAL_TRACE(3);
        __syncthreads();  // U and dU complete
        LOCAL_TRACE(4);

        // ---- phase 2 (key channels [n0, n0 + 16)): dQ~ = s dO S^T, dK' = U dS_end^T,
        // dW = -dU S^T, dgamma_L = diag(dS_end S^T); dW K~^T into the dM partial sum
        float dqa[2][4] = {}, dkp[2][4] = {}, dwa[2][4] = {}, dga[2][4] = {};
#pragma unroll
        for (int k0 = 0; k0 < D; k0 += 16) {  // k = value column
            uint32_t ao[4], au[4], adu[4], ads[4], bs[4], bd[4];
            ld_a_sw(DO, k0, ao);
            ld_a(U16, PB, k0, au);
            ld_a(DU16, PB, k0, adu);
            ld_b_kn(SB, PB, k0, n0, bs);       // B[v][key] = S^T tile [v][key]
            ld_b_kn(DSB, PB, k0, n0, bd);
            ld_a_t(DSB, PB, k0, n0, ads);      // A[key][v] = dS_end[key][v]
            mma16816(dqa[0], ao, bs[0], bs[1]);
            mma16816(dqa[1], ao, bs[2], bs[3]);
            mma16816(dkp[0], au, bd[0], bd[1]);
            mma16816(dkp[1], au, bd[2], bd[3]);
            mma16816(dwa[0], adu, bs[0], bs[1]);
            mma16816(dwa[1], adu, bs[2], bs[3]);
            mma16816(dga[0], ads, bs[0], bs[1]);
            mma16816(dga[1], ads, bs[2], bs[3]);
        }
#pragma unroll
        for (int tt = 0; tt < 2; ++tt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                dqa[tt][i] *= scale;
                dwa[tt][i] = -dwa[tt][i];
            }
        // dgamma_L: the diagonal of dga sits on lanes g4 >> 1 == l4; lane 9 l4 holds keys
        // n0 + 2 l4 and n0 + 8 + 2 l4, lane 9 l4 + 4 the keys one above
        float dgl[2][2];
        {
            const float d0 = (g4 & 1) ? dga[0][1] : dga[0][0];
            const float d1 = (g4 & 1) ? dga[1][3] : dga[1][2];
            dgl[0][0] = __shfl_sync(0xffffffffu, d0, 9 * l4);
            dgl[0][1] = __shfl_sync(0xffffffffu, d0, 9 * l4 + 4);
            dgl[1][0] = __shfl_sync(0xffffffffu, d1, 9 * l4);
            dgl[1][1] = __shfl_sync(0xffffffffu, d1, 9 * l4 + 4);
        }
        {
            const uint32_t aw[4] = {pack2(dwa[0][0], dwa[0][1]), pack2(dwa[0][2], dwa[0][3]),
                                    pack2(dwa[1][0], dwa[1][1]), pack2(dwa[1][2], dwa[1][3])};
            uint32_t bk[4];
            ld_b_nk(KT, PB, 0, n0, bk);        // B[key][t'] = K~[t'][key]
            mma16816(dmp[0], aw, bk[0], bk[1]);
            mma16816(dmp[1], aw, bk[2], bk[3]);
            store_c16(reinterpret_cast<__nv_bfloat16 *>(sl + LS_DW), PB, n0, dwa);
            float *pw = part + warp * 2 * C * C;  // summed in warp order (deterministic)
#pragma unroll
            for (int tt = 0; tt < 2; ++tt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int e = (g4 + 8 * hh) * C + 8 * tt + 2 * l4;
                    *reinterpret_cast<float2 *>(pw + e) = make_float2(dmp[tt][2 * hh], dmp[tt][2 * hh + 1]);
                    *reinterpret_cast<float2 *>(pw + C * C + e) =
                        make_float2(dpp[tt][2 * hh], dpp[tt][2 * hh + 1]);
                }
        }
        LOCAL_TRACE(5);
        __syncthreads();  // the states' last readers are done; dM and dP sums complete
        LOCAL_TRACE(6);
        if (more && tid == 0) issue_states(nxt);

        // ---- phase 3: dP = s lower(dO U^T); dT = dM diag(beta), dA = strict_lower(-T^T dT
        // T^T), dZ = diag(beta) dA; dbeta
        const float *T = reinterpret_cast<const float *>(R + TR_T);
        const float *TT = reinterpret_cast<const float *>(R + TR_TT);
        const float *Z = reinterpret_cast<const float *>(R + TR_Z);
        const float *BT = reinterpret_cast<const float *>(R + TR_B);
        {
            const int r = tid >> 4, j = tid & 15;
            float dm = 0.f, dp = 0.f;
#pragma unroll
            for (int w = 0; w < LT_THREADS / 32; ++w) {
                dm += part[w * 2 * C * C + tid];
                dp += part[w * 2 * C * C + C * C + tid];
            }
            dP16[r * PS + j] = __float2bfloat16_rn(j <= r ? scale * dp : 0.f);
            dTs[tid] = dm * BT[j];
            dMs[tid] = dm;
        }
        __syncthreads();
        {
            const int r = tid >> 4, j = tid & 15;
            float y = 0.f;
#pragma unroll
            for (int l = 0; l < C; ++l) y = fmaf(dTs[r * C + l], TT[l * C + j], y);  // (dT T^T)_rj
            Ys[tid] = y;
            if (tid < C) {  // dbeta from M = T diag(beta)
                float acc = 0.f;
#pragma unroll
                for (int i = 0; i < C; ++i) acc = fmaf(dMs[i * C + tid], T[i * C + tid], acc);
                dbs[tid] = acc;
            }
        }
        __syncthreads();
        {
            const int r = tid >> 4, j = tid & 15;
            float acc = 0.f;
#pragma unroll
            for (int l = 0; l < C; ++l) acc = fmaf(T[l * C + r], Ys[l * C + j], acc);
            const float dA = j < r ? -acc : 0.f;
            dZ16[r * PS + j] = __float2bfloat16_rn(BT[r] * dA);
            float x = dA * Z[tid];  // dbeta from A = strict_lower(diag(beta) Z)
#pragma unroll
            for (int o = 1; o < C; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
            if (j == 0 && r < L) dbeta[(size_t)(c0 + r) * H + h] = dbs[r] + x;
        }
        __syncthreads();  // dP, dZ complete
        LOCAL_TRACE(7);

        // ---- phase 4 (key channels [n0, n0 + 16)): dQ~ += dP K^, dK~ = M^T dW + dZ K^,
        // dK^ = dP^T Q~ + dZ^T K~; then dq, dk and da on the fragments. dG takes Q~, K~, K^
        // and K' as the bf16 values the products above used: its terms cancel pairwise
        // across rows (dP_ri Q~_r K^_i enters row r through dQ~ and row i through dK^, and
        // likewise for dZ), exactly only with the same operand values on both sides.
        float dkt[2][4] = {}, dkh[2][4] = {};
        {
            uint32_t bkh[4], bb[4], af[4];
            ld_b_kn(KH, PB, 0, n0, bkh);       // B[t'][key] = K^[t'][key]
            ld_a(DP, PS, 0, af);               // dP
            mma16816(dqa[0], af, bkh[0], bkh[1]);
            mma16816(dqa[1], af, bkh[2], bkh[3]);
            ld_a(DZ, PS, 0, af);               // dZ
            mma16816(dkt[0], af, bkh[0], bkh[1]);
            mma16816(dkt[1], af, bkh[2], bkh[3]);
            ld_a_t(M16, PS, 0, 0, af);         // M^T
            ld_b_kn(DW16, PB, 0, n0, bb);      // B[t'][key] = dW[t'][key]
            mma16816(dkt[0], af, bb[0], bb[1]);
            mma16816(dkt[1], af, bb[2], bb[3]);
            ld_a_t(DP, PS, 0, 0, af);          // dP^T
            ld_b_kn(QT, PB, 0, n0, bb);
            mma16816(dkh[0], af, bb[0], bb[1]);
            mma16816(dkh[1], af, bb[2], bb[3]);
            ld_a_t(DZ, PS, 0, 0, af);          // dZ^T
            ld_b_kn(KT, PB, 0, n0, bb);
            mma16816(dkh[0], af, bb[0], bb[1]);
            mma16816(dkh[1], af, bb[2], bb[3]);
        }
        const float *GS = reinterpret_cast<const float *>(R + TR_GS);
        const float *GLv = reinterpret_cast<const float *>(R + TR_GL);
        float dG[2][4], kps[2][2] = {};
#pragma unroll
        for (int tt = 0; tt < 2; ++tt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int t = g4 + 8 * hh, key = n0 + 8 * tt + 2 * l4;
                auto tile2 = [&](int off) {
                    return __bfloat1622float2(
                        *reinterpret_cast<const __nv_bfloat162 *>(R + off + (t * 136 + key) * 2));
                };
                const float2 q2 = tile2(TR_Q), t2 = tile2(TR_KT), h2 = tile2(TR_KH), p2 = tile2(TR_K);
                float oq[2], ok2[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int fi = 2 * hh + e;
                    const float G = GS[t * GP + key + e], GL = GS[(C - 1) * GP + key + e];
                    const float eg = __expf(G), en = __expf(-G), ep = __expf(GL - G);
                    const float Qt = e ? q2.y : q2.x, Kt = e ? t2.y : t2.x;
                    const float Kh = e ? h2.y : h2.x, Kp = e ? p2.y : p2.x;
                    const float gq = dqa[tt][fi], gt = dkt[tt][fi], gh = dkh[tt][fi], gp = dkp[tt][fi];
                    oq[e] = gq * eg;
                    ok2[e] = gt * eg + gh * en + gp * ep;
                    dG[tt][fi] = gq * Qt + gt * Kt - gh * Kh - gp * Kp;
                    kps[tt][e] += gp * Kp;
                }
                if (t < L) {
                    const size_t o = ((size_t)(c0 + t) * H + h) * D + key;
                    *reinterpret_cast<uint32_t *>(dq + o) = pack2(oq[0], oq[1]);
                    *reinterpret_cast<uint32_t *>(dk_out + o) = pack2(ok2[0], ok2[1]);
                }
            }
#pragma unroll
        for (int tt = 0; tt < 2; ++tt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float x = kps[tt][e];  // colsum over the 16 rows of dK' K'
                x += __shfl_xor_sync(0xffffffffu, x, 4);
                x += __shfl_xor_sync(0xffffffffu, x, 8);
                x += __shfl_xor_sync(0xffffffffu, x, 16);
                const int key = n0 + 8 * tt + 2 * l4 + e;
                if (g4 == 7) dG[tt][2 + e] += GLv[key] * dgl[tt][e] + x;  // row 15
                // reverse cumulative sum over the rows: g4 + 8 (hi), then g4 (lo)
                float hi = dG[tt][2 + e], lo = dG[tt][e];
#pragma unroll
                for (int d = 1; d < 8; d <<= 1) {
                    const float yh = __shfl_down_sync(0xffffffffu, hi, 4 * d);
                    const float yl = __shfl_down_sync(0xffffffffu, lo, 4 * d);
                    if (g4 + d < 8) {
                        hi += yh;
                        lo += yl;
                    }
                }
                lo += __shfl_sync(0xffffffffu, hi, l4);
                dG[tt][2 + e] = hi;
                dG[tt][e] = lo;
            }
#pragma unroll
        for (int tt = 0; tt < 2; ++tt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int t = g4 + 8 * hh;
                if (t < L) {
                    const float2 ax = av[tt][hh];
                    const float s0 = __fdividef(1.f, 1.f + __expf(-ax.x));
                    const float s1 = __fdividef(1.f, 1.f + __expf(-ax.y));
                    const size_t o = ((size_t)(c0 + t) * H + h) * D + n0 + 8 * tt + 2 * l4;
                    *reinterpret_cast<float2 *>(da + o) =
                        make_float2(dG[tt][2 * hh] * (kGMin * s0 * (1.f - s0)),
                                    dG[tt][2 * hh + 1] * (kGMin * s1 * (1.f - s1)));
                }
            }
        LOCAL_TRACE(8);
        idx = nidx;
        cur = nxt;
    }
}

// ---- 0b. the tensor-core record (bf16 I/O, d_k = d_v = 128)
// Phase stamps of the prep kernel (CTA 0, thread 0, first 64 items), compiled only with
// -DKDA_BWD_TRACE; the default build has no trace code.
#ifdef KDA_BWD_TRACE
__device__ long long g_prep_trace[64][12];
#define PREP_TRACE(i) \
    do { \
        if (blockIdx.x == 0 && tid == 0 && m < 64) g_prep_trace[m][i] = clock64(); \
    } while (0)
#else
#define PREP_TRACE(i) \
    do { \
    } while (0)
#endif
// Two CTAs per SM walk contiguous ranges of items (chunk slot, head). Per item: the q, k, v
// and gate-logit rows arrive by bulk copies one item ahead (double-buffered); G and gamma_L
// per key channel; Q~, K~, K^, K' elementwise; Z = K~ K^^T and P = Q~ K^^T on the tensor
// cores with each operand split into a bf16 high and low part (hi hi + lo hi + hi lo: close
// to fp32 products); T = (I + A)^-1 by forward substitution on one warp; W = M K~ and
// U~ = M V with M split the same way. The record is assembled in shared memory in its
// global layout and written by one bulk copy.
constexpr int PT_THREADS = 256;
constexpr int IT16 = C * 128 * 2;               // a dense bf16 input tile [16][128]
constexpr int IBUF = 3 * IT16 + C * 128 * 4;     // q, k, v [16][128] bf16; a [16][128] fp32
constexpr int PS_REC = 2 * IBUF;
constexpr int PS_QL = PS_REC + RECB, PS_KTL = PS_QL + T128;
constexpr int PS_KHL = PS_KTL + T128, PS_A = PS_KHL + T128, PS_ML = PS_A + C * C * 4;
constexpr int PS_BT = PS_ML + C * PS * 2;
constexpr int PS_TS = PS_BT + C * 4, PS_YS = PS_TS + C * C * 4, PS_PART = PS_YS + 64 * 4;
constexpr int PS_GT = PS_PART + 8 * C * C * 4;  // first-half totals of G [128]
constexpr int PS_BYTES = PS_GT + 128 * 4;
static_assert(IBUF % 16 == 0 && PS_QL % 16 == 0 && PS_A % 16 == 0 && 2 * (PS_BYTES + 1024) <= 228 * 1024,
              "two prep CTAs per SM");

// hi = bf16(x), lo = bf16(x - hi)
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    hi = pack2(x0, x1);
    const float2 h = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&hi));
    lo = pack2(x0 - h.x, x1 - h.y);
}

__global__ void __launch_bounds__(PT_THREADS, 2)
    prep_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_a,
                   const float *__restrict__ beta, const int32_t *__restrict__ cu,
                   unsigned char *__restrict__ ws, int H, int n_seq, long long n_items,
                   float scale) {
    constexpr int D = 128;
    extern __shared__ __align__(128) unsigned char sp[];
    __shared__ __align__(8) unsigned long long bars[2];  // input buffers 0, 1
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g4 = lane >> 2, l4 = lane & 3, n0 = 16 * warp;
    const long long beg = (long long)blockIdx.x * n_items / gridDim.x;
    const long long end = (long long)(blockIdx.x + 1) * n_items / gridDim.x;
    const uint32_t sb = static_cast<uint32_t>(__cvta_generic_to_shared(sp));
    auto bar = [&](int i) { return static_cast<uint32_t>(__cvta_generic_to_shared(&bars[i])); };
    unsigned char *rec = sp + PS_REC;
    float *As = reinterpret_cast<float *>(sp + PS_A), *bts = reinterpret_cast<float *>(sp + PS_BT);
    if (tid == 0) {
        bar_init(bar(0), 1);
        bar_init(bar(1), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // one thread: the item's 16 token rows of q, k, v and the gate logits into input buffer
    // b, one tensor copy each (rows past the end of the tensor arrive as zeros; rows past the
    // sequence's end hold other tokens, masked where they are used)
    auto issue_in = [&](const Item &it, int b) {
        const int64_t c0 = it.c0;
        const uint32_t bb = sb + b * IBUF;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        bar_arrive_tx(bar(b), (uint32_t)IBUF);
        tma_load_3d(bb, &tm_q, 0, it.h, (int)c0, bar(b));
        tma_load_3d(bb + IT16, &tm_k, 0, it.h, (int)c0, bar(b));
        tma_load_3d(bb + 2 * IT16, &tm_v, 0, it.h, (int)c0, bar(b));
        tma_load_3d(bb + 3 * IT16, &tm_a, 0, it.h, (int)c0, bar(b));
    };

    ItemCursor ic;
    ic.start(cu, n_seq, H, beg, end);
    Item cur = ic.item(), nxt;
    long long idx = ic.idx;
    if (idx < end && tid == 0) issue_in(cur, 0);
    auto load_beta = [&](const Item &it) {  // beta of an item's rows, 0 past its end
        return tid < it.L ? beta[(size_t)(it.c0 + tid) * H + it.h] : 0.f;
    };
    float bta = (idx < end && tid < C) ? load_beta(cur) : 0.f;  // loaded an item ahead
    for (int m = 0; idx < end; ++m) {
        ic.advance();
        const long long nidx = ic.idx;
        nxt = ic.item();
        const bool more = nidx < end;
        const int L = cur.L;
        const int h = cur.h;
        const float bta_next = (more && tid < C) ? load_beta(nxt) : 0.f;
        PREP_TRACE(0);
        if (tid == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        PREP_TRACE(1);
        __syncthreads();  // the record staging is free; the other input buffer's readers are done
        PREP_TRACE(2);
        if (more && tid == 0) issue_in(nxt, (m + 1) & 1);
        PREP_TRACE(3);
        if (tid < C) {
            bts[tid] = bta;
            reinterpret_cast<float *>(rec + TR_B)[tid] = bta;
        }
        const int ib = m & 1;
        const bool ok = bar_wait(bar(ib), (uint32_t)((m >> 1) & 1));
        if (__syncthreads_or(!ok)) break;
        PREP_TRACE(4);
        const unsigned char *in = sp + ib * IBUF;
        const uint32_t inb = sb + ib * IBUF;
        float *GS = reinterpret_cast<float *>(rec + TR_GS);

        // ---- G = cumsum of g = -5 sigmoid(a) per key channel, gamma_L = e^{G_15}: thread
        // (channel x, half) sums rows [8 half, 8 half + 8); the second half then adds the
        // first half's total
        float *Gtot = reinterpret_cast<float *>(sp + PS_GT);
        {
            const int x = tid & (D - 1), half = tid >> 7;
            const float *Ain = reinterpret_cast<const float *>(in + 3 * IT16);
            float G = 0.f;
#pragma unroll
            for (int r8 = 0; r8 < C / 2; ++r8) {
                const int r = 8 * half + r8;
                const float g = r < L ? __fdividef(kGMin, 1.f + __expf(-Ain[r * D + x])) : 0.f;
                G += g;
                GS[r * GP + x] = G;
            }
            if (half == 0) Gtot[x] = G;
        }
        __syncthreads();
        if (tid >= D) {
            const int x = tid - D;
            const float g0 = Gtot[x];
            float G = 0.f;
#pragma unroll
            for (int r = C / 2; r < C; ++r) {
                G = GS[r * GP + x] + g0;
                GS[r * GP + x] = G;
            }
            const float gl = __expf(G);
            reinterpret_cast<float *>(rec + TR_GL)[x] = gl;
            reinterpret_cast<float *>(rec + TR_G)[gperm_tc(x)] = gl;
        } else if (L < C) {  // V rows past the sequence's end to zero (they meet M's zero columns)
            unsigned char *vt = sp + ib * IBUF + 2 * IT16;
            for (int i = tid; i < (C - L) * 16; i += D)
                *reinterpret_cast<uint4 *>(vt + L * 256 + i * 16) = make_uint4(0u, 0u, 0u, 0u);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // before the buffer's next copy
        }
        __syncthreads();

        PREP_TRACE(5);
        // ---- Q~ = q e^G, K~ = k e^G, K^ = k e^-G, K' = k e^{G_15 - G}: 8 channels per thread
        {
            const int r = tid >> 4, x0 = (tid & 15) * 8;
            uint4 qr = *reinterpret_cast<const uint4 *>(in + (r * 128 + x0) * 2);
            uint4 kr = *reinterpret_cast<const uint4 *>(in + IT16 + (r * 128 + x0) * 2);
            if (r >= L) qr = kr = make_uint4(0u, 0u, 0u, 0u);  // past the sequence's end
            const uint32_t qw[4] = {qr.x, qr.y, qr.z, qr.w}, kw[4] = {kr.x, kr.y, kr.z, kr.w};
            uint32_t okp[4], okt[4], okh[4], oqh[4], oql[4], oktl[4], okhl[4];
#pragma unroll
            for (int p2 = 0; p2 < 4; ++p2) {
                const float2 qf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qw[p2]));
                const float2 kf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kw[p2]));
                float Qt[2], Kt[2], Kh[2], Kp[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int x = x0 + 2 * p2 + e;
                    const float G = GS[r * GP + x], GL = GS[(C - 1) * GP + x];
                    const float qx = e ? qf.y : qf.x, kx = e ? kf.y : kf.x;
                    const float eg = __expf(G), en = __expf(-G);
                    Qt[e] = qx * eg;
                    Kt[e] = kx * eg;
                    Kh[e] = kx * en;
                    Kp[e] = kx * __expf(GL - G);
                }
                okp[p2] = pack2(Kp[0], Kp[1]);
                split2(Qt[0], Qt[1], oqh[p2], oql[p2]);
                split2(Kt[0], Kt[1], okt[p2], oktl[p2]);
                split2(Kh[0], Kh[1], okh[p2], okhl[p2]);
            }
            const int off = (r * 136 + x0) * 2;
            auto st4 = [&](unsigned char *base, const uint32_t (&w)[4]) {
                *reinterpret_cast<uint4 *>(base + off) = make_uint4(w[0], w[1], w[2], w[3]);
            };
            st4(rec + TR_K, okp);
            st4(rec + TR_Q, oqh);
            st4(rec + TR_KT, okt);
            st4(rec + TR_KH, okh);
            st4(sp + PS_QL, oql);
            st4(sp + PS_KTL, oktl);
            st4(sp + PS_KHL, okhl);
        }
        __syncthreads();

        PREP_TRACE(6);
        // ---- Z = K~ K^^T and P = Q~ K^^T, split-bf16 products: warp w takes product w & 1
        // over key channels [32 (w >> 1), +32); the four partial sums are added in order
        float *part = reinterpret_cast<float *>(sp + PS_PART);  // [8 warps][16][16]
        {
            const int prod = warp & 1, kq = warp >> 1;
            const uint32_t ah_b = prod == 0 ? sb + PS_REC + TR_KT : sb + PS_REC + TR_Q;
            const uint32_t al_b = prod == 0 ? sb + PS_KTL : sb + PS_QL;
            const uint32_t bh_b = sb + PS_REC + TR_KH, bl_b = sb + PS_KHL;
            float c0a[2][4] = {}, c1a[2][4] = {}, c2a[2][4] = {};
#pragma unroll
            for (int k0 = 32 * kq; k0 < 32 * kq + 32; k0 += 16) {
                uint32_t ah[4], al[4], bh[4], bl[4];
                ld_a(ah_b, PB, k0, ah);
                ld_a(al_b, PB, k0, al);
                ld_b_nk(bh_b, PB, 0, k0, bh);  // B[key][t'] = K^[t'][key]
                ld_b_nk(bl_b, PB, 0, k0, bl);
                mma16816(c0a[0], ah, bh[0], bh[1]);
                mma16816(c0a[1], ah, bh[2], bh[3]);
                mma16816(c1a[0], al, bh[0], bh[1]);
                mma16816(c1a[1], al, bh[2], bh[3]);
                mma16816(c2a[0], ah, bl[0], bl[1]);
                mma16816(c2a[1], ah, bl[2], bl[3]);
            }
            float *pw = part + warp * C * C;
#pragma unroll
            for (int tt = 0; tt < 2; ++tt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
                    *reinterpret_cast<float2 *>(pw + (g4 + 8 * hh) * C + 8 * tt + 2 * l4) =
                        make_float2(c0a[tt][2 * hh] + (c1a[tt][2 * hh] + c2a[tt][2 * hh]),
                                    c0a[tt][2 * hh + 1] + (c1a[tt][2 * hh + 1] + c2a[tt][2 * hh + 1]));
        }
        __syncthreads();
        {
            const int r = tid >> 4, j = tid & 15;
            const float z = part[0 * C * C + tid] + part[2 * C * C + tid] + part[4 * C * C + tid] +
                            part[6 * C * C + tid];
            const float pq = part[1 * C * C + tid] + part[3 * C * C + tid] + part[5 * C * C + tid] +
                             part[7 * C * C + tid];
            reinterpret_cast<float *>(rec + TR_Z)[tid] = z;
            As[tid] = j < r ? bts[r] * z : 0.f;
            reinterpret_cast<__nv_bfloat16 *>(rec + TR_P)[r * PS + j] = __float2bfloat16_rn(j <= r ? pq : 0.f);
        }
        __syncthreads();

        PREP_TRACE(7);
        // ---- T = (I + A)^-1 in 8 x 8 blocks on warp 0: T11 = (I + A11)^-1 (lanes 0-7, one
        // column each) and T22 = (I + A22)^-1 (lanes 8-15) by forward substitution, then
        // T21 = -T22 (A21 T11); T12 = 0
        float *Ts = reinterpret_cast<float *>(sp + PS_TS), *Ys = reinterpret_cast<float *>(sp + PS_YS);
        if (warp == 0) {
            const int o = lane & 8, j = lane & 7;
            float col[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                float x = r == j ? 1.f : 0.f;
#pragma unroll
                for (int i = 0; i < r; ++i) x = fmaf(-As[(o + r) * C + o + i], col[i], x);
                col[r] = x;
            }
            if (lane < 16) {
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    Ts[(o + r) * C + o + j] = col[r];
                    if (o == 0) Ts[r * C + 8 + j] = 0.f;
                }
            }
            __syncwarp();
#pragma unroll
            for (int e = lane; e < 64; e += 32) {  // Y = A21 T11
                const int r = 8 + (e >> 3), jj = e & 7;
                float y = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) y = fmaf(As[r * C + i], Ts[i * C + jj], y);
                Ys[e] = y;
            }
            __syncwarp();
#pragma unroll
            for (int e = lane; e < 64; e += 32) {  // T21 = -T22 Y
                const int r = 8 + (e >> 3), jj = e & 7;
                float t = 0.f;
#pragma unroll
                for (int i = 8; i < C; ++i) t = fmaf(Ts[r * C + i], Ys[(i - 8) * 8 + jj], t);
                Ts[r * C + jj] = -t;
            }
        }
        __syncthreads();
        PREP_TRACE(8);
        {  // T, T^T and M = T diag(beta) (high and low bf16 parts) into the record
            const int r = tid >> 4, j = tid & 15;
            const float tv = Ts[tid];
            reinterpret_cast<float *>(rec + TR_T)[tid] = tv;
            reinterpret_cast<float *>(rec + TR_TT)[j * C + r] = tv;
            const float mv = tv * bts[j];
            const __nv_bfloat16 mh = __float2bfloat16_rn(mv);
            reinterpret_cast<__nv_bfloat16 *>(rec + TR_M)[r * PS + j] = mh;
            reinterpret_cast<__nv_bfloat16 *>(sp + PS_ML)[r * PS + j] =
                __float2bfloat16_rn(mv - __bfloat162float(mh));
        }
        __syncthreads();

        PREP_TRACE(9);
        // ---- W = M K~ (stored as -W, bf16) and U~ = M V (fp32, transposed): columns [n0, n0 + 16)
        {
            uint32_t mh[4], ml[4], bh[4], bl[4], bv[4];
            ld_a(sb + PS_REC + TR_M, PS, 0, mh);
            ld_a(sb + PS_ML, PS, 0, ml);
            ld_b_kn(sb + PS_REC + TR_KT, PB, 0, n0, bh);  // B[t][x] = K~[t][x]
            ld_b_kn(sb + PS_KTL, PB, 0, n0, bl);
            ld_b_kn(inb + 2 * IT16, 128, 0, n0, bv);     // B[t][v] = V[t][v]
            float w[2][4] = {}, w2[2][4] = {}, u[2][4] = {}, u2[2][4] = {};
            mma16816(w[0], mh, bh[0], bh[1]);
            mma16816(w[1], mh, bh[2], bh[3]);
            mma16816(w2[0], ml, bh[0], bh[1]);
            mma16816(w2[1], ml, bh[2], bh[3]);
            mma16816(w2[0], mh, bl[0], bl[1]);
            mma16816(w2[1], mh, bl[2], bl[3]);
            mma16816(u[0], mh, bv[0], bv[1]);
            mma16816(u[1], mh, bv[2], bv[3]);
            mma16816(u2[0], ml, bv[0], bv[1]);
            mma16816(u2[1], ml, bv[2], bv[3]);
            float *Ut = reinterpret_cast<float *>(rec + TR_UT);  // [v][16 t]
#pragma unroll
            for (int tt = 0; tt < 2; ++tt) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    w[tt][i] = -(w[tt][i] + w2[tt][i]);
                    const int t = g4 + 8 * (i >> 1), vc = n0 + 8 * tt + 2 * l4 + (i & 1);
                    Ut[vc * C + t] = u[tt][i] + u2[tt][i];
                }
            }
            store_c16(reinterpret_cast<__nv_bfloat16 *>(rec + TR_W), PB, n0, w);
        }
        PREP_TRACE(10);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the record, to the copy
        __syncthreads();
        if (tid == 0) {
            unsigned char *dst = ws + ((size_t)cur.slot * H + h) * REC_TC + TC_REC;
            asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                         ::"l"(dst), "r"(sb + PS_REC), "r"((uint32_t)RECB) : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
        PREP_TRACE(11);
        idx = nidx;
        cur = nxt;
        bta = bta_next;
    }
    if (tid == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// [n_tok][H][128] row-major as a 3-D tensor (channel, head, token) with boxes of box_x
// channels x 1 head x 16 tokens; tokens past n_tok read as zero.
PFN_cuTensorMapEncodeTiled_v12000 map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}
bool token_map(CUtensorMap *m, const void *base, bool f32, int64_t n_tok, int H, int box_x,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
    auto enc = map_encoder();
    if (!enc) return false;
    const cuuint64_t es = f32 ? 4 : 2;
    cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)n_tok};
    cuuint64_t strides[2] = {128 * es, (cuuint64_t)H * 128 * es};
    cuuint32_t box[3] = {(cuuint32_t)box_x, 1, (cuuint32_t)C};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
               const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per-kernel timing of backward calls (a measurement aid): events before the first kernel
// and after each of the four, for up to `capacity` calls.
struct BwdTiming {
    std::mutex mu;
    std::vector<cudaEvent_t> ev;  // capacity x 5
    int capacity = 0, used = 0;
    bool active = false;
};
BwdTiming &bwd_timing() {
    static BwdTiming t;
    return t;
}
struct CallEvents {  // the events of one call, or none
    cudaEvent_t *ev = nullptr;
    cudaStream_t stream = nullptr;
    void mark(int i) const {
        if (ev) cudaEventRecord(ev[i], stream);
    }
};
CallEvents claim_events(cudaStream_t stream) {
    BwdTiming &t = bwd_timing();
    std::lock_guard<std::mutex> lock(t.mu);
    CallEvents c;
    if (t.active && t.used < t.capacity) {
        c.ev = t.ev.data() + 5 * t.used++;
        c.stream = stream;
    }
    return c;
}

template <typename IO>
cudaError_t launch_bwd_t(const BwdArgs &p, cudaStream_t stream) {
    const int H = p.n_heads, dk = p.d_k, dv = p.d_v;
    const float scale = 1.0f / sqrtf((float)dk);
    const unsigned items = (unsigned)p.n_seq * (unsigned)H;
    const size_t slots = bwd_slots(p.n_tok, p.n_seq);
    float *ck = p.workspace;
    float *dck = ck + slots * (size_t)H * dk * dv;
    float *prep = dck + slots * (size_t)H * dk * dv;
    const IO *q = (const IO *)p.q, *k = (const IO *)p.k, *v = (const IO *)p.v;
    const IO *dout = (const IO *)p.dout;

    const size_t sm0 = chunk_floats(dk, dv) * 4;
    const size_t sm1 = ((size_t)2 * stage_floats(dk) + (size_t)RG * C * JS + C * JS) * 4;
    const size_t sm2 = sm1 + (size_t)C * JS * 4;
    const size_t sm3 = local_floats(dk, dv) * 4;
    // bf16 I/O at d_k = d_v = 128 runs on the tensor cores (bf16 operand rounding is within
    // that I/O's precision) when the bulk copies' 16-byte alignment holds; fp32 FMA loops
    // otherwise
    // (inputs and workspace: 16-byte bulk copies; dq, dk, dv: 4-byte pair stores; dgate:
    // 8-byte pair stores)
    auto al = [](const void *x, uintptr_t m) { return ((uintptr_t)x & (m - 1)) == 0; };
    const bool use_tc = sizeof(IO) == 2 && dk == 128 && dv == 128 && al(p.workspace, 16) &&
                        al(p.q, 16) && al(p.k, 16) && al(p.v, 16) && al(p.a, 16) &&
                        al(p.dout, 16) && al(p.dq, 4) && al(p.dk, 4) && al(p.dv, 4) &&
                        al(p.da, 8);
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(prep_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm0)) != cudaSuccess)
        return e;
    // the chunks of a sequence spread over gridDim.y CTAs: a few per SM over the launch,
    // so uneven sequences balance
    const int64_t max_chunks = (p.n_tok + C - 1) / C;
    int64_t gy = (4 * 152 + (int64_t)items - 1) / (int64_t)items;
    if (gy > max_chunks) gy = max_chunks;
    if (gy < 1) gy = 1;
    if (gy > 65535) gy = 65535;
    const dim3 par(items, (unsigned)gy), cols(items, (unsigned)((dv + JS - 1) / JS));
    const CallEvents tev = claim_events(stream);
    if (use_tc) {
        // serial passes with the state in mma fragments, then the local gradients with one
        // CTA per SM over all (chunk slot, head) items
        unsigned char *wsb = reinterpret_cast<unsigned char *>(p.workspace);
        const int smc = NS * SLOT + 4 * CT_ROWS;
        int dev = 0, sms = 0;
        if ((e = cudaFuncSetAttribute(chains_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smc)) != cudaSuccess ||
            (e = cudaFuncSetAttribute(local_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, LS_BYTES)) != cudaSuccess ||
            (e = cudaFuncSetAttribute(prep_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PS_BYTES)) != cudaSuccess ||
            (e = cudaGetDevice(&dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return e;
        const __nv_bfloat16 *d16 = reinterpret_cast<const __nv_bfloat16 *>(p.dout);
        const long long n_items = ((long long)(p.n_tok >> 4) + p.n_seq) * H;
        const __nv_bfloat16 *b16[3] = {reinterpret_cast<const __nv_bfloat16 *>(p.q),
                                       reinterpret_cast<const __nv_bfloat16 *>(p.k),
                                       reinterpret_cast<const __nv_bfloat16 *>(p.v)};
        const int pgrid = (int)(n_items < 2 * sms ? n_items : 2 * sms);
        CUtensorMap mq, mk, mv, ma;
        if (!token_map(&mq, b16[0], false, p.n_tok, H, 128) ||
            !token_map(&mk, b16[1], false, p.n_tok, H, 128) ||
            !token_map(&mv, b16[2], false, p.n_tok, H, 128) ||
            !token_map(&ma, p.a, true, p.n_tok, H, 128))
            return cudaErrorInvalidValue;
        tev.mark(0);
        prep_tc_kernel<<<pgrid, PT_THREADS, PS_BYTES, stream>>>(mq, mk, mv, ma, p.beta,
                                                               p.cu_seqlens, wsb, H, p.n_seq,
                                                               n_items, scale);
        tev.mark(1);
        CUtensorMap mo;
        if (!token_map(&mo, d16, false, p.n_tok, H, 32)) return cudaErrorInvalidValue;
        chains_tc_kernel<<<items * 8, 128, smc, stream>>>(p.cu_seqlens, wsb, mo, p.h0, p.dh_final,
                                                         p.dh0, H, scale, (int)(items * 4));
        tev.mark(2);  // both serial passes in the one launch: the reverse pass's entry is 0
        tev.mark(3);
        const int grid = (int)(n_items < sms ? n_items : sms);
        CUtensorMap mvs, mos;  // V and dO in 64-column, 128-byte-swizzled boxes
        if (!token_map(&mvs, b16[2], false, p.n_tok, H, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !token_map(&mos, d16, false, p.n_tok, H, 64, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        local_tc_kernel<<<grid, LT_THREADS, LS_BYTES, stream>>>(
            mvs, ma, p.a, p.cu_seqlens, mos, wsb,
            reinterpret_cast<__nv_bfloat16 *>(p.dq), reinterpret_cast<__nv_bfloat16 *>(p.dk),
            reinterpret_cast<__nv_bfloat16 *>(p.dv), p.da, p.dbeta, H, p.n_seq, n_items, scale);
        tev.mark(4);
    } else {
        if ((e = cudaFuncSetAttribute(ckpt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1)) != cudaSuccess ||
            (e = cudaFuncSetAttribute(chain_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2)) != cudaSuccess ||
            (e = cudaFuncSetAttribute(local_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3)) != cudaSuccess)
            return e;
        tev.mark(0);
        prep_kernel<IO><<<par, kThreads, sm0, stream>>>(q, k, v, p.a, p.beta, p.cu_seqlens, prep,
                                                       H, dk, dv);
        tev.mark(1);
        ckpt_kernel<<<cols, kThreads, sm1, stream>>>(p.h0, p.cu_seqlens, prep, ck, H, dk, dv);
        tev.mark(2);
        chain_kernel<IO><<<cols, kThreads, sm2, stream>>>(p.cu_seqlens, dout, p.dh_final, prep,
                                                         dck, p.dh0, H, dk, dv, scale);
        tev.mark(3);
        local_kernel<IO><<<par, kThreads, sm3, stream>>>(
            q, k, v, p.a, p.beta, p.cu_seqlens, dout, ck, dck, (IO *)p.dq, (IO *)p.dk,
            (IO *)p.dv, p.da, p.dbeta, H, dk, dv, scale);
        tev.mark(4);
    }
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(use_tc ? 3 : 4);
    return e;
}

}  // namespace

size_t bwd_slots(int64_t n_tok, int32_t n_seq) { return (size_t)(n_tok >> 4) + (size_t)n_seq + 1; }

// a * b, or SIZE_MAX when the product does not fit
static size_t mul_saturating(size_t a, size_t b) {
    return (a != 0 && b > SIZE_MAX / a) ? SIZE_MAX : a * b;
}

size_t bwd_workspace_bytes(int64_t n_tok, int32_t n_seq, int32_t n_heads, int32_t d_k,
                           int32_t d_v) {
    // saturates instead of wrapping, so that no size check passes on an overflowed figure
    const size_t per_slot_head =
        mul_saturating(mul_saturating(2, (size_t)d_k), (size_t)d_v) + prep_floats(d_k, d_v);
    return mul_saturating(mul_saturating(mul_saturating(bwd_slots(n_tok, n_seq), (size_t)n_heads),
                                         per_slot_head),
                          sizeof(float));
}

cudaError_t launch_bwd(const BwdArgs &p, cudaStream_t stream) {
    if (p.n_seq == 0) return cudaSuccess;
    return p.bf16 ? launch_bwd_t<__nv_bfloat16>(p, stream) : launch_bwd_t<float>(p, stream);
}

cudaError_t bwd_timing_start(int capacity) {
    BwdTiming &t = bwd_timing();
    std::lock_guard<std::mutex> lock(t.mu);
    for (cudaEvent_t e : t.ev) cudaEventDestroy(e);
    t.ev.assign((size_t)capacity * 5, nullptr);
    t.capacity = t.used = 0;
    t.active = false;
    for (size_t i = 0; i < t.ev.size(); ++i) {
        const cudaError_t e = cudaEventCreate(&t.ev[i]);
        if (e != cudaSuccess) {
            for (size_t j = 0; j < i; ++j) cudaEventDestroy(t.ev[j]);
            t.ev.clear();
            return e;
        }
    }
    t.capacity = capacity;
    t.active = true;
    return cudaSuccess;
}

cudaError_t bwd_timing_read(float ms[4], int *calls) {
    BwdTiming &t = bwd_timing();
    std::lock_guard<std::mutex> lock(t.mu);
    t.active = false;
    for (int i = 0; i < 4; ++i) ms[i] = 0.f;
    for (int c = 0; c < t.used; ++c) {
        cudaError_t e = cudaEventSynchronize(t.ev[5 * c + 4]);
        if (e != cudaSuccess) return e;
        for (int i = 0; i < 4; ++i) {
            float x = 0.f;
            if ((e = cudaEventElapsedTime(&x, t.ev[5 * c + i], t.ev[5 * c + i + 1])) != cudaSuccess) return e;
            ms[i] += x;
        }
    }
    *calls = t.used;
    return cudaSuccess;
}

}  // namespace kda

namespace kda {
cudaError_t read_bwd_flags(unsigned int *flags, bool reset, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(flags, g_bwd_flags, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    if (reset) {
        static const unsigned int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_bwd_flags, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                                    stream);
        if (e != cudaSuccess) return e;
    }
    return cudaStreamSynchronize(stream);
}
}  // namespace kda

#ifdef KDA_BWD_TRACE
extern "C" int kda_debug_prep_trace_dump(long long *host) {
    return (int)cudaMemcpyFromSymbol(host, kda::g_prep_trace, sizeof(kda::g_prep_trace));
}
#endif
#ifdef KDA_BWD_TRACE
extern "C" int kda_debug_local_trace_dump(long long *host) {
    return (int)cudaMemcpyFromSymbol(host, kda::g_local_trace, sizeof(kda::g_local_trace));
}
#endif
