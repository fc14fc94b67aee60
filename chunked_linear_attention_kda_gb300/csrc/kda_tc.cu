// kda_tc.cu -- tensor-core kernel for the chunked KDA forward pass, bf16 I/O,
// d_k = d_v = 128, fp32 state and accumulation, for sm_103a.
//
// Work decomposition. One thread-block cluster of kCS = 4 CTAs per (sequence,
// head). CTA rank r owns value columns [32 r, 32 r + 32) of the state, i.e. 32 rows
// of S^T (d_v x d_k), held in registers by two "state" warps (16 rows each) for the
// whole sequence. Columns of the state evolve independently, so the four CTAs of a
// head never exchange state. What they share is the per-chunk "prologue" -- the gate,
// the in-chunk cumulative decay and the diagonal (intra-chunk) tile -- which does not
// depend on the state: chunk n's prologue is computed once, by CTA n mod 4, and
// broadcast into the other three CTAs' shared memory with DSMEM bulk copies.
//
// Per chunk of L <= 16 tokens (rows past L act as q = k = v = 0, beta = 0, g = 0):
//   prologue   g = -5 sigmoid(a) per key channel; Gamma_r = prod_{i<=r} exp(g_i)
//              (= exp(G_r), G the in-chunk cumulative log-decay), gamma_L = Gamma_15;
//              Q~ = q Gamma, K~ = k Gamma, K' = k exp(G_L - G), K^ = K' / gamma_L
//              (= k exp(-G) <= exp(80), representable in bf16 because the bound keeps
//              16 x (-5) = -80: "From Numerical Stability to Load Balancing", §2.1-2.2;
//              "Demystifying Trillion-Parameter MoE Models", Breakthrough 1 §2);
//              A = strict_lower(beta K~ K^^T), P = lower(Q~ K^^T)   [tensor cores];
//              TB = (I + A)^-1 diag(beta)  [fp32 forward substitution];
//              -W = -TB K~                 [tensor cores]
//   state      U^T = V^T TB^T - S^T W^T; O^T = S^T Q~^T + U^T P^T;
//              S^T <- S^T diag(gamma_L) + U^T K'   [tensor cores, S^T in registers]
// The diagonal tile is thus dense tensor-core products with no per-position branch
// ("Architecting Long-Context LLMs", §2.2-2.3), and the state recurrence runs serially
// across chunks ("From Numerical Stability to Load Balancing", §2.1).
//
// Tensor-core instruction: mma.sync m16n8k16 bf16 -> fp32. Its M = 16 matches the
// 16-token tile exactly, and its accumulator fragment layout, converted to bf16, is the
// operand fragment layout of the next product, so the serial chain S -> U -> S stays
// in registers with no shuffles and no shared-memory round trip.
//
// Data movement: q, k, gate logits and v tiles arrive by TMA (cp.async.bulk.tensor)
// into mbarrier-tracked rings; prologue products travel between the CTAs of a
// cluster by cp.async.bulk shared::cta -> shared::cluster with complete_tx on the
// receiver's mbarrier. Every wait is bounded: a wait that exceeds its limit sets a
// device flag (kda_read_device_flags), releases every other wait in the grid and lets
// the kernel finish with unspecified output.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_internal.h"

namespace kda {

__device__ unsigned int g_device_flags;  // bit 0: a pipeline wait exceeded its limit

namespace {

constexpr int D = 128;          // d_k = d_v
constexpr int C = kChunk;       // 16 tokens
constexpr int kCS = 4;          // CTAs per (sequence, head) = cluster size
constexpr int VB = D / kCS;     // value columns per CTA (32)
constexpr int NSW = VB / 16;    // state warps per CTA (2)
constexpr int NPW = 4;          // prologue warps
constexpr int kThreads = 32 * (1 + NPW + NSW);
constexpr int NP = 8;           // product-ring depth (multiple of kCS)
constexpr int NR = 2;           // raw-input ring depth (owned chunks)
constexpr int LDP = 136;        // pitch (elements) of 16 x 128 bf16 tiles: 272 B rows
constexpr int LDS = 24;         // pitch of 16 x 16 bf16 tiles: 48 B rows
constexpr long long kWaitLimit = 4000000000LL;  // cycles (~2 s) before a wait gives up

static_assert(NP % kCS == 0, "slot ownership must be static");

// ---- shared-memory layout (bytes) ----
constexpr int OFF_PQ = 0;                        // Q~   [16][LDP] bf16
constexpr int OFF_PW = OFF_PQ + C * LDP * 2;     // -W   [16][LDP] bf16
constexpr int OFF_PK = OFF_PW + C * LDP * 2;     // K'   [16][LDP] bf16
constexpr int OFF_PTB = OFF_PK + C * LDP * 2;    // TB   [16][LDS] bf16
constexpr int OFF_PP = OFF_PTB + C * LDS * 2;    // P    [16][LDS] bf16
constexpr int OFF_PG = OFF_PP + C * LDS * 2;     // gamma_L [128] f32
constexpr int SLOT_BYTES = OFF_PG + D * 4;       // 15104
static_assert(SLOT_BYTES % 16 == 0, "bulk copies move 16-byte multiples");

constexpr int RAW_Q = 0, RAW_K = C * D * 2, RAW_A = 2 * C * D * 2;
constexpr int RAW_BYTES = RAW_A + C * D * 4;     // 16384
constexpr int V_BYTES = C * VB * 2;              // 1024

constexpr int SM_RAW = 0;
constexpr int SM_V = SM_RAW + NR * RAW_BYTES;
constexpr int SM_PROD = SM_V + NP * V_BYTES;
constexpr int SM_KT = SM_PROD + NP * SLOT_BYTES; // K~ [16][LDP] bf16 (prologue scratch)
constexpr int SM_KH = SM_KT + C * LDP * 2;       // K^ [16][LDP] bf16
constexpr int SM_A = SM_KH + C * LDP * 2;        // A  [16][16] f32
constexpr int SM_BETA = SM_A + C * C * 4;        // beta [16] f32
constexpr int SM_OST = SM_BETA + C * 4;          // O staging [NSW][16][LDS] bf16
constexpr int SM_BAR = SM_OST + NSW * C * LDS * 2;
constexpr int NBARS = 3 * NP + 2 * NR;
constexpr int SM_MISC = SM_BAR + NBARS * 8;
constexpr int SMEM_BYTES = SM_MISC + 64;
static_assert(SM_V % 128 == 0 && SM_PROD % 16 == 0 && SM_BAR % 8 == 0, "alignment");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

// barrier indices
__host__ __device__ constexpr int B_FULL(int s) { return s; }           // products + V in
__host__ __device__ constexpr int B_FREE(int s) { return NP + s; }      // local state warps done
__host__ __device__ constexpr int B_CFREE(int s) { return 2 * NP + s; } // all CTAs done (owner)
__host__ __device__ constexpr int B_RFULL(int s) { return 3 * NP + s; }
__host__ __device__ constexpr int B_REMPTY(int s) { return 3 * NP + NR + s; }

struct TcParams {
    const float *beta, *h0;
    const int32_t *cu;
    __nv_bfloat16 *out;
    float *h_final;
    int n_seq, H;
};

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t a, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint32_t a) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t a, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t a, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok) : "r"(a), "r"(parity) : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_try_cluster(uint32_t a, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok) : "r"(a), "r"(parity) : "memory");
    return ok != 0;
}
// Bounded wait. Returns false when this or any other wait of the grid gave up.
template <bool kClusterScope>
__device__ __forceinline__ bool mbar_wait(uint32_t a, uint32_t parity) {
    if (kClusterScope ? mbar_try_cluster(a, parity) : mbar_try(a, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (kClusterScope ? mbar_try_cluster(a, parity) : mbar_try(a, parity)) return true;
        if ((it & 63u) == 0) {
            if (*(volatile unsigned int *)&g_device_flags != 0u) return false;
            if (clock64() - t0 > kWaitLimit) {
                atomicOr(&g_device_flags, 1u);
                return false;
            }
        }
    }
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
    return r;
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst_cluster, uint32_t src,
                                                  uint32_t bytes, uint32_t mbar_cluster) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst_cluster), "r"(src), "r"(bytes), "r"(mbar_cluster) : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            int z, uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(map), "r"(x), "r"(y), "r"(z), "r"(mbar) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ bool named_sync_or(int id, int n, bool pred) {
    uint32_t out;
    asm volatile(
        "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, %2, %3, p; selp.u32 %0, 1, 0, q; }"
        : "=r"(out) : "r"((uint32_t)pred), "r"(id), "r"(n) : "memory");
    return out != 0;
}
__device__ __forceinline__ void ldsm_x4(uint32_t a, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t a, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(a));
}
__device__ __forceinline__ void ldsm_x2(uint32_t a, uint32_t &r0, uint32_t &r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r0), "=r"(r1) : "r"(a));
}
__device__ __forceinline__ void stsm_x4_t(uint32_t a, uint32_t r0, uint32_t r1, uint32_t r2,
                                          uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1,%2,%3,%4};"
                 ::"r"(a), "r"(r0), "r"(r1), "r"(r2), "r"(r3) : "memory");
}
// D (16x8 f32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma16816(float *d, const uint32_t *a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (lower address)
    return *reinterpret_cast<uint32_t *>(&v);
}

// Item for this cluster: sequences ordered longest first (ties by index), heads
// innermost, so the longest serial chains are scheduled first.
__device__ void resolve_item(const TcParams &p, int ci, int *seq_out, int *head_out) {
    const int H = p.H;
    const int target = ci / H;
    if (threadIdx.x == 0) *seq_out = target;  // natural order when not ranked below
    __syncthreads();
    if (p.n_seq <= kThreads) {
        const int s = threadIdx.x;
        if (s < p.n_seq) {
            const int ls = p.cu[s + 1] - p.cu[s];
            int rank = 0;
            for (int o = 0; o < p.n_seq; ++o) {
                const int lo = p.cu[o + 1] - p.cu[o];
                rank += (lo > ls) || (lo == ls && o < s);
            }
            if (rank == target) *seq_out = s;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) *head_out = ci % H;
    __syncthreads();
}

template <bool kShare>
__global__ void __launch_bounds__(kThreads, 1)
    kda_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_v,
                  const TcParams p) {
    extern __shared__ __align__(128) unsigned char sm[];
    const uint32_t sbase = smem_u32(sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = kShare ? cluster_rank() : (uint32_t)(blockIdx.x % kCS);
    const int ci = blockIdx.x / kCS;
    int *misc = reinterpret_cast<int *>(sm + SM_MISC);
    resolve_item(p, ci, &misc[0], &misc[1]);
    const int seq = misc[0], head = misc[1];
    const int H = p.H;
    const int t0 = p.cu[seq], t1 = p.cu[seq + 1];
    const int nchunks = (t1 - t0 + C - 1) / C;
    auto bar = [&](int i) { return sbase + SM_BAR + 8u * (uint32_t)i; };
    auto owner = [&](int n) -> uint32_t { return kShare ? (uint32_t)(n % kCS) : rank; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < NP; ++s) {
            mbar_init(bar(B_FULL(s)), owner(s) == rank ? 2 : 1);
            mbar_init(bar(B_FREE(s)), NSW);
            mbar_init(bar(B_CFREE(s)), (kShare ? kCS : 1) * NSW);
        }
        for (int s = 0; s < NR; ++s) {
            mbar_init(bar(B_RFULL(s)), 1);
            mbar_init(bar(B_REMPTY(s)), 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (kShare) cluster_sync(); else __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------ producer (one lane)
        if (lane == 0) {
            int owned = 0;
            for (int n = 0; n < nchunks; ++n) {
                const int s = n % NP, use = n / NP;
                if (!mbar_wait<false>(bar(B_FREE(s)), (use & 1) ^ 1)) break;
                const bool mine = owner(n) == rank;
                mbar_arrive_tx(bar(B_FULL(s)), V_BYTES + (mine ? 0 : SLOT_BYTES));
                tma_load_3d(sbase + SM_V + s * V_BYTES, &tm_v, (int)rank * VB, head, t0 + n * C,
                            bar(B_FULL(s)));
                if (mine) {
                    const int rs = owned % NR, ru = owned / NR;
                    ++owned;
                    if (!mbar_wait<false>(bar(B_REMPTY(rs)), (ru & 1) ^ 1)) break;
                    mbar_arrive_tx(bar(B_RFULL(rs)), RAW_BYTES);
                    const uint32_t dst = sbase + SM_RAW + rs * RAW_BYTES;
                    tma_load_3d(dst + RAW_Q, &tm_q, 0, head, t0 + n * C, bar(B_RFULL(rs)));
                    tma_load_3d(dst + RAW_K, &tm_k, 0, head, t0 + n * C, bar(B_RFULL(rs)));
                    tma_load_3d(dst + RAW_A, &tm_a, 0, head, t0 + n * C, bar(B_RFULL(rs)));
                }
            }
        }
        __syncwarp();
    } else if (warp <= NPW) {
        // ------------------------------------------------ prologue (4 warps, 128 threads)
        const int c = threadIdx.x - 32;  // key channel of the gate pass
        const int pw = warp - 1;
        const int nt = 128;
        __nv_bfloat16 *Kt = reinterpret_cast<__nv_bfloat16 *>(sm + SM_KT);
        __nv_bfloat16 *Kh = reinterpret_cast<__nv_bfloat16 *>(sm + SM_KH);
        float *As = reinterpret_cast<float *>(sm + SM_A);
        float *bs = reinterpret_cast<float *>(sm + SM_BETA);
        int owned = 0;
        for (int n = 0; n < nchunks; ++n) {
            if (owner(n) != rank) continue;
            const int rs = owned % NR, ru = owned / NR;
            ++owned;
            const int s = n % NP, use = n / NP;
            const int c0 = t0 + n * C;
            const int L = min(C, t1 - c0);
            bool bad = !mbar_wait<false>(bar(B_RFULL(rs)), ru & 1);
            bad |= !mbar_wait<true>(bar(B_CFREE(s)), (use & 1) ^ 1);
            if (named_sync_or(1, nt, bad)) break;
            unsigned char *slot = sm + SM_PROD + s * SLOT_BYTES;
            __nv_bfloat16 *Pq = reinterpret_cast<__nv_bfloat16 *>(slot + OFF_PQ);
            __nv_bfloat16 *Pk = reinterpret_cast<__nv_bfloat16 *>(slot + OFF_PK);
            float *Pg = reinterpret_cast<float *>(slot + OFF_PG);
            const unsigned char *raw = sm + SM_RAW + rs * RAW_BYTES;
            const __nv_bfloat16 *rq = reinterpret_cast<const __nv_bfloat16 *>(raw + RAW_Q);
            const __nv_bfloat16 *rk = reinterpret_cast<const __nv_bfloat16 *>(raw + RAW_K);
            const float *ra = reinterpret_cast<const float *>(raw + RAW_A);
            // -- gate pass: one key channel per thread, 16 tokens in order
            {
                float eg[C], kk[C];
                float gam = 1.f;
#pragma unroll
                for (int r = 0; r < C; ++r) {
                    float qv = 0.f, kv = 0.f, e = 1.f;
                    if (r < L) {
                        qv = __bfloat162float(rq[r * D + c]);
                        kv = __bfloat162float(rk[r * D + c]);
                        const float sig = __fdividef(1.f, 1.f + __expf(-ra[r * D + c]));
                        e = __expf(kGMin * sig);  // exp(g), g = -5 sigmoid(a)
                    }
                    eg[r] = e;
                    kk[r] = kv;
                    gam *= e;  // Gamma_r = exp(G_r)
                    Pq[r * LDP + c] = __float2bfloat16_rn(qv * gam);
                    Kt[r * LDP + c] = __float2bfloat16_rn(kv * gam);
                }
                Pg[c] = gam;                        // gamma_L = exp(G_L)
                const float inv_gl = __fdividef(1.f, gam);  // exp(-G_L) <= exp(80)
                float suf = 1.f;                     // exp(G_L - G_r)
#pragma unroll
                for (int r = C - 1; r >= 0; --r) {
                    Pk[r * LDP + c] = __float2bfloat16_rn(kk[r] * suf);
                    Kh[r * LDP + c] = __float2bfloat16_rn(kk[r] * (suf * inv_gl));
                    suf *= eg[r];
                }
                if (c < C) bs[c] = c < L ? p.beta[(size_t)(c0 + c) * H + head] : 0.f;
            }
            named_sync(1, nt);
            if (c == 0) mbar_arrive(bar(B_REMPTY(rs)));  // raw tile consumed
            // -- A = strict_lower(beta K~ K^^T), P = lower(Q~ K^^T): warps 0, 1 (token halves)
            if (pw < 2) {
                float accA[2][4] = {}, accP[2][4] = {};
#pragma unroll
                for (int kt = 0; kt < D / 16; ++kt) {
                    const int i = lane >> 3;
                    const int ra_ = (i & 1) * 8 + (lane & 7), ca = kt * 16 + (i >> 1) * 8;
                    uint32_t a[4], aq[4], b0, b1;
                    ldsm_x4(smem_u32(Kt + ra_ * LDP + ca), a[0], a[1], a[2], a[3]);
                    ldsm_x4(smem_u32(Pq + ra_ * LDP + ca), aq[0], aq[1], aq[2], aq[3]);
                    const int rb = pw * 8 + (lane & 7), cb = kt * 16 + ((lane >> 3) & 1) * 8;
                    ldsm_x2(smem_u32(Kh + rb * LDP + cb), b0, b1);
                    mma16816(accA[kt & 1], a, b0, b1);
                    mma16816(accP[kt & 1], aq, b0, b1);
                }
                __nv_bfloat16 *Pp = reinterpret_cast<__nv_bfloat16 *>(slot + OFF_PP);
                const int r0 = lane >> 2, j0 = pw * 8 + 2 * (lane & 3);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int r = r0 + 8 * hh;
                    float pv[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int j = j0 + e;
                        const float va = accA[0][2 * hh + e] + accA[1][2 * hh + e];
                        const float vp = accP[0][2 * hh + e] + accP[1][2 * hh + e];
                        As[r * C + j] = j < r ? bs[r] * va : 0.f;
                        pv[e] = j <= r ? vp : 0.f;
                    }
                    *reinterpret_cast<uint32_t *>(Pp + r * LDS + j0) = pack_bf16(pv[0], pv[1]);
                }
            }
            named_sync(1, nt);
            // -- TB = (I + A)^-1 diag(beta): forward substitution, one column per lane
            if (pw == 0 && lane < C) {
                const int j = lane;
                float x[C];
#pragma unroll
                for (int r = 0; r < C; ++r) {
                    float acc = r == j ? 1.f : 0.f;
#pragma unroll
                    for (int i = 0; i < r; ++i) acc = fmaf(-As[r * C + i], x[i], acc);
                    x[r] = acc;
                }
                __nv_bfloat16 *Ptb = reinterpret_cast<__nv_bfloat16 *>(slot + OFF_PTB);
                const float bj = bs[j];
#pragma unroll
                for (int r = 0; r < C; ++r) Ptb[r * LDS + j] = __float2bfloat16_rn(x[r] * bj);
            }
            named_sync(1, nt);
            // -- -W = -TB K~: warp pw covers key channels [32 pw, 32 pw + 32)
            {
                const __nv_bfloat16 *Ptb = reinterpret_cast<const __nv_bfloat16 *>(slot + OFF_PTB);
                __nv_bfloat16 *Pw = reinterpret_cast<__nv_bfloat16 *>(slot + OFF_PW);
                uint32_t tb[4];
                {
                    const int i = lane >> 3;
                    const int r = (i & 1) * 8 + (lane & 7), j = (i >> 1) * 8;
                    ldsm_x4(smem_u32(Ptb + r * LDS + j), tb[0], tb[1], tb[2], tb[3]);
                }
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int cb = pw * 32 + half * 16;
                    const int i = lane >> 3;
                    const int j = (i & 1) * 8 + (lane & 7), cc = cb + (i >> 1) * 8;
                    uint32_t k0, k1, k2, k3;
                    ldsm_x4_t(smem_u32(Kt + j * LDP + cc), k0, k1, k2, k3);
                    float acc0[4] = {}, acc1[4] = {};
                    mma16816(acc0, tb, k0, k1);
                    mma16816(acc1, tb, k2, k3);
                    const int r = lane >> 2, col = cb + 2 * (lane & 3);
                    *reinterpret_cast<uint32_t *>(Pw + r * LDP + col) = pack_bf16(-acc0[0], -acc0[1]);
                    *reinterpret_cast<uint32_t *>(Pw + (r + 8) * LDP + col) = pack_bf16(-acc0[2], -acc0[3]);
                    *reinterpret_cast<uint32_t *>(Pw + r * LDP + col + 8) = pack_bf16(-acc1[0], -acc1[1]);
                    *reinterpret_cast<uint32_t *>(Pw + (r + 8) * LDP + col + 8) = pack_bf16(-acc1[2], -acc1[3]);
                }
            }
            fence_proxy_async();  // generic writes of the slot -> async-proxy bulk reads
            named_sync(1, nt);
            if (c == 0) {
                if (kShare) {
                    const uint32_t src = sbase + SM_PROD + s * SLOT_BYTES;
#pragma unroll
                    for (uint32_t peer = 0; peer < (uint32_t)kCS; ++peer) {
                        if (peer == rank) continue;
                        bulk_copy_to_peer(map_to_rank(src, peer), src, SLOT_BYTES,
                                          map_to_rank(bar(B_FULL(s)), peer));
                    }
                }
                mbar_arrive(bar(B_FULL(s)));  // own state warps
            }
        }
    } else {
        // ------------------------------------------------ state warps
        const int sw = warp - 1 - NPW;  // 0 .. NSW-1
        const int vrow0 = (int)rank * VB + sw * 16;  // first value column (row of S^T)
        const int g4 = lane >> 2, l4 = lane & 3;
        const size_t sidx = ((size_t)seq * H + head) * D * D;
        float S[16][4];  // S^T fragments: n-tile j covers key channels 8j .. 8j+7
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int kc = 8 * j + 2 * l4, v0 = vrow0 + g4;
            if (p.h0) {
                S[j][0] = p.h0[sidx + (size_t)kc * D + v0];
                S[j][1] = p.h0[sidx + (size_t)(kc + 1) * D + v0];
                S[j][2] = p.h0[sidx + (size_t)kc * D + v0 + 8];
                S[j][3] = p.h0[sidx + (size_t)(kc + 1) * D + v0 + 8];
            } else {
                S[j][0] = S[j][1] = S[j][2] = S[j][3] = 0.f;
            }
        }
        const float scale = rsqrtf((float)D);
        __nv_bfloat16 *ost = reinterpret_cast<__nv_bfloat16 *>(sm + SM_OST) + sw * C * LDS;
        for (int n = 0; n < nchunks; ++n) {
            const int s = n % NP, use = n / NP;
            const bool ok = mbar_wait<false>(bar(B_FULL(s)), use & 1);
            if (__any_sync(0xffffffffu, !ok)) break;
            const unsigned char *slot = sm + SM_PROD + s * SLOT_BYTES;
            const __nv_bfloat16 *Pq = reinterpret_cast<const __nv_bfloat16 *>(slot + OFF_PQ);
            const __nv_bfloat16 *Pw = reinterpret_cast<const __nv_bfloat16 *>(slot + OFF_PW);
            const __nv_bfloat16 *Pk = reinterpret_cast<const __nv_bfloat16 *>(slot + OFF_PK);
            const __nv_bfloat16 *Ptb = reinterpret_cast<const __nv_bfloat16 *>(slot + OFF_PTB);
            const __nv_bfloat16 *Pp = reinterpret_cast<const __nv_bfloat16 *>(slot + OFF_PP);
            const float *Pg = reinterpret_cast<const float *>(slot + OFF_PG);
            const __nv_bfloat16 *Vs = reinterpret_cast<const __nv_bfloat16 *>(sm + SM_V + s * V_BYTES);
            const int i8 = lane >> 3, r8 = lane & 7;

            // U~^T = V^T TB^T  (initial value of the U^T accumulators)
            float accU[2][2][4] = {};  // [k parity][token n-tile][frag]
            {
                uint32_t va[4], tb[4];
                const int t = (i8 >> 1) * 8 + r8, vv = sw * 16 + (i8 & 1) * 8;
                ldsm_x4_t(smem_u32(Vs + t * VB + vv), va[0], va[1], va[2], va[3]);
                const int r = (i8 >> 1) * 8 + r8, j = (i8 & 1) * 8;
                ldsm_x4(smem_u32(Ptb + r * LDS + j), tb[0], tb[1], tb[2], tb[3]);
                mma16816(accU[0][0], va, tb[0], tb[1]);
                mma16816(accU[0][1], va, tb[2], tb[3]);
            }
            // S^T as bf16 A fragments
            uint32_t Sa[8][4];
#pragma unroll
            for (int kt = 0; kt < 8; ++kt) {
                Sa[kt][0] = pack_bf16(S[2 * kt][0], S[2 * kt][1]);
                Sa[kt][1] = pack_bf16(S[2 * kt][2], S[2 * kt][3]);
                Sa[kt][2] = pack_bf16(S[2 * kt + 1][0], S[2 * kt + 1][1]);
                Sa[kt][3] = pack_bf16(S[2 * kt + 1][2], S[2 * kt + 1][3]);
            }
            // U^T += S^T (-W)^T
#pragma unroll
            for (int kt = 0; kt < 8; ++kt) {
                uint32_t w0, w1, w2, w3;
                const int r = (i8 >> 1) * 8 + r8, cc = kt * 16 + (i8 & 1) * 8;
                ldsm_x4(smem_u32(Pw + r * LDP + cc), w0, w1, w2, w3);
                mma16816(accU[kt & 1][0], Sa[kt], w0, w1);
                mma16816(accU[kt & 1][1], Sa[kt], w2, w3);
            }
            uint32_t Ua[4];
            Ua[0] = pack_bf16(accU[0][0][0] + accU[1][0][0], accU[0][0][1] + accU[1][0][1]);
            Ua[1] = pack_bf16(accU[0][0][2] + accU[1][0][2], accU[0][0][3] + accU[1][0][3]);
            Ua[2] = pack_bf16(accU[0][1][0] + accU[1][1][0], accU[0][1][1] + accU[1][1][1]);
            Ua[3] = pack_bf16(accU[0][1][2] + accU[1][1][2], accU[0][1][3] + accU[1][1][3]);
            // O^T = S^T Q~^T + U^T P^T  (uses the state before this chunk's update)
            float accO[2][2][4] = {};
#pragma unroll
            for (int kt = 0; kt < 8; ++kt) {
                uint32_t q0, q1, q2, q3;
                const int r = (i8 >> 1) * 8 + r8, cc = kt * 16 + (i8 & 1) * 8;
                ldsm_x4(smem_u32(Pq + r * LDP + cc), q0, q1, q2, q3);
                mma16816(accO[kt & 1][0], Sa[kt], q0, q1);
                mma16816(accO[kt & 1][1], Sa[kt], q2, q3);
            }
            {
                uint32_t p0, p1, p2, p3;
                const int r = (i8 >> 1) * 8 + r8, j = (i8 & 1) * 8;
                ldsm_x4(smem_u32(Pp + r * LDS + j), p0, p1, p2, p3);
                mma16816(accO[0][0], Ua, p0, p1);
                mma16816(accO[0][1], Ua, p2, p3);
            }
            // S^T <- S^T diag(gamma_L) + U^T K'
#pragma unroll
            for (int np = 0; np < 8; ++np) {
                const float2 g0 = *reinterpret_cast<const float2 *>(Pg + 16 * np + 2 * l4);
                const float2 g1 = *reinterpret_cast<const float2 *>(Pg + 16 * np + 8 + 2 * l4);
                S[2 * np][0] *= g0.x; S[2 * np][1] *= g0.y; S[2 * np][2] *= g0.x; S[2 * np][3] *= g0.y;
                S[2 * np + 1][0] *= g1.x; S[2 * np + 1][1] *= g1.y;
                S[2 * np + 1][2] *= g1.x; S[2 * np + 1][3] *= g1.y;
                uint32_t k0, k1, k2, k3;
                const int t = (i8 & 1) * 8 + r8, cc = np * 16 + (i8 >> 1) * 8;
                ldsm_x4_t(smem_u32(Pk + t * LDP + cc), k0, k1, k2, k3);
                mma16816(S[2 * np], Ua, k0, k1);
                mma16816(S[2 * np + 1], Ua, k2, k3);
            }
            // release the slot (V tile and products) to the producer and the owner
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(B_FREE(s)));
                if (kShare)
                    mbar_arrive_remote(map_to_rank(bar(B_CFREE(s)), owner(n)));
                else
                    mbar_arrive(bar(B_CFREE(s)));
            }
            // output tile: scale, bf16, transpose through shared memory, 16-byte stores
            {
                uint32_t o0 = pack_bf16(scale * (accO[0][0][0] + accO[1][0][0]),
                                        scale * (accO[0][0][1] + accO[1][0][1]));
                uint32_t o1 = pack_bf16(scale * (accO[0][0][2] + accO[1][0][2]),
                                        scale * (accO[0][0][3] + accO[1][0][3]));
                uint32_t o2 = pack_bf16(scale * (accO[0][1][0] + accO[1][1][0]),
                                        scale * (accO[0][1][1] + accO[1][1][1]));
                uint32_t o3 = pack_bf16(scale * (accO[0][1][2] + accO[1][1][2]),
                                        scale * (accO[0][1][3] + accO[1][1][3]));
                // matrices: (v 0-7, t 0-7), (v 8-15, t 0-7), (v 0-7, t 8-15), (v 8-15, t 8-15)
                const int t = (i8 >> 1) * 8 + r8, vv = (i8 & 1) * 8;
                stsm_x4_t(smem_u32(ost + t * LDS + vv), o0, o1, o2, o3);
                __syncwarp();
                const int c0 = t0 + n * C;
                const int L = min(C, t1 - c0);
                const int tt = lane >> 1, hv = (lane & 1) * 8;
                if (tt < L) {
                    const uint4 val = *reinterpret_cast<const uint4 *>(ost + tt * LDS + hv);
                    *reinterpret_cast<uint4 *>(p.out + ((size_t)(c0 + tt) * H + head) * D +
                                               vrow0 + hv) = val;
                }
                __syncwarp();
            }
        }
        if (p.h_final) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int kc = 8 * j + 2 * l4, v0 = vrow0 + g4;
                p.h_final[sidx + (size_t)kc * D + v0] = S[j][0];
                p.h_final[sidx + (size_t)(kc + 1) * D + v0] = S[j][1];
                p.h_final[sidx + (size_t)kc * D + v0 + 8] = S[j][2];
                p.h_final[sidx + (size_t)(kc + 1) * D + v0 + 8] = S[j][3];
            }
        }
    }
    // no CTA may leave while a peer can still write into its shared memory
    __syncwarp();
    if (kShare) cluster_sync();
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

bool encode_map(CUtensorMap *m, const void *base, bool f32, int64_t n_tok, int H, int box_x) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t es = f32 ? 4 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)n_tok};
    cuuint64_t strides[2] = {D * es, (cuuint64_t)H * D * es};
    cuuint32_t box[3] = {(cuuint32_t)box_x, 1, (cuuint32_t)C};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                     const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <bool kShare>
cudaError_t launch_tc_t(const FwdArgs &a, cudaStream_t stream) {
    CUtensorMap mq, mk, ma, mv;
    if (!encode_map(&mq, a.q, false, a.n_tok, a.n_heads, D) ||
        !encode_map(&mk, a.k, false, a.n_tok, a.n_heads, D) ||
        !encode_map(&ma, a.a, true, a.n_tok, a.n_heads, D) ||
        !encode_map(&mv, a.v, false, a.n_tok, a.n_heads, VB))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kda_tc_kernel<kShare>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    TcParams p;
    p.beta = a.beta; p.h0 = a.h0; p.cu = a.cu_seqlens;
    p.out = reinterpret_cast<__nv_bfloat16 *>(a.out); p.h_final = a.h_final;
    p.n_seq = a.n_seq; p.H = a.n_heads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((int64_t)a.n_seq * a.n_heads * kCS));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kShare ? kCS : 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kda_tc_kernel<kShare>, mq, mk, ma, mv, p);
    if (e == cudaSuccess) count_launches(1);
    return e;
}

}  // namespace

bool tc_supported(const FwdArgs &a) {
    return a.bf16 && a.d_k == D && a.d_v == D && a.n_tok > 0 &&
           (int64_t)a.n_seq * a.n_heads * kCS < 0x7fffffffLL && a.n_tok < 0x7fffffffLL;
}

cudaError_t launch_tc(const FwdArgs &a, cudaStream_t stream) {
#ifdef KDA_TC_NO_CLUSTER
    return launch_tc_t<false>(a, stream);
#else
    return launch_tc_t<true>(a, stream);
#endif
}

cudaError_t read_device_flags(unsigned int *flags, bool reset, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(flags, g_device_flags, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess || !reset) return e;
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_device_flags, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                                stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}

}  // namespace kda
