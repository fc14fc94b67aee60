// kda_tc.cu -- tensor-core kernel for the chunked KDA forward pass, bf16 I/O,
// d_k = d_v = 128, fp32 state and accumulation, for sm_103a.
//
// Work decomposition. One thread-block cluster of kCS = 4 CTAs per (sequence,
// head). CTA rank r owns value columns [32 r, 32 r + 32) of the state, i.e. 32 rows
// of S^T (d_v x d_k), held in registers by two "state" warps (16 rows each) for the
// whole sequence. Columns of the state evolve independently, so the four CTAs of a
// head never exchange state. What they share is the per-chunk "prologue" -- the gate,
// the in-chunk cumulative decay and the diagonal (intra-chunk) tile -- which does not
// depend on the state: chunk n's prologue is computed once, by CTA n mod 4, and copied
// into every CTA's ring slot (its own included) with DSMEM bulk copies. Per CTA, two
// state warps carry the serial chain, two output warps form the outputs from the bf16
// state the state warps hand them, and two prologue groups of four warps alternate over
// the CTA's own chunks.
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
// into mbarrier-tracked rings. Prologue products are computed into a per-group staging
// buffer and copied into every CTA's ring slot by cp.async.bulk shared::cta ->
// shared::cluster, completing on the receiver's mbarrier; two forwarding warps tell the
// owner when a CTA has freed a slot and when a copy has landed. Every wait is bounded: a
// wait that exceeds its limit sets a device flag (kda_read_device_flags), releases every
// other wait in the grid and lets the kernel finish with unspecified output.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_internal.h"

namespace kda {

__device__ unsigned int g_device_flags;  // bit 0: a pipeline wait exceeded its limit

// Phase timestamps (SM clock) of the first cluster, first 32 chunks: a profiling aid
// compiled only with -DKDA_TC_TRACE; the default build has no trace code. Stamps go to
// shared memory and are copied out when the CTA finishes, so that tracing adds no
// global stores to the pipeline. Slots: 0/1 producer loop top / slot free; 2 raw tiles
// requested; 3/4 prologue group loop top / inputs in; 5-8 gate, A and P, solve, W done;
// 9 copies issued; 10-13 state warp iteration top / chain done / handoff published /
// iteration end; 14 output warp done; 15 receipt forwarder saw the products land.
#ifdef KDA_TC_TRACE
__device__ long long g_trace[4][32][16];
__device__ __forceinline__ long long trace_clock() {
#ifdef KDA_TC_TRACE_GLOBALTIMER
    long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
#else
    return clock64();
#endif
}
#define KDA_TRACE(n, slot)                                                              \
    do {                                                                                \
        if ((n) < 32)                                                                   \
            reinterpret_cast<long long *>(sm + SM_TRACE)[(n) * 16 + (slot)] = trace_clock(); \
    } while (0)
#else
#define KDA_TRACE(n, slot) \
    do {                   \
    } while (0)
#endif

namespace {

constexpr int D = 128;          // d_k = d_v
constexpr int C = kChunk;       // 16 tokens
constexpr int kCS = 4;          // CTAs per (sequence, head) = cluster size
constexpr int VB = D / kCS;     // value columns per CTA (32)
static_assert(VB * 2 == 64, "the v tile rows are one 64-byte swizzle span");
constexpr int NSW = VB / 16;    // state warps per CTA (2), 16 value columns each, and as
                                // many output warps
constexpr int NGRP = 2;         // prologue groups, alternating owned chunks
constexpr int NPW = 4;          // warps per prologue group (one key channel per thread)
// Warp roles by warpgroup: 0 = producer warp (+ 3 idle warps), 1 and 2 = the prologue
// groups, 3 = state warps then output warps.
constexpr int W_PRO0 = 4;                      // first prologue warp
constexpr int W_STATE0 = W_PRO0 + NGRP * NPW;  // first state warp
constexpr int W_OUT0 = W_STATE0 + NSW;         // first output warp
constexpr int kThreads = 32 * (W_OUT0 + NSW);  // 512
// Registers per thread. The block is launched with kRegsLaunch for every thread; each
// warpgroup then moves to its own allotment (setmaxnreg), and the allotments add up to
// the launch total, so every increase is covered by the decreases. The state and output
// warps need the room: 64 fp32 state values plus their bf16 copy plus ~100 registers of
// operand fragments are live at once.
constexpr int kRegsLaunch = 128, kRegsProducer = 40, kRegsPrologue = 120, kRegsConsumer = 232;
static_assert(kThreads == 512 && NGRP == 2 && NPW == 4 && NSW == 2, "one warpgroup per role");
static_assert(kRegsProducer + NGRP * kRegsPrologue + kRegsConsumer == 4 * kRegsLaunch,
              "warpgroup register allotments must add up to the launch allotment");
static_assert(kRegsLaunch * kThreads == 65536, "the launch takes the whole register file");
constexpr int NP = 8;           // product-ring depth (multiple of kCS)
constexpr int LDP = 136;        // pitch (elements) of 16 x 128 bf16 tiles: 272 B rows
constexpr int LDS = 24;         // pitch of 16 x 16 bf16 tiles: 48 B rows
constexpr long long kWaitLimit = 4000000000LL;  // cycles (~2 s) before a wait gives up

static_assert(NP % kCS == 0, "slot ownership must be static");

// Channel-major 128 x 16 bf16 tiles ("[c][t]"): one 32-byte row per key channel c
// holding its 16 tokens; the two 16-byte halves of a row swap places every four rows,
// which keeps 8-row ldmatrix accesses free of bank conflicts without padding.
__device__ __forceinline__ uint32_t cmaj(int c, int t0) {
    return (uint32_t)(c * 32 + ((((t0 >> 3) ^ (c >> 2)) & 1) << 4));
}
constexpr int CMAJ_BYTES = D * C * 2;  // 4096

// ---- shared-memory layout (bytes) ----
// product slot: everything the state warps need for one chunk
constexpr int OFF_PQ = 0;                        // Q~ [c][t] bf16, channel-major
constexpr int OFF_PW = OFF_PQ + CMAJ_BYTES;      // -W [16][LDP] bf16, token-major
constexpr int OFF_PK = OFF_PW + C * LDP * 2;     // K' [c][t] bf16, channel-major
constexpr int OFF_PTB = OFF_PK + CMAJ_BYTES;     // TB [16][LDS] bf16
constexpr int OFF_PP = OFF_PTB + C * LDS * 2;    // P  [16][LDS] bf16
constexpr int OFF_PG = OFF_PP + C * LDS * 2;     // gamma_L [128] f32, permuted (gperm)
constexpr int SLOT_BYTES = OFF_PG + D * 4;       // 14592
static_assert(SLOT_BYTES % 16 == 0, "bulk copies move 16-byte multiples");

// raw slot (one per prologue group): the owner's TMA tiles of one chunk
constexpr int RAW_Q = 0, RAW_K = C * D * 2, RAW_A = 2 * C * D * 2;
constexpr int RAW_BYTES = RAW_A + C * D * 4;     // 16384 (q, k, a)
constexpr int V_BYTES = C * VB * 2;              // 1024
// prologue-group scratch
constexpr int GS_KT = 0;                         // K~ [c][t]
constexpr int GS_KH = GS_KT + CMAJ_BYTES;        // K^ [c][t]
constexpr int GS_A = GS_KH + CMAJ_BYTES;         // A  [16][16] f32
constexpr int GS_BETA = GS_A + C * C * 4;        // beta [2][16] f32 (double buffer)
constexpr int GS_BYTES = GS_BETA + 2 * C * 4;
// state -> output warp handoff: [state warp][2 buffers][32 lanes][36 u32]
constexpr int HO_LANE = 36 * 4;
constexpr int HO_BYTES = 32 * HO_LANE;

constexpr int SM_RAW = 0;
constexpr int SM_V = SM_RAW + NGRP * RAW_BYTES;
constexpr int SM_PROD = SM_V + NP * V_BYTES;
constexpr int SM_STAGE = SM_PROD + NP * SLOT_BYTES;  // one product staging buffer per group
constexpr int SM_GS = SM_STAGE + NGRP * SLOT_BYTES;
constexpr int SM_HO = (SM_GS + NGRP * GS_BYTES + 127) / 128 * 128;
constexpr int SM_BAR = SM_HO + NSW * 2 * HO_BYTES;
constexpr int NBARS = 2 * NP + NGRP * kCS + 2 * NGRP + 4 * NSW;
constexpr int SM_MISC = SM_BAR + NBARS * 8;
#ifdef KDA_TC_TRACE
constexpr int SM_TRACE = SM_MISC + 64;
constexpr int SMEM_BYTES = SM_TRACE + 32 * 16 * 8;
#else
constexpr int SMEM_BYTES = SM_MISC + 64;
#endif
static_assert(RAW_BYTES % 128 == 0 && SM_V % 128 == 0 && SM_PROD % 128 == 0, "TMA alignment");
static_assert(SM_STAGE % 16 == 0 && SM_GS % 16 == 0 && GS_BYTES % 16 == 0 && SM_HO % 16 == 0,
              "alignment");
static_assert(SM_BAR % 8 == 0, "alignment");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

// gamma_L[c], c = 16 np + 8 h + 2 l4 + e, is stored at 16 np + 4 l4 + 2 h + e: the lane
// holding S^T columns 2 l4 (+1, +8, +9) of 16-column group np reads its four decay
// factors as one float4, and the four lanes l4 = 0..3 read 64 contiguous bytes (one
// conflict-free shared-memory access)
__host__ __device__ constexpr int gperm(int c) {
    return ((c >> 4) * 4 + ((c >> 1) & 3)) * 4 + ((c >> 3) & 1) * 2 + (c & 1);
}

// Barrier indices. Slot s of every CTA is filled by CTA s % kCS (the owner of the chunks
// n with n % NP == s), from the staging buffer of its group s / kCS.
__host__ __device__ constexpr int B_FULL(int s) { return s; }       // products + V of slot s in
__host__ __device__ constexpr int B_FREE(int s) { return NP + s; }  // local consumers done with s
// (owner side) CTA p has consumed the previous chunk of the group-g slot
__host__ __device__ constexpr int B_PFREE(int g, int p) { return 2 * NP + kCS * g + p; }
// (owner side) all CTAs have received group g's last copy: its staging buffer is free
__host__ __device__ constexpr int B_RECV(int g) { return 2 * NP + kCS * NGRP + g; }
__host__ __device__ constexpr int B_RFULL(int g) { return 2 * NP + kCS * NGRP + NGRP + g; }  // raw tiles
__host__ __device__ constexpr int B_HFULL(int w, int b) { return 2 * NP + kCS * NGRP + 2 * NGRP + 2 * w + b; }
__host__ __device__ constexpr int B_HEMPTY(int w, int b) {
    return 2 * NP + kCS * NGRP + 2 * NGRP + 2 * NSW + 2 * w + b;
}
static_assert(NP == NGRP * kCS, "each slot belongs to one group of one owner");

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
// arrive without release semantics: for "these reads have completed" signals, whose
// values the arriving warp has already consumed
__device__ __forceinline__ void mbar_arrive_relaxed(uint32_t a) {
    asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t a, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes)
                 : "memory");
}
// Remote arrive without release semantics. Measured: a cluster-scope release arrive
// costs the issuing thread well over a thousand cycles, which paced the whole pipeline.
// Used only for signals that order no memory accesses of their own: "the slot's reads
// have completed" (the values were already consumed) and "the copy has landed".
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t a, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok) : "r"(a), "r"(parity) : "memory");
    return ok != 0;
}
// non-blocking probe of a phase (never suspends the thread)
__device__ __forceinline__ bool mbar_test(uint32_t a, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
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
__device__ __forceinline__ bool mbar_wait(uint32_t a, uint32_t parity,
                                          long long limit = kWaitLimit) {
    if (kClusterScope ? mbar_try_cluster(a, parity) : mbar_try(a, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (kClusterScope ? mbar_try_cluster(a, parity) : mbar_try(a, parity)) return true;
        if ((it & 63u) == 0) {
            if (*(volatile unsigned int *)&g_device_flags != 0u) return false;
            if (clock64() - t0 > limit) {
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
// transpose of an 8 x 8 b16 matrix held in mma fragment layout (one warp)
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
// D (16x8 f32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma16816(float *d, const uint32_t *a, uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// warpgroup-wide register reallocation; all four warps of the warpgroup execute it
template <int R>
__device__ __forceinline__ void regs_increase() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}
template <int R>
__device__ __forceinline__ void regs_decrease() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}
// (a, b) *= (ga, gb) as one packed f32x2 multiply
__device__ __forceinline__ void mul2(float &a, float &b, float ga, float gb) {
    asm("{ .reg .b64 x, y; mov.b64 x, {%0, %1}; mov.b64 y, {%2, %3}; mul.rn.f32x2 x, x, y; "
        "mov.b64 {%0, %1}, x; }"
        : "+f"(a), "+f"(b) : "f"(ga), "f"(gb));
}
__device__ __forceinline__ float ex2_approx(float x) {  // 2^x, flushes denormals
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {  // 1/x; 1/inf = 0
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr float kLog2e = 1.4426950408889634f;  // log2(e): exp(x) = 2^(x log2 e)
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (lower address)
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes) : "memory");
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

__global__ void __launch_bounds__(kThreads, 1)
    kda_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_v,
                  const TcParams p) {
    extern __shared__ __align__(128) unsigned char sm[];
    const uint32_t sbase = smem_u32(sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int ci = blockIdx.x / kCS;
    int *misc = reinterpret_cast<int *>(sm + SM_MISC);
    resolve_item(p, ci, &misc[0], &misc[1]);
    const int seq = misc[0], head = misc[1];
    const int H = p.H;
    const int t0 = p.cu[seq], t1 = p.cu[seq + 1];
    const int nchunks = (t1 - t0 + C - 1) / C;
    auto bar = [&](int i) { return sbase + SM_BAR + 8u * (uint32_t)i; };
    auto owner = [&](int n) -> uint32_t { return (uint32_t)(n % kCS); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < NP; ++s) {
            mbar_init(bar(B_FULL(s)), 1);        // producer (expects V and the product copy)
            mbar_init(bar(B_FREE(s)), 2 * NSW);  // state and output warps
        }
        for (int g = 0; g < NGRP; ++g) {
            for (int q = 0; q < kCS; ++q) mbar_init(bar(B_PFREE(g, q)), 1);
            mbar_init(bar(B_RECV(g)), kCS);
            mbar_init(bar(B_RFULL(g)), 1);
        }
        for (int w = 0; w < NSW; ++w)
            for (int b = 0; b < 2; ++b) {
                mbar_init(bar(B_HFULL(w, b)), 1);
                mbar_init(bar(B_HEMPTY(w, b)), 1);
            }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
#ifdef KDA_TC_TRACE
    for (int i = threadIdx.x; i < 32 * 16; i += blockDim.x)
        reinterpret_cast<long long *>(sm + SM_TRACE)[i] = 0;
#endif
    cluster_sync();

    if (warp < W_PRO0) {
        regs_decrease<kRegsProducer>();
        if (warp == 0) {
            // -------------------------------------------- producer warp
            // Lane 0 loads the v tiles by TMA once the slot is free locally (the owner's
            // prologue loads q, k and the gate logits itself).
            for (int n = 0; n < nchunks; ++n) {
                const int s = n % NP, use = n / NP;
                KDA_TRACE(n, 0);
                int ok = 1;
                if (lane == 0) ok = mbar_wait<false>(bar(B_FREE(s)), (use & 1) ^ 1);
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
                KDA_TRACE(n, 1);
                if (lane == 0) {
                    mbar_arrive_tx(bar(B_FULL(s)), V_BYTES + SLOT_BYTES);
                    tma_load_3d(sbase + SM_V + s * V_BYTES, &tm_v, (int)rank * VB, head,
                                t0 + n * C, bar(B_FULL(s)));
                }
                __syncwarp();
            }
        } else if (warp == 1) {
            // -------------------------------------------- release forwarder
            // Lane 0 tells the owner of chunk n that this CTA has consumed chunk n - NP, the
            // previous occupant of slot n % NP, so the owner may copy chunk n into it. A
            // cluster-scope release waits for the issuing thread's earlier memory
            // operations -- including, as measured, TMA loads still in flight -- so these
            // signals come from threads that have no memory operations of their own.
            if (lane == 0) {
                for (int n = NP; n < nchunks; ++n) {
                    const int s = n % NP, use = n / NP;
                    if (!mbar_wait<false>(bar(B_FREE(s)), (use & 1) ^ 1)) break;
                    mbar_arrive_remote_relaxed(map_to_rank(bar(B_PFREE(s / kCS, (int)rank)), owner(n)));
                }
            }
            __syncwarp();
        } else if (warp == 2) {
            // -------------------------------------------- receipt forwarder
            // Lane 0 tells the owner of chunk n that its copy of chunk n has landed here, so
            // that once every CTA has it the owner may reuse the staging buffer for chunk
            // n + NP. (Slot n % NP cannot be refilled before this thread has seen the
            // phase: the refill needs this very signal.)
            if (lane == 0) {
                for (int n = 0; n + NP < nchunks; ++n) {
                    const int s = n % NP, use = n / NP;
                    if (!mbar_wait<false>(bar(B_FULL(s)), use & 1)) break;
                    KDA_TRACE(n, 15);
                    mbar_arrive_remote_relaxed(map_to_rank(bar(B_RECV(s / kCS)), owner(n)));
                }
            }
            __syncwarp();
        }
        // warp 3 only holds registers back for the consumers
    } else if (warp < W_STATE0) {
        regs_decrease<kRegsPrologue>();
        // ------------------------------------------------ prologue groups
        // Group g of owner CTA r handles the chunks n with n % NP == r + kCS g, i.e. the
        // chunks of slot r + kCS g. It computes a chunk's products into its staging
        // buffer as soon as every CTA has received the previous copy out of it, then
        // copies them into each CTA's slot as soon as that CTA has consumed the slot's
        // previous chunk.
        const int g = (warp - W_PRO0) / NPW;
        const int pw = (warp - W_PRO0) % NPW;
        const int c = threadIdx.x - 32 * (W_PRO0 + NPW * g);  // key channel of the gate pass
        const int nt = 32 * NPW;
        const int bar_id = 1 + g;
        // the thread that waits, issues the TMA loads and the product copies, and the
        // warp that fetches beta: both on the group's warps 2 and 3, which share no
        // scheduler with the state warps
        constexpr int kLead = 64;
        unsigned char *gs = sm + SM_GS + g * GS_BYTES;
        unsigned char *KtB = gs + GS_KT;  // K~ [c][t]
        unsigned char *KhB = gs + GS_KH;  // K^ [c][t]
        const uint32_t Kt_s = smem_u32(KtB), Kh_s = smem_u32(KhB);
        float *As = reinterpret_cast<float *>(gs + GS_A);
        const int i8 = lane >> 3, r8 = lane & 7;
        const uint32_t raw_s = sbase + SM_RAW + g * RAW_BYTES;
        const unsigned char *raw = sm + SM_RAW + g * RAW_BYTES;
        // q, k and gate-logit tiles of chunk n into this group's raw slot (the lead
        // thread), beta of chunk n into beta buffer b (warp 3's lanes 0-15, cp.async,
        // which no barrier or fence of another thread waits for)
        auto fetch = [&](int n, int b) {
            if (n >= nchunks) return;
            const int c0n = t0 + n * C;
            if (c == kLead) {
                mbar_arrive_tx(bar(B_RFULL(g)), RAW_BYTES);
                tma_load_3d(raw_s + RAW_Q, &tm_q, 0, head, c0n, bar(B_RFULL(g)));
                tma_load_3d(raw_s + RAW_K, &tm_k, 0, head, c0n, bar(B_RFULL(g)));
                tma_load_3d(raw_s + RAW_A, &tm_a, 0, head, c0n, bar(B_RFULL(g)));
                KDA_TRACE(n, 2);
            }
            if (pw == 3) {
                if (lane < C) {
                    const int row = c0n + lane;
                    const bool in = row < t1;
                    cp_async_4(smem_u32(gs + GS_BETA) + (b * C + lane) * 4,
                               p.beta + (size_t)(in ? row : t0) * H + head, in ? 4u : 0u);
                }
                asm volatile("cp.async.commit_group;" ::: "memory");
            }
        };
        fetch((int)rank + kCS * g, 0);
        int k = 0;  // chunks this group has processed (= n / NP)
        for (int n = (int)rank + kCS * g; n < nchunks; n += NP, ++k) {
            const int s = n % NP;
            const int c0 = t0 + n * C;
            const int L = min(C, t1 - c0);
            if (c == kLead) KDA_TRACE(n, 3);
            // one thread waits on the pipeline; the rest of the group blocks on the
            // hardware named barrier, then observes the completed phases once
            bool bad = false;
            if (c == kLead) {
                bad = !mbar_wait<false>(bar(B_RFULL(g)), k & 1);
                if (k > 0) bad |= !mbar_wait<true>(bar(B_RECV(g)), (k & 1) ^ 1);
            }
            if (pw == 3) asm volatile("cp.async.wait_group 0;" ::: "memory");  // this chunk's beta
            if (named_sync_or(bar_id, nt, bad)) break;
            if (c != kLead) {  // acquire the completed phases (they do not block now)
                mbar_try(bar(B_RFULL(g)), k & 1);
                if (k > 0) mbar_try_cluster(bar(B_RECV(g)), (k & 1) ^ 1);
            }
            if (c == kLead) KDA_TRACE(n, 4);
            const float *bs = reinterpret_cast<const float *>(gs + GS_BETA) + (k & 1) * C;
            // this group's staging buffer, laid out as a slot
            unsigned char *slot = sm + SM_STAGE + g * SLOT_BYTES;
            const uint32_t slot_s = sbase + SM_STAGE + g * SLOT_BYTES;
            float *Pg = reinterpret_cast<float *>(slot + OFF_PG);
            const __nv_bfloat16 *rq = reinterpret_cast<const __nv_bfloat16 *>(raw + RAW_Q);
            const __nv_bfloat16 *rk = reinterpret_cast<const __nv_bfloat16 *>(raw + RAW_K);
            const float *ra = reinterpret_cast<const float *>(raw + RAW_A);
            // -- gate pass: one key channel at a time, 16 tokens in order; outputs are
            //    written channel-major as packed bf16 pairs, 16 bytes at a time. Only the
            //    group's warps 2 and 3 run it (two channels per thread): warps 0 and 1 share
            //    their schedulers with the state warps, whose chain this arithmetic would
            //    slow (measured: 3 % on the 64K workload).
            if (pw >= 2)
#pragma unroll 1
            for (int rep = 0; rep < 2; ++rep) {
                const int c = 32 * (pw - 2) + lane + 64 * rep;
                // rows past the end hold another sequence's (finite) data or TMA
                // zeros: compute every row, then select, in separate passes so that
                // the 16 independent exponential chains overlap
                float eg[C], kk[C], qq[C];
#pragma unroll
                for (int r = 0; r < C; ++r) eg[r] = ra[r * D + c];
#pragma unroll
                for (int r = 0; r < C; ++r)  // sigmoid(a) = 1 / (1 + exp(-a))
                    eg[r] = rcp_approx(1.f + ex2_approx(-kLog2e * eg[r]));
#pragma unroll
                for (int r = 0; r < C; ++r) {  // exp(g), g = -5 sigmoid(a)
                    const float e = ex2_approx((kGMin * kLog2e) * eg[r]);
                    eg[r] = r < L ? e : 1.f;
                    qq[r] = r < L ? __bfloat162float(rq[r * D + c]) : 0.f;
                    kk[r] = r < L ? __bfloat162float(rk[r * D + c]) : 0.f;
                }
                uint32_t wq[C / 2], wk[C / 2];
                float gam = 1.f;
#pragma unroll
                for (int r = 0; r < C; r += 2) {
                    const float g0 = gam * eg[r];  // Gamma_r = exp(G_r)
                    const float g1 = g0 * eg[r + 1];
                    gam = g1;
                    wq[r >> 1] = pack_bf16(qq[r] * g0, qq[r + 1] * g1);
                    wk[r >> 1] = pack_bf16(kk[r] * g0, kk[r + 1] * g1);
                }
                *reinterpret_cast<uint4 *>(slot + OFF_PQ + cmaj(c, 0)) = make_uint4(wq[0], wq[1], wq[2], wq[3]);
                *reinterpret_cast<uint4 *>(slot + OFF_PQ + cmaj(c, 8)) = make_uint4(wq[4], wq[5], wq[6], wq[7]);
                *reinterpret_cast<uint4 *>(KtB + cmaj(c, 0)) = make_uint4(wk[0], wk[1], wk[2], wk[3]);
                *reinterpret_cast<uint4 *>(KtB + cmaj(c, 8)) = make_uint4(wk[4], wk[5], wk[6], wk[7]);
                Pg[gperm(c)] = gam;                    // gamma_L = exp(G_L)
                const float inv_gl = rcp_approx(gam);  // exp(-G_L) <= exp(80)
                float suf = 1.f;                       // exp(G_L - G_r)
                uint32_t wp[C / 2], wh[C / 2];
                float hp = 0.f, hk = 0.f;
#pragma unroll
                for (int r = C - 1; r >= 0; --r) {
                    const float kp = kk[r] * suf, kh = kk[r] * (suf * inv_gl);
                    if (r & 1) {
                        hp = kp;
                        hk = kh;
                    } else {
                        wp[r >> 1] = pack_bf16(kp, hp);
                        wh[r >> 1] = pack_bf16(kh, hk);
                    }
                    suf *= eg[r];
                }
                *reinterpret_cast<uint4 *>(slot + OFF_PK + cmaj(c, 0)) = make_uint4(wp[0], wp[1], wp[2], wp[3]);
                *reinterpret_cast<uint4 *>(slot + OFF_PK + cmaj(c, 8)) = make_uint4(wp[4], wp[5], wp[6], wp[7]);
                *reinterpret_cast<uint4 *>(KhB + cmaj(c, 0)) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                *reinterpret_cast<uint4 *>(KhB + cmaj(c, 8)) = make_uint4(wh[4], wh[5], wh[6], wh[7]);
            }
            named_sync(bar_id, nt);
            if (c == kLead) KDA_TRACE(n, 5);
            // the raw slot is free again: request this group's next chunk now
            fetch(n + NP, (k + 1) & 1);
            // -- A = strict_lower(beta K~ K^^T) and P = lower(Q~ K^^T) on the group's warps 2
            //    and 3 (the warps that share no scheduler with the state warps); each warp
            //    one 8-token column tile (j in [8 jh, 8 jh + 8)) of both
            if (pw >= 2) {
                const int jh = pw & 1;
                uint32_t b[D / 32][4];
#pragma unroll
                for (int kp = 0; kp < D / 32; ++kp)  // K^^T fragments of key tiles 2kp, 2kp+1
                    ldsm_x4_t(Kh_s + cmaj(kp * 32 + i8 * 8 + r8, jh * 8), b[kp][0], b[kp][1],
                              b[kp][2], b[kp][3]);
#pragma unroll 1
                for (int prod = 0; prod < 2; ++prod) {
                const bool isA = prod == 0;
                const uint32_t lhs = isA ? Kt_s : slot_s + OFF_PQ;
                uint32_t a[D / 16][4];
#pragma unroll
                for (int kt = 0; kt < D / 16; ++kt)
                    ldsm_x4_t(lhs + cmaj(kt * 16 + (i8 >> 1) * 8 + r8, (i8 & 1) * 8), a[kt][0],
                              a[kt][1], a[kt][2], a[kt][3]);
                float acc[2][4] = {};
#pragma unroll
                for (int kt = 0; kt < D / 16; ++kt)
                    mma16816(acc[kt & 1], a[kt], b[kt >> 1][2 * (kt & 1)], b[kt >> 1][2 * (kt & 1) + 1]);
                __nv_bfloat16 *Pp = reinterpret_cast<__nv_bfloat16 *>(slot + OFF_PP);
                const int r0 = lane >> 2, j0 = jh * 8 + 2 * (lane & 3);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int r = r0 + 8 * hh;
                    const float v0 = acc[0][2 * hh] + acc[1][2 * hh];
                    const float v1 = acc[0][2 * hh + 1] + acc[1][2 * hh + 1];
                    if (isA) {
                        As[r * C + j0] = j0 < r ? bs[r] * v0 : 0.f;
                        As[r * C + j0 + 1] = j0 + 1 < r ? bs[r] * v1 : 0.f;
                    } else {
                        *reinterpret_cast<uint32_t *>(Pp + r * LDS + j0) =
                            pack_bf16(j0 <= r ? v0 : 0.f, j0 + 1 <= r ? v1 : 0.f);
                    }
                }
                }
            }
            named_sync(bar_id, nt);
            if (c == kLead) KDA_TRACE(n, 6);
            // -- TB = (I + A)^-1 diag(beta): forward substitution, one column per lane
            if (pw == 2 && lane < C) {
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
            named_sync(bar_id, nt);
            if (c == kLead) KDA_TRACE(n, 7);
            // -- -W = -TB K~: warps 2 and 3, warp pw covering key channels
            //    [64 (pw - 2), 64 (pw - 2) + 64)
            if (pw >= 2) {
                __nv_bfloat16 *Pw = reinterpret_cast<__nv_bfloat16 *>(slot + OFF_PW);
                uint32_t tb[4];
                {
                    const int r = (i8 & 1) * 8 + r8, j = (i8 >> 1) * 8;
                    ldsm_x4(slot_s + OFF_PTB + (r * LDS + j) * 2, tb[0], tb[1], tb[2], tb[3]);
                }
#pragma unroll
                for (int half = 0; half < 4; ++half) {
                    const int cb = (pw - 2) * 64 + half * 16;
                    uint32_t k0, k1, k2, k3;
                    ldsm_x4(Kt_s + cmaj(cb + (i8 >> 1) * 8 + r8, (i8 & 1) * 8), k0, k1, k2, k3);
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
            named_sync(bar_id, nt);
            if (c == kLead) KDA_TRACE(n, 8);
            if (c == kLead) {
                // into slot s of every CTA (this one last), each once it has consumed the
                // slot's previous chunk; completion lands on that CTA's FULL barrier
                const uint32_t dst = sbase + SM_PROD + s * SLOT_BYTES;
                for (uint32_t q = 1; q <= (uint32_t)kCS; ++q) {
                    const uint32_t peer = (rank + q) % kCS;
                    if (k > 0 && !mbar_wait<true>(bar(B_PFREE(g, (int)peer)), (k & 1) ^ 1)) break;
                    bulk_copy_to_peer(map_to_rank(dst, peer), slot_s, SLOT_BYTES,
                                      map_to_rank(bar(B_FULL(s)), peer));
                }
                KDA_TRACE(n, 9);
            }
        }
        if (pw == 3) asm volatile("cp.async.wait_group 0;" ::: "memory");
    } else {
        regs_increase<kRegsConsumer>();
        if (warp < W_OUT0) {
        // ------------------------------------------------ state warps
        // State warp sw owns value columns [vrow0, vrow0 + 16) of the state, i.e. 16
        // rows of S^T over all 128 key channels, in registers for the whole sequence.
        // Per chunk: U^T = V^T TB^T - S^T W^T, then S^T <- S^T diag(gamma_L) + U^T K'.
        // The bf16 S^T (before the update) and U^T fragments go to the paired output
        // warp, which forms the output; nothing on this serial chain waits for it.
        const int sw = warp - W_STATE0;
        const int vrow0 = (int)rank * VB + sw * 16;  // first value column (row of S^T)
        const int g4 = lane >> 2, l4 = lane & 3;
        const int i8 = lane >> 3, r8 = lane & 7;
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
        // handoff buffer b of this state warp, this lane's row (9 x 16 bytes)
        auto handoff = [&](int b) {
            return reinterpret_cast<uint4 *>(sm + SM_HO + (sw * 2 + b) * HO_BYTES + lane * HO_LANE);
        };
        // U^T operands of the chunk in slot s: V^T and TB^T fragments, and key tile kt of
        // the (-W)^T fragments
        auto load_vt = [&](int s, uint32_t (&va)[4], uint32_t (&tb)[4]) {
            const uint32_t slot_s = sbase + SM_PROD + s * SLOT_BYTES;
            const uint32_t vs = sbase + SM_V + s * V_BYTES;
            // the v tile arrives 64-byte swizzled (16-byte granule g of each 64-byte token
            // row sits at g ^ address bits 7-8), so the 8 rows an 8 x 8 transposed read
            // touches fall in 8 different bank groups
            const int t = (i8 >> 1) * 8 + r8, g = sw * 2 + (i8 & 1);
            const uint32_t row = vs + (uint32_t)(t * VB * 2);
            ldsm_x4_t(row + 16u * ((uint32_t)g ^ ((row >> 7) & 3u)), va[0], va[1], va[2], va[3]);
            const int r = (i8 >> 1) * 8 + r8, j = (i8 & 1) * 8;
            ldsm_x4(slot_s + OFF_PTB + (r * LDS + j) * 2, tb[0], tb[1], tb[2], tb[3]);
        };
        auto load_w = [&](int s, int kt, uint32_t (&w)[4]) {
            const uint32_t slot_s = sbase + SM_PROD + s * SLOT_BYTES;
            const int r = (i8 >> 1) * 8 + r8;
            ldsm_x4(slot_s + OFF_PW + (r * LDP + kt * 16 + (i8 & 1) * 8) * 2, w[0], w[1], w[2], w[3]);
        };
        auto load_u_ops = [&](int s, uint32_t (&va)[4], uint32_t (&tb)[4], uint32_t (&wf)[8][4]) {
            load_vt(s, va, tb);
#pragma unroll
            for (int kt = 0; kt < 8; ++kt) load_w(s, kt, wf[kt]);
        };
        // one 16-key step of U^T = V^T TB^T + S^T (-W)^T: S^T key tile kt as bf16 A fragment,
        // also handed to the output warp
        auto u_step = [&](int kt, const uint32_t (&wf)[8][4], float (&accU)[2][2][4], uint4 *ho) {
            uint32_t a[4];
            a[0] = pack_bf16(S[2 * kt][0], S[2 * kt][1]);
            a[1] = pack_bf16(S[2 * kt][2], S[2 * kt][3]);
            a[2] = pack_bf16(S[2 * kt + 1][0], S[2 * kt + 1][1]);
            a[3] = pack_bf16(S[2 * kt + 1][2], S[2 * kt + 1][3]);
            mma16816(accU[kt & 1][0], a, wf[kt][0], wf[kt][1]);
            mma16816(accU[kt & 1][1], a, wf[kt][2], wf[kt][3]);
            ho[kt] = make_uint4(a[0], a[1], a[2], a[3]);
        };
        auto u_finish = [&](const float (&accU)[2][2][4], uint32_t (&Ua)[4]) {
            Ua[0] = pack_bf16(accU[0][0][0] + accU[1][0][0], accU[0][0][1] + accU[1][0][1]);
            Ua[1] = pack_bf16(accU[0][0][2] + accU[1][0][2], accU[0][0][3] + accU[1][0][3]);
            Ua[2] = pack_bf16(accU[0][1][0] + accU[1][1][0], accU[0][1][1] + accU[1][1][1]);
            Ua[3] = pack_bf16(accU[0][1][2] + accU[1][1][2], accU[0][1][3] + accU[1][1][3]);
        };
        // one 16-key step of S^T <- S^T diag(gamma_L) + U^T K'
        auto s_step = [&](int np, const float4 &g, const uint32_t (&kf)[4], const uint32_t (&Ua)[4]) {
            mul2(S[2 * np][0], S[2 * np][1], g.x, g.y);
            mul2(S[2 * np][2], S[2 * np][3], g.x, g.y);
            mul2(S[2 * np + 1][0], S[2 * np + 1][1], g.z, g.w);
            mul2(S[2 * np + 1][2], S[2 * np + 1][3], g.z, g.w);
            mma16816(S[2 * np], Ua, kf[0], kf[1]);
            mma16816(S[2 * np + 1], Ua, kf[2], kf[3]);
        };
        // state-update operands of the chunk in slot s, key tile np: K' fragments and
        // gamma_L
        auto load_s = [&](int s, int np, uint32_t (&k)[4], float4 &g) {
            const uint32_t slot_s = sbase + SM_PROD + s * SLOT_BYTES;
            const float4 *Pg = reinterpret_cast<const float4 *>(sm + SM_PROD + s * SLOT_BYTES + OFF_PG);
            ldsm_x4(slot_s + OFF_PK + cmaj(np * 16 + (i8 >> 1) * 8 + r8, (i8 & 1) * 8), k[0], k[1], k[2],
                    k[3]);
            g = Pg[np * 4 + l4];
        };
        // chunk m's products are in, and its handoff buffer is free
        auto wait_chunk = [&](int m) {
            bool ok = mbar_wait<false>(bar(B_FULL(m % NP)), (m / NP) & 1);
            ok = ok && mbar_wait<false>(bar(B_HEMPTY(sw, m & 1)), ((m >> 1) & 1) ^ 1);
            return !__any_sync(0xffffffffu, !ok);
        };
        // Software pipeline. Iteration n applies chunk n's state update and, interleaved
        // with it key tile by key tile, forms U^T of chunk n + 1 from the freshly updated
        // tiles, so the two serial halves of consecutive chunks overlap. Each operand tile
        // of the next iteration is loaded into the registers of the tile just consumed
        // (K' and gamma_L of chunk n + 1, (-W)^T of chunk n + 2), so loads stream through
        // the iteration; the barriers of chunk n + 2 are probed without blocking at the
        // start of iteration n. U^T of chunk 0 is formed before the loop.
        uint32_t Ua[4] = {0u, 0u, 0u, 0u};
        uint32_t va[4], tb[4], wf[8][4], kf[8][4];
        float4 gl[8];
        int n_end = 0;  // iterations that may run (all operands of iteration n are loaded)
        if (nchunks > 0 && wait_chunk(0)) {
            load_u_ops(0, va, tb, wf);
            float accU[2][2][4] = {};
            mma16816(accU[1][0], va, tb[0], tb[1]);
            mma16816(accU[1][1], va, tb[2], tb[3]);
            uint4 *ho = handoff(0);
#pragma unroll
            for (int kt = 0; kt < 8; ++kt) u_step(kt, wf, accU, ho);
            u_finish(accU, Ua);
            ho[8] = make_uint4(Ua[0], Ua[1], Ua[2], Ua[3]);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_HFULL(sw, 0)));
            n_end = 1;
            if (nchunks > 1) {
                if (wait_chunk(1)) {
                    load_u_ops(1, va, tb, wf);
                } else {
                    n_end = 0;
                }
            }
#pragma unroll
            for (int np = 0; np < 8; ++np) load_s(0, np, kf[np], gl[np]);
        }
        for (int n = 0; n < n_end; ++n) {
            const int s = n % NP;
            const bool has_next = n + 1 < nchunks, has_next2 = n + 2 < nchunks;
            if (sw == 0 && lane == 0) KDA_TRACE(n, 10);
            bool ready2 = true;
            if (has_next2) {
                const int m = n + 2;
                ready2 = mbar_test(bar(B_FULL(m % NP)), (m / NP) & 1) &&
                         mbar_test(bar(B_HEMPTY(sw, m & 1)), ((m >> 1) & 1) ^ 1);
            }
            if (has_next) {
                const int s1 = (n + 1) % NP, s2 = (n + 2) % NP;
                // whether chunk n + 2's operands may stream in during this iteration is
                // decided at key tile 2, when the probe's result has long arrived
                bool roll = false;
                float accU[2][2][4] = {};
                mma16816(accU[1][0], va, tb[0], tb[1]);
                mma16816(accU[1][1], va, tb[2], tb[3]);
                uint4 *ho = handoff((n + 1) & 1);
                s_step(0, gl[0], kf[0], Ua);
#pragma unroll
                for (int np = 1; np < 8; ++np) {
                    s_step(np, gl[np], kf[np], Ua);
                    load_s(s1, np - 1, kf[np - 1], gl[np - 1]);
                    u_step(np - 1, wf, accU, ho);
                    if (np == 2) {
                        roll = has_next2 && __all_sync(0xffffffffu, ready2);
                        if (roll) {
                            load_vt(s2, va, tb);
                            load_w(s2, 0, wf[0]);
                        }
                    }
                    if (roll && np >= 2) load_w(s2, np - 1, wf[np - 1]);
                }
                // every read of slot n by this warp has completed (its values were consumed)
                __syncwarp();
                if (lane == 0) mbar_arrive_relaxed(bar(B_FREE(s)));
                load_s(s1, 7, kf[7], gl[7]);
                u_step(7, wf, accU, ho);
                if (roll) load_w(s2, 7, wf[7]);
                if (sw == 0 && lane == 0) KDA_TRACE(n, 11);
                u_finish(accU, Ua);
                ho[8] = make_uint4(Ua[0], Ua[1], Ua[2], Ua[3]);
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_HFULL(sw, (n + 1) & 1)));
                if (sw == 0 && lane == 0) KDA_TRACE(n, 12);
                n_end = n + 2;
                if (has_next2 && !roll) {  // chunk n + 2 was not in yet: wait, then load
                    if (!wait_chunk(n + 2)) break;
                    load_u_ops(s2, va, tb, wf);
                }
            } else {
#pragma unroll
                for (int np = 0; np < 8; ++np) s_step(np, gl[np], kf[np], Ua);
                __syncwarp();
                if (lane == 0) mbar_arrive_relaxed(bar(B_FREE(s)));
            }
            if (sw == 0 && lane == 0) KDA_TRACE(n, 13);
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
    } else {
        // ------------------------------------------------ output warps
        // O^T = S^T Q~^T + U^T P^T for the paired state warp's 16 value columns, scaled
        // by d_k^-1/2; the 16 x 16 tile is transposed in registers (movmatrix) and
        // written with 4-byte global stores, rows past the sequence end skipped.
        const int ow = warp - W_OUT0;  // pairs with state warp ow
        const int vrow0 = (int)rank * VB + ow * 16;
        const int g4 = lane >> 2, l4 = lane & 3;
        const int i8 = lane >> 3, r8 = lane & 7;
        const float scale = rsqrtf((float)D);
        for (int n = 0; n < nchunks; ++n) {
            const int s = n % NP, use = n / NP;
            const int hb = n & 1;
            bool ok = mbar_wait<false>(bar(B_FULL(s)), use & 1);
            if (__any_sync(0xffffffffu, !ok)) break;
            const uint32_t slot_s = sbase + SM_PROD + s * SLOT_BYTES;
            uint32_t qf[8][4], pf[4];
#pragma unroll
            for (int kt = 0; kt < 8; ++kt)
                ldsm_x4_t(slot_s + OFF_PQ + cmaj(kt * 16 + (i8 & 1) * 8 + r8, (i8 >> 1) * 8),
                          qf[kt][0], qf[kt][1], qf[kt][2], qf[kt][3]);
            {
                const int r = (i8 >> 1) * 8 + r8, j = (i8 & 1) * 8;
                ldsm_x4(slot_s + OFF_PP + (r * LDS + j) * 2, pf[0], pf[1], pf[2], pf[3]);
            }
            ok = mbar_wait<false>(bar(B_HFULL(ow, hb)), (n >> 1) & 1);
            if (__any_sync(0xffffffffu, !ok)) break;
            uint32_t Sa[8][4], Ua[4];
            {
                const uint4 *ho = reinterpret_cast<const uint4 *>(sm + SM_HO + (ow * 2 + hb) * HO_BYTES +
                                                                  lane * HO_LANE);
#pragma unroll
                for (int kt = 0; kt < 8; ++kt) {
                    const uint4 v = ho[kt];
                    Sa[kt][0] = v.x; Sa[kt][1] = v.y; Sa[kt][2] = v.z; Sa[kt][3] = v.w;
                }
                const uint4 v = ho[8];
                Ua[0] = v.x; Ua[1] = v.y; Ua[2] = v.z; Ua[3] = v.w;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_HEMPTY(ow, hb)));
            float accO[2][2][4] = {};
#pragma unroll
            for (int kt = 0; kt < 8; ++kt) {
                mma16816(accO[kt & 1][0], Sa[kt], qf[kt][0], qf[kt][1]);
                mma16816(accO[kt & 1][1], Sa[kt], qf[kt][2], qf[kt][3]);
            }
            mma16816(accO[0][0], Ua, pf[0], pf[1]);
            mma16816(accO[0][1], Ua, pf[2], pf[3]);
            __syncwarp();
            if (lane == 0) mbar_arrive_relaxed(bar(B_FREE(s)));
            // 8x8 blocks (value rows x tokens) transposed to (tokens x value columns)
            const int c0 = t0 + n * C;
            const int L = min(C, t1 - c0);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hv = 0; hv < 2; ++hv) {
                    const uint32_t blk = movm_t(pack_bf16(
                        scale * (accO[0][nt][2 * hv] + accO[1][nt][2 * hv]),
                        scale * (accO[0][nt][2 * hv + 1] + accO[1][nt][2 * hv + 1])));
                    const int t = nt * 8 + g4;
                    if (t < L)
                        *reinterpret_cast<uint32_t *>(p.out + ((size_t)(c0 + t) * H + head) * D +
                                                      vrow0 + hv * 8 + 2 * l4) = blk;
                }
            if (ow == 0 && lane == 0) KDA_TRACE(n, 14);
        }
        }
    }
    // no CTA may leave while a peer can still write into its shared memory
    __syncwarp();
    cluster_sync();
#ifdef KDA_TC_TRACE
    __syncthreads();
    if (blockIdx.x < 4)
        for (int i = threadIdx.x; i < 32 * 16; i += blockDim.x)
            g_trace[blockIdx.x][i / 16][i % 16] = reinterpret_cast<long long *>(sm + SM_TRACE)[i];
#endif
}

// A wait on an mbarrier that nothing ever completes: exercises the bounded-wait path
// (flag set, wait returns) without any fault. One thread; `limit` in SM cycles.
__global__ void bounded_wait_selftest_kernel(long long limit, int *returned) {
    __shared__ __align__(8) unsigned long long mbar;
    const uint32_t a = smem_u32(&mbar);
    mbar_init(a, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const bool completed = mbar_wait<false>(a, 0, limit);
    *returned = completed ? 2 : 1;  // 1: gave up as designed
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

bool encode_map(CUtensorMap *m, const void *base, bool f32, int64_t n_tok, int H, int box_x,
                CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE, int box_t = C) {
    // [n_tok][H][128] row-major viewed as a 3-D tensor (channel, head, token); boxes
    // are box_x channels x 1 head x 16 tokens. Out-of-range tokens read as zero.
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t es = f32 ? 4 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)n_tok};
    cuuint64_t strides[2] = {D * es, (cuuint64_t)H * D * es};
    cuuint32_t box[3] = {(cuuint32_t)box_x, 1, (cuuint32_t)box_t};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                     const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

cudaError_t launch_tc_impl(const FwdArgs &a, cudaStream_t stream) {
    CUtensorMap mq, mk, ma, mv;
    if (!encode_map(&mq, a.q, false, a.n_tok, a.n_heads, D) ||
        !encode_map(&mk, a.k, false, a.n_tok, a.n_heads, D) ||
        !encode_map(&ma, a.a, true, a.n_tok, a.n_heads, D) ||
        !encode_map(&mv, a.v, false, a.n_tok, a.n_heads, VB, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kda_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    // The warpgroups' register increase is only covered when the block is launched with
    // exactly kRegsLaunch registers per thread; with fewer it could never be granted.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kda_tc_kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kRegsLaunch) return cudaErrorInvalidConfiguration;
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
    attr[0].val.clusterDim.x = kCS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kda_tc_kernel, mq, mk, ma, mv, p);
    if (e == cudaSuccess) count_launches(1);
    return e;
}

}  // namespace

bool tc_supported(const FwdArgs &a) {
    return a.bf16 && a.d_k == D && a.d_v == D && a.n_tok > 0 &&
           (int64_t)a.n_seq * a.n_heads * kCS < 0x7fffffffLL && a.n_tok < 0x7fffffffLL;
}

cudaError_t launch_tc(const FwdArgs &a, cudaStream_t stream) {
    return launch_tc_impl(a, stream);
}

#ifdef KDA_TC_TRACE
extern "C" int kda_debug_trace_dump(long long *host) {
    return (int)cudaMemcpyFromSymbol(host, g_trace, sizeof(g_trace));
}
#endif

cudaError_t bounded_wait_selftest(long long limit_cycles, int *d_returned, cudaStream_t stream) {
    bounded_wait_selftest_kernel<<<1, 1, 0, stream>>>(limit_cycles, d_returned);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
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
