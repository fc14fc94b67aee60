// kda_fwd64.cu -- the chunked KDA forward pass with 64-token serial steps on tcgen05
// tensor cores, bf16 I/O, d_k = d_v = 128, fp32 state and accumulation, for sm_103a.
//
// The method's bounded tile is 16 tokens: with g = -5 sigmoid(a) a tile spans at most
// 16 x (-5) = -80 in log-decay, so exp(+-G) inside a tile stays within exp(+-80) and the
// diagonal tile is a dense tensor-core product ("From Numerical Stability to Load
// Balancing", §2.1-2.3; "Architecting Long-Context LLMs", §2.2-2.3). This kernel keeps
// that tile and advances the serial state recurrence 64 tokens (four tiles) per step.
// Between tiles I > J of a step the pairwise factor exp(G_r - G_j) is the product of
// tile I's own Q~ / K~ scaling (<= 1), the decays of the tiles in between (<= 1) and tile
// J's K' scaling (<= 1), so no exponent outside the 16-token bound is ever formed. Per
// step of B = 64 tokens of one (sequence, head), with G^B the log-decay restarted at the
// step:
//   A  = strict_lower(diag(beta) [K K^T with the factors above])     64 x 64
//   P  = lower([Q K^T with the same factors])                        64 x 64
//   TB = (I + A)^-1 diag(beta),   W = TB K~B,   K~B = K exp(G^B)
//   Q' = Q~B - P W,               P' = P TB,    K'B = K exp(G^B_end - G^B)
//   U  = TB V - W S,   O = d_k^-1/2 (P' V + Q' S),   S <- Diag(exp G^B_end) S + K'B^T U
// (the output line is d_k^-1/2 (Q~B S + P U) with U substituted).
//
// Work decomposition: one cluster of 1 + kPro CTAs per (sequence, head).
//  * rank 0, the chain CTA, runs the serial recurrence. Transposed, with the state S^T
//    (d_v x d_k) as the A operand of the tensor core: per step one group of MMAs
//        D1 (128 x 128, tensor memory) = V^T [TB | P']^T + S^T [-W | Q']^T
//    gives U^T (columns 0..63) and O^T / scale (64..127) at once; a second group
//        D2 = U^T K'B
//    gives the state increment. S^T lives in fp32 registers of eight "state" warps (two
//    warpgroups; one value row and 64 keys per thread) and is mirrored as bf16 into
//    tensor memory as the next A operand; U^T likewise. Four "output" warps store O.
//    One thread issues every tcgen05.mma. A producer warp loads each step's V tile by
//    TMA into one of two buffers; the products arrive in one of three operand slots.
//  * ranks 1..kPro, the prologue CTAs, each compute every kPro-th step's products (the
//    gate, the four tiles' scaled operands, A, P, the 64 x 64 solve, TB, P', and
//    [W; -Q'] as one tcgen05 product on their own tensor core) into a staging buffer
//    laid out exactly as the chain CTA's operand slot, and copy it there with bulk
//    copies (shared::cta -> shared::cluster) once the chain CTA has freed the slot
//    (with three slots and three prologue CTAs, each prologue CTA always fills the
//    same slot).
// Every wait is bounded: one that exceeds its limit sets bit 3 of the status word
// (kda_read_device_flags); every other wait of the grid then gives up and the kernel
// finishes with unspecified output.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_internal.h"
#include "kda_ptx.h"

namespace kda {

__device__ unsigned int g_fwd64_flags;  // bit 3: a pipeline wait exceeded its limit

// Phase timestamps (SM clock) of the first cluster's first 64 steps: a profiling aid
// compiled only with -DKDA_FWD64_TRACE. Slots 0-6 (chain CTA, per step): loop top, state
// products issued, D1 complete, U stored, state-update products issued, D2 complete,
// state stored; slots 8-15 (the prologue CTA owning the step): loop top, raw tiles in,
// gate, cross-tile decays, A and P, solve, W and Q', P' (copy issued at slot 7).
#ifdef KDA_FWD64_TRACE
__device__ long long g_f64_trace[64][24];
#define F64_TRACE(n, slot)                                      \
    do {                                                        \
        if (blockIdx.x < kCluster && (n) < 64) g_f64_trace[(n)][(slot)] = clock64(); \
    } while (0)
#else
#define F64_TRACE(n, slot) \
    do {                   \
    } while (0)
#endif

namespace {

using namespace ptx;

constexpr int D = 128;           // d_k = d_v
constexpr int BT = 64;           // tokens per serial step
constexpr int TL = kChunk;       // bounded tile (16 tokens)
constexpr int NT = BT / TL;      // tiles per step (4)
constexpr int kPro = 3;          // prologue CTAs per cluster
constexpr int kCluster = 1 + kPro;
constexpr int kThreads = 512;
constexpr long long kWaitLimit = 4000000000LL;  // cycles (~2 s)
constexpr float kScale = 0.08838834764831845f;  // 128^-1/2
static_assert(NT == 4, "the tile-pair tables below assume four tiles per step");

// ---- operand slot (identical layout in the chain CTA's ring and a prologue's staging)
// B1: [n][j] K-major, 128-byte swizzle: rows 0..63 = TB, rows 64..127 = P'   (K = tokens)
// B2: [n][c] K-major, two 64-channel atom columns: rows 0..63 = -W, 64..127 = Q'
// B3: [c][t] K-major: K'B^T (K = tokens)
// G : gamma^B[c] = exp(G^B_end), fp32
constexpr int SL_B1 = 0, SL_B2 = 16384, SL_B3 = 49152, SL_G = 65536;
constexpr int SLOT_BYTES = SL_G + D * 4;  // 66048 (the gamma^B vector lives in its own ring)
constexpr int SLOT_STRIDE = SL_G;         // 64 KB per slot: every slot 1024-byte aligned
constexpr int NSLOT = 3;                  // operand slots of the chain CTA
constexpr int V_BYTES = BT * D * 2;       // V tile: two [64 t][64 v] swizzled halves
static_assert(SLOT_BYTES % 16 == 0 && SLOT_STRIDE % 1024 == 0, "slot alignment");

// ---- chain CTA shared memory
constexpr int CH_SLOT = 0;                     // NSLOT slots (B1, B2, B3)
constexpr int CH_V = NSLOT * SLOT_STRIDE;      // 2 V tiles
constexpr int CH_G = CH_V + 2 * V_BYTES;       // NSLOT gamma^B vectors
constexpr int CH_BAR = CH_G + NSLOT * D * 4;
static_assert(CH_V % 1024 == 0, "swizzled tiles need 1024-byte alignment");
// barrier indices (8 bytes each)
constexpr int B_FULL = 0;     // [NSLOT] slot s: products (bulk copies) + V (TMA) landed
constexpr int B_FREE = 3;     // [NSLOT] slot s: its MMAs completed and gamma read (2 arrivals)
constexpr int B_D1FULL = 6;   // [2] D1 buffer b complete
constexpr int B_D1FREE = 8;   // [2] D1 buffer b read out by the output warps (4 arrivals)
constexpr int B_D2FULL = 10;  // D2 complete
constexpr int B_DRAIN = 11;   // every MMA complete (before the tensor memory is released)
constexpr int NBARS = 12;
static_assert(NSLOT == 3 && B_FREE == NSLOT, "barrier table");
// tensor-memory columns
constexpr uint32_t TM_D1 = 0;     // 2 x 128 columns
constexpr uint32_t TM_D2 = 256;   // 128 columns
constexpr uint32_t TM_AS = 384;   // S^T bf16: 64 columns (128 keys)
constexpr uint32_t TM_AU = 448;   // U^T bf16: 32 columns (64 tokens)
constexpr uint32_t kTmemCols = 512;

// ---- prologue CTA shared memory
constexpr int PR_Q = 0, PR_K = 16384, PR_A = 32768;  // raw tiles [64 t][128 c] (TMA)
constexpr int PR_TILES = 65536;                      // 19 channel-major 128 x 16 tiles
constexpr int TILE_BYTES = D * TL * 2;               // 4096
constexpr int T_KT = 0, T_QT = 4, T_KH = 8, T_KP = 12, T_KX = 16;
constexpr int PR_AT = PR_TILES + 19 * TILE_BYTES;    // A, then T, fp32 [64][64]
constexpr int PR_STG = PR_AT + BT * BT * 4;          // staging slot
constexpr int PR_GAM = PR_STG + SLOT_BYTES;          // gamma_I[c] fp32 [4][128]
constexpr int PR_PRE = PR_GAM + NT * D * 4;          // prod_{m<I} gamma_m[c] [4][128]
constexpr int PR_BETA = PR_PRE + NT * D * 4;         // beta [2][64]
constexpr int PR_BAR = PR_BETA + 2 * BT * 4;         // RAWFULL, SLOTFREE, MMA done
constexpr int PR_END = PR_BAR + 24;
// after the A / P products the K^ and K' tiles are dead: K~B and Q~B ([c][64 t], 128-byte
// swizzle, the B operand of the W / Q' product) take their place; after the solve the
// fp32 A / T area holds the constant [0; -I] A-operand tile
constexpr int PR_KB = PR_TILES + T_KH * TILE_BYTES;
constexpr int PR_QB = PR_TILES + T_KP * TILE_BYTES;
static_assert(PR_KB % 1024 == 0 && PR_QB % 1024 == 0 && PR_AT % 1024 == 0, "swizzled tiles");
constexpr uint32_t kProTmemCols = 256;  // [W; -Q'] (128) and P' (64)
static_assert(PR_STG % 1024 == 0 && PR_AT % 16 == 0, "alignment");
constexpr int SMEM_USED = (PR_END > CH_BAR + NBARS * 8 ? PR_END : CH_BAR + NBARS * 8);
constexpr int SMEM_BYTES = SMEM_USED + 1024;  // + alignment slack of the dynamic base
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
// scratch inside the staging slot's B2 area until the W / Q' product overwrites it:
// 19 fp32 16 x 16 tiles (per-warp left operands, M, M^2, the diagonal T tiles)
constexpr int STG_XS = PR_STG + SL_B2;

// registers per thread (chain CTA): the block is launched with 128; each warpgroup then
// moves to its own share and the shares add up to the launch total
constexpr int kRegsLaunch = 128, kRegsMisc = 56, kRegsState = 168, kRegsOut = 120;
static_assert(kRegsMisc + 2 * kRegsState + kRegsOut == 4 * kRegsLaunch, "register split");
// setmaxnreg.inc may only raise and setmaxnreg.dec only lower a warpgroup's allotment
template <int R>
__device__ __forceinline__ void regs_set() {
    static_assert(R % 8 == 0 && R >= 24 && R <= 256, "setmaxnreg range");
    if constexpr (R > kRegsLaunch) regs_increase<R>();
    else if constexpr (R < kRegsLaunch) regs_decrease<R>();
}

struct F64Params {
    const float *beta, *h0;
    const int32_t *cu;
    __nv_bfloat16 *out;
    float *h_final;
    int n_seq, H;
};

// byte offset of element (row, k) in a K-major tile of 128-byte rows (64 bf16) with the
// 128-byte swizzle: the 16-byte chunk index is XORed with the row index mod 8
__device__ __forceinline__ uint32_t sw128(int row, int k) {
    return (uint32_t)(row * 128 + ((((k >> 3) ^ row) & 7) << 4) + (k & 7) * 2);
}
// channel-major 128 x 16 bf16 tile ([c][t], 32-byte rows); the two 16-byte halves of a
// row swap places every four rows, which keeps 8-row ldmatrix accesses conflict-free
__device__ __forceinline__ uint32_t cmaj(int c, int t0) {
    return (uint32_t)(c * 32 + ((((t0 >> 3) ^ (c >> 2)) & 1) << 4));
}

// Bounded wait. Returns false when this or any other wait of the grid gave up.
__device__ bool wait_bar(uint32_t a, uint32_t parity) {
    if (mbar_try(a, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try(a, parity)) return true;
        if ((it & 63u) == 0) {
            if (*(volatile unsigned int *)&g_fwd64_flags != 0u) return false;
            if (clock64() - t0 > kWaitLimit) {
                atomicOr(&g_fwd64_flags, 8u);
                return false;
            }
        }
    }
}

// Item of this cluster: sequences ordered longest first (ties by index), heads
// innermost, so that the longest serial chains start first.
__device__ void resolve_item(const F64Params &p, int ci, int *seq_out, int *head_out) {
    const int target = ci / p.H;
    if (threadIdx.x == 0) *seq_out = target;
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
    if (threadIdx.x == 0) *head_out = ci % p.H;
    __syncthreads();
}

// ================================================================== chain CTA
__device__ void chain_cta(unsigned char *sm, uint32_t sbase, const CUtensorMap *tm_v,
                          const F64Params &p, int seq, int head, int t0, int t1,
                          uint32_t *tmem_slot) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = p.H;
    const int nblocks = (t1 - t0 + BT - 1) / BT;
    auto bar = [&](int i) { return sbase + CH_BAR + 8u * (uint32_t)i; };

    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {
        regs_set<kRegsMisc>();
        if (warp == 0 && lane == 0) {
            // ---------------------------------------------- producer: V tiles
            // step m's V goes to buffer m & 1, last read by step m - 2's products
            for (int m = 0; m < nblocks; ++m) {
                if (m >= 2 && !wait_bar(bar(B_FREE + (m - 2) % NSLOT), ((m - 2) / NSLOT) & 1)) break;
                const int s = m % NSLOT;
                mbar_arrive_tx(bar(B_FULL + s), SLOT_BYTES + V_BYTES);
                const uint32_t dst = sbase + CH_V + (m & 1) * V_BYTES;
                tma_load_3d(dst, tm_v, 0, head, t0 + m * BT, bar(B_FULL + s));
                tma_load_3d(dst + V_BYTES / 2, tm_v, 64, head, t0 + m * BT, bar(B_FULL + s));
            }
        } else if (warp == 1 && lane == 0) {
            // ---------------------------------------------- release forwarder
            // once step n has consumed slot n % NSLOT, the owner of step n + NSLOT may copy
            // its products into it
            for (int n = 0; n + NSLOT < nblocks; ++n) {
                if (!wait_bar(bar(B_FREE + n % NSLOT), (n / NSLOT) & 1)) break;
                const uint32_t owner = 1u + (uint32_t)((n + NSLOT) % kPro);
                mbar_arrive_remote_relaxed(map_to_rank(sbase + PR_BAR + 8u, owner));
            }
        }
    } else if (warp < 12) {
        regs_set<kRegsState>();
        // -------------------------------------------------- state warps (two warpgroups)
        // Thread (value row v = TMEM lane, key half kh) holds S^T[v][64 kh .. 64 kh + 63]
        // in fp32 registers; the two warpgroups split each step's conversions by half.
        const int kh = (warp - 4) >> 2;
        const int v = ((warp & 3) << 5) + lane;                 // value row = TMEM lane
        const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;  // lane quarter
        const bool elect = warp == 4 && lane == 0;
        constexpr int KH = D / 2;
        float S[KH];
        {
            const float *h0 = p.h0 ? p.h0 + ((size_t)seq * H + head) * D * D : nullptr;
#pragma unroll
            for (int c = 0; c < KH; ++c) S[c] = h0 ? h0[(size_t)(KH * kh + c) * D + v] : 0.f;
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) w[j] = pack_bf16(S[32 * q + 2 * j], S[32 * q + 2 * j + 1]);
            tmem_st16(tmem + lb + TM_AS + 32 * kh + 16 * q, w);
        }
        tmem_st_wait();
        tc_fence_before();
        named_sync(1, 256);
        // descriptors: only the start-address field changes along K
        const uint32_t idesc_v = idesc_bf16(128, 128, 1, 0);  // A = V^T (MN-major)
        const uint32_t idesc_k = idesc_bf16(128, 128, 0, 0);
        // slot s's descriptors are slot 0's plus s x the slot stride (16-byte units)
        const uint64_t dV0 = sdesc_sw128(sbase + CH_V, 8192, 1024);
        const uint64_t dB10 = sdesc_sw128(sbase + CH_SLOT + SL_B1, 16, 1024);
        const uint64_t dB20 = sdesc_sw128(sbase + CH_SLOT + SL_B2, 16, 1024);
        const uint64_t dB30 = sdesc_sw128(sbase + CH_SLOT + SL_B3, 16, 1024);
        constexpr uint64_t kSlotStep = SLOT_STRIDE >> 4, kVStep = V_BYTES >> 4;
        // V^T [TB | P']^T into D1 buffer n & 1 (needs step n's slot and the buffer free)
        auto issue_v = [&](int n) -> bool {
            const int s = n % NSLOT, b = n & 1;
            if (!wait_bar(bar(B_FULL + s), (n / NSLOT) & 1)) return false;
            if (n >= 2 && !wait_bar(bar(B_D1FREE + b), ((n >> 1) - 1) & 1)) return false;
            tc_fence_after();
            const uint32_t d1 = tmem + TM_D1 + 128u * (uint32_t)b;
#pragma unroll
            for (int j = 0; j < 4; ++j)  // K = 16 tokens per MMA
                umma_ss(d1, dV0 + b * kVStep + (uint64_t)(128 * j), dB10 + s * kSlotStep + (uint64_t)(2 * j),
                        idesc_v, j > 0);
            return true;
        };
        bool ok = true;
        if (elect && nblocks > 0) ok = issue_v(0);
        __syncwarp();
        int n = 0;
        for (; n < nblocks; ++n) {
            const int s = n % NSLOT, b = n & 1;
            const uint32_t d1 = tmem + TM_D1 + 128u * (uint32_t)b;
            if (elect) F64_TRACE(n, 0);
            if (elect && ok) {
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k)  // S^T [-W | Q']^T, K = 16 keys per MMA
                    umma_ts(d1, tmem + TM_AS + 8u * k,
                            dB20 + s * kSlotStep + (uint64_t)((((k >> 2) * 16384) + (k & 3) * 32) >> 4), idesc_k, 1);
                umma_commit(bar(B_D1FULL + b));
                F64_TRACE(n, 1);
            }
            // ---- U^T: columns 0..63 of D1 -> bf16 A operand, 32 tokens per warpgroup
            const bool got1 = ok && wait_bar(bar(B_D1FULL + b), (n >> 1) & 1);
            if (named_sync_or(1, 256, !got1)) break;
            if (elect) F64_TRACE(n, 2);
            tc_fence_after();
            {
                uint32_t r[32], w[16];
                tmem_ld32(d1 + lb + 32u * kh, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    w[j] = pack_bf16(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
                tmem_st16(tmem + lb + TM_AU + 16 * kh, w);
            }
            tmem_st_wait();
            tc_fence_before();
            named_sync(1, 256);
            if (elect) {
                F64_TRACE(n, 3);
                tc_fence_after();
#pragma unroll
                for (int j = 0; j < 4; ++j)  // U^T K'B, K = 16 tokens per MMA
                    umma_ts(tmem + TM_D2, tmem + TM_AU + 8u * j, dB30 + s * kSlotStep + (uint64_t)(2 * j), idesc_k,
                            j > 0);
                umma_commit(bar(B_D2FULL));
                umma_commit(bar(B_FREE + s));
                if (n + 1 < nblocks) ok = issue_v(n + 1);
                F64_TRACE(n, 4);
            }
            __syncwarp();
            // ---- S^T <- S^T diag(gamma^B) + D2 on this warpgroup's 64 keys, then bf16
            const bool got2 = ok && wait_bar(bar(B_D2FULL), n & 1);
            if (named_sync_or(1, 256, !got2)) break;
            if (elect) F64_TRACE(n, 5);
            tc_fence_after();
            const float4 *gam = reinterpret_cast<const float4 *>(sm + CH_G + s * D * 4) + 16 * kh;
            {
                uint32_t r[64];
                tmem_ld32(tmem + lb + TM_D2 + 64u * kh, r);
                tmem_ld32(tmem + lb + TM_D2 + 64u * kh + 32u, r + 32);
                tmem_ld_wait();
#pragma unroll
                for (int j4 = 0; j4 < 16; ++j4) {
                    const float4 g = gam[j4];
                    const int c = 4 * j4;
                    S[c] = fmaf(g.x, S[c], __uint_as_float(r[c]));
                    S[c + 1] = fmaf(g.y, S[c + 1], __uint_as_float(r[c + 1]));
                    S[c + 2] = fmaf(g.z, S[c + 2], __uint_as_float(r[c + 2]));
                    S[c + 3] = fmaf(g.w, S[c + 3], __uint_as_float(r[c + 3]));
                }
            }
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                uint32_t w[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) w[j] = pack_bf16(S[32 * q + 2 * j], S[32 * q + 2 * j + 1]);
                tmem_st16(tmem + lb + TM_AS + 32 * kh + 16 * q, w);
            }
            tmem_st_wait();
            tc_fence_before();
            named_sync(1, 256);  // every thread has read gamma^B and stored its state half
            if (elect) {
                mbar_arrive(bar(B_FREE + s));
                F64_TRACE(n, 6);
            }
        }
        if (p.h_final) {
            float *hf = p.h_final + ((size_t)seq * H + head) * D * D;
#pragma unroll
            for (int c = 0; c < KH; ++c) hf[(size_t)(KH * kh + c) * D + v] = S[c];
        }
        if (elect) {  // every MMA has completed before the tensor memory is released
            umma_commit(bar(B_DRAIN));
            wait_bar(bar(B_DRAIN), 0);
        }
        __syncwarp();
    } else {
        regs_set<kRegsOut>();
        // -------------------------------------------------- output warps
        const int v = threadIdx.x - 384;
        const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
        const size_t tstride = (size_t)H * D;
        for (int n = 0; n < nblocks; ++n) {
            const int s = n & 1;  // D1 buffer
            const bool got = wait_bar(bar(B_D1FULL + s), (n >> 1) & 1);
            if (!__all_sync(0xffffffffu, got)) break;
            tc_fence_after();
            uint32_t r0[32], r1[32];
            const uint32_t d1 = tmem + TM_D1 + 128u * (uint32_t)s;
            tmem_ld32(d1 + lb + 64u, r0);
            tmem_ld32(d1 + lb + 96u, r1);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_D1FREE + s));
            const int L = min(BT, t1 - (t0 + n * BT));
            __nv_bfloat16 *o = p.out + ((size_t)(t0 + n * BT) * H + head) * D + v;
#pragma unroll
            for (int t = 0; t < 32; ++t)
                if (t < L) o[(size_t)t * tstride] = __float2bfloat16_rn(kScale * __uint_as_float(r0[t]));
#pragma unroll
            for (int t = 0; t < 32; ++t)
                if (t + 32 < L)
                    o[(size_t)(t + 32) * tstride] = __float2bfloat16_rn(kScale * __uint_as_float(r1[t]));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ================================================================== prologue CTA
// index of off-diagonal tile (I, J), J < I, in the off-diagonal T store: by distance
__device__ __forceinline__ int off_blk(int I, int J) {
    const int d = I - J;
    return d == 1 ? J : (d == 2 ? 3 + J : 5);
}
// the six off-diagonal tile pairs (I, J), in off_blk order
__device__ __constant__ int kOffI[6] = {1, 2, 3, 2, 3, 3};
__device__ __constant__ int kOffJ[6] = {0, 1, 2, 0, 1, 0};
// a 16 x 16 accumulator (two m16n8 fragments) into a row-major fp32 tile, scaled
__device__ __forceinline__ void store16(float *dst, const float (&acc)[2][4], float sc, int g, int t4) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        *reinterpret_cast<float2 *>(dst + g * 16 + 8 * nt + 2 * t4) = make_float2(sc * acc[nt][0], sc * acc[nt][1]);
        *reinterpret_cast<float2 *>(dst + (g + 8) * 16 + 8 * nt + 2 * t4) = make_float2(sc * acc[nt][2], sc * acc[nt][3]);
    }
}
// acc (16 x 16 as two m16n8 fragments) += L (16 x 16 fp32, row pitch lp) x R (16 x 16
// fp32, row pitch rp), the operands rounded to bf16 (one mma.sync per 8-column tile).
// Used inside the 64 x 64 solve, whose result is itself rounded to bf16: the products'
// rounding is about two orders of magnitude below that.
__device__ __forceinline__ void mma16_f32(float (&acc)[2][4], const float *L, int lp, const float *R,
                                          int rp, int g, int t4) {
    uint32_t a[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int row = g + 8 * (q & 1), col = 2 * t4 + 8 * (q >> 1);
        const float2 v = *reinterpret_cast<const float2 *>(L + row * lp + col);
        a[q] = pack_bf16(v.x, v.y);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int n = 8 * nt + g;
        const uint32_t b0 = pack_bf16(R[(2 * t4) * rp + n], R[(2 * t4 + 1) * rp + n]);
        const uint32_t b1 = pack_bf16(R[(2 * t4 + 8) * rp + n], R[(2 * t4 + 9) * rp + n]);
        mma16816(acc[nt], a, b0, b1);
    }
}

__device__ void prologue_cta(unsigned char *sm, uint32_t sbase, const CUtensorMap *tm_q,
                             const CUtensorMap *tm_k, const CUtensorMap *tm_a,
                             const F64Params &p, int head, int t0, int t1, int prank,
                             uint32_t *tmem_slot) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H;
    const int nblocks = (t1 - t0 + BT - 1) / BT;
    const uint32_t rawfull = sbase + PR_BAR, slotfree = sbase + PR_BAR + 8, mmabar = sbase + PR_BAR + 16;
    const uint32_t stg = sbase + PR_STG;
    const int i8 = lane >> 3, r8 = lane & 7, g = lane >> 2, t4 = lane & 3;
    auto tile = [&](int i) { return sbase + PR_TILES + (uint32_t)(i * TILE_BYTES); };
    float *AT = reinterpret_cast<float *>(sm + PR_AT);
    float *XS = reinterpret_cast<float *>(sm + STG_XS);  // 6 warps x 16 x 16 fp32 scratch
    float *MM = XS + 6 * 256;                             // M = L^-1 N, 6 tiles
    float *M2 = MM + 6 * 256;                             // M^2: (2,0), (3,1), (3,0)
    float *TD = M2 + 3 * 256;                             // T_II, 4 tiles
    float *GAM = reinterpret_cast<float *>(sm + PR_GAM);
    float *PRE = reinterpret_cast<float *>(sm + PR_PRE);

    // q, k and gate-logit tiles of step m (one thread), beta (warp 15, cp.async)
    auto fetch = [&](int m, int buf) {
        if (m >= nblocks) return;
        const int r0 = t0 + m * BT;
        if (warp == 15 && lane == 0) {
            mbar_arrive_tx(rawfull, 2 * BT * D * 2 + BT * D * 4);
            tma_load_3d(sbase + PR_Q, tm_q, 0, head, r0, rawfull);
            tma_load_3d(sbase + PR_K, tm_k, 0, head, r0, rawfull);
            tma_load_3d(sbase + PR_A, tm_a, 0, head, r0, rawfull);
        }
        if (warp == 15) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int i = lane + 32 * h, row = r0 + i;
                const bool in = row < t1;
                cp_async_4(sbase + PR_BETA + (uint32_t)((buf * BT + i) * 4),
                           p.beta + (size_t)(in ? row : t0) * H + head, in ? 4u : 0u);
            }
            cp_async_commit();
        }
    };
    // the staging slot into the chain CTA's slot m % NSLOT (operands) and gamma ring entry;
    // completion (SLOT_BYTES in all) is counted on that slot's FULL barrier
    auto copy_out = [&](int m) {
        const uint32_t s = (uint32_t)(m % NSLOT);
        const uint32_t full = map_to_rank(sbase + CH_BAR + 8u * (B_FULL + s), 0);
        bulk_copy_to_peer(map_to_rank(sbase + CH_SLOT + s * SLOT_STRIDE, 0), stg, SL_G, full);
        bulk_copy_to_peer(map_to_rank(sbase + CH_G + s * D * 4, 0), stg + SL_G, D * 4, full);
        bulk_commit();
    };
    fetch(prank, 0);
    // tensor memory for the W / Q' product; the tiles of TB above the diagonal stay zero
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kProTmemCols);
    for (int i = tid; i < 8192 / 16; i += kThreads)
        reinterpret_cast<uint4 *>(sm + PR_STG + SL_B1)[i] = make_uint4(0u, 0u, 0u, 0u);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t ptmem = *tmem_slot;
    bool bad = false;   // (thread 0) a wait gave up
    int nfree = 0;      // slot-free signals consumed (thread 0)
    int k = 0;
    for (int m = prank; m < nblocks; m += kPro, ++k) {
        const int L = min(BT, t1 - (t0 + m * BT));
        const float *bet = reinterpret_cast<const float *>(sm + PR_BETA) + (k & 1) * BT;
        // ---- P0: this step's raw tiles are in
        if (tid == 0) F64_TRACE(m, 8);
        if (tid == 0 && !bad) bad = !wait_bar(rawfull, k & 1);
        if (warp == 15) cp_async_wait0();
        if (__syncthreads_or(bad)) break;
        if (tid != 0) mbar_try(rawfull, k & 1);  // observe the completed phase
        if (tid == 0) F64_TRACE(m, 9);
        // ---- P1: gate pass, one (key channel, tile) per thread
        const int c = tid & (D - 1), I = tid >> 7, rb = TL * I;
        float kk[TL];
        {
            const float *ra = reinterpret_cast<const float *>(sm + PR_A);
            const __nv_bfloat16 *rq = reinterpret_cast<const __nv_bfloat16 *>(sm + PR_Q);
            const __nv_bfloat16 *rk = reinterpret_cast<const __nv_bfloat16 *>(sm + PR_K);
            float eg[TL], qq[TL];
#pragma unroll
            for (int r = 0; r < TL; ++r) eg[r] = ra[(rb + r) * D + c];
#pragma unroll
            for (int r = 0; r < TL; ++r) eg[r] = __fdividef(1.f, 1.f + __expf(-eg[r]));  // sigmoid
#pragma unroll
            for (int r = 0; r < TL; ++r) {
                const bool in = rb + r < L;
                const float e = __expf(kGMin * eg[r]);  // exp(g), g = -5 sigmoid(a)
                eg[r] = in ? e : 1.f;
                qq[r] = in ? __bfloat162float(rq[(rb + r) * D + c]) : 0.f;
                kk[r] = in ? __bfloat162float(rk[(rb + r) * D + c]) : 0.f;
            }
            uint32_t wq[TL / 2], wk[TL / 2];
            float gam = 1.f;
#pragma unroll
            for (int r = 0; r < TL; r += 2) {  // Gamma_r = exp(G_r), inclusive
                const float g0 = gam * eg[r];
                const float g1 = g0 * eg[r + 1];
                gam = g1;
                wq[r >> 1] = pack_bf16(qq[r] * g0, qq[r + 1] * g1);
                wk[r >> 1] = pack_bf16(kk[r] * g0, kk[r + 1] * g1);
            }
            unsigned char *tq = sm + PR_TILES + (T_QT + I) * TILE_BYTES;
            unsigned char *tk = sm + PR_TILES + (T_KT + I) * TILE_BYTES;
            *reinterpret_cast<uint4 *>(tq + cmaj(c, 0)) = make_uint4(wq[0], wq[1], wq[2], wq[3]);
            *reinterpret_cast<uint4 *>(tq + cmaj(c, 8)) = make_uint4(wq[4], wq[5], wq[6], wq[7]);
            *reinterpret_cast<uint4 *>(tk + cmaj(c, 0)) = make_uint4(wk[0], wk[1], wk[2], wk[3]);
            *reinterpret_cast<uint4 *>(tk + cmaj(c, 8)) = make_uint4(wk[4], wk[5], wk[6], wk[7]);
            GAM[I * D + c] = gam;                  // gamma_I = exp(G_end), >= exp(-80)
            const float inv = __frcp_rn(gam);      // exp(-G_end) <= exp(80)
            float sf = 1.f;                        // exp(G_end - G_r)
            uint32_t wp[TL / 2], wh[TL / 2];
            float hp = 0.f, hh = 0.f;
#pragma unroll
            for (int r = TL - 1; r >= 0; --r) {
                const float kp = kk[r] * sf, kh = kk[r] * (sf * inv);
                kk[r] = kp;                        // keep K' for the step-level operands
                if (r & 1) {
                    hp = kp;
                    hh = kh;
                } else {
                    wp[r >> 1] = pack_bf16(kp, hp);
                    wh[r >> 1] = pack_bf16(kh, hh);
                }
                sf *= eg[r];
            }
            unsigned char *tp = sm + PR_TILES + (T_KP + I) * TILE_BYTES;
            unsigned char *th = sm + PR_TILES + (T_KH + I) * TILE_BYTES;
            *reinterpret_cast<uint4 *>(tp + cmaj(c, 0)) = make_uint4(wp[0], wp[1], wp[2], wp[3]);
            *reinterpret_cast<uint4 *>(tp + cmaj(c, 8)) = make_uint4(wp[4], wp[5], wp[6], wp[7]);
            *reinterpret_cast<uint4 *>(th + cmaj(c, 0)) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
            *reinterpret_cast<uint4 *>(th + cmaj(c, 8)) = make_uint4(wh[4], wh[5], wh[6], wh[7]);
        }
        if (tid == 0) F64_TRACE(m, 20);
        if (tid == 511) F64_TRACE(m, 21);
        if (tid == 0) bulk_wait_read0();  // the previous step's copies have read the staging slot
        if (tid == 0) F64_TRACE(m, 22);
        __syncthreads();
        if (tid == 0) F64_TRACE(m, 10);
        // ---- P2: decays across tiles; K'B into the slot; cross-tile K' tiles
        {
            float pre = 1.f, post = 1.f;
#pragma unroll
            for (int J = 0; J < NT; ++J) {
                const float gj = GAM[J * D + c];
                if (J < I) pre *= gj;
                if (J > I) post *= gj;
            }
            PRE[I * D + c] = pre;
            uint32_t w0[4], w1[4];
#pragma unroll
            for (int r = 0; r < 8; r += 2) {
                w0[r >> 1] = pack_bf16(kk[r] * post, kk[r + 1] * post);
                w1[r >> 1] = pack_bf16(kk[r + 8] * post, kk[r + 9] * post);
            }
            unsigned char *b3 = sm + PR_STG + SL_B3;
            *reinterpret_cast<uint4 *>(b3 + sw128(c, 16 * I)) = make_uint4(w0[0], w0[1], w0[2], w0[3]);
            *reinterpret_cast<uint4 *>(b3 + sw128(c, 16 * I + 8)) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
            // K' of tile J scaled by the decay of the tiles strictly between J and I:
            // x0 = K'^0 gamma_1 (pair 2,0), x1 = K'^0 gamma_1 gamma_2 (3,0), x2 = K'^1 gamma_2 (3,1)
            auto put = [&](int x, float sc) {
                uint32_t w[8];
#pragma unroll
                for (int r = 0; r < TL; r += 2) w[r >> 1] = pack_bf16(kk[r] * sc, kk[r + 1] * sc);
                unsigned char *tx = sm + PR_TILES + (T_KX + x) * TILE_BYTES;
                *reinterpret_cast<uint4 *>(tx + cmaj(c, 0)) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4 *>(tx + cmaj(c, 8)) = make_uint4(w[4], w[5], w[6], w[7]);
            };
            if (I == 0) {
                const float g1 = GAM[D + c], g2 = GAM[2 * D + c];
                put(0, g1);
                put(1, g1 * g2);
                reinterpret_cast<float *>(sm + PR_STG + SL_G)[c] =
                    GAM[c] * g1 * g2 * GAM[3 * D + c];  // gamma^B = exp(G^B_end)
            } else if (I == 1) {
                put(2, GAM[2 * D + c]);
            }
        }
        fence_proxy_async();
        __syncthreads();
        if (tid == 0) F64_TRACE(m, 11);

        // ---- P3: A = strict_lower(beta K~ X^T) per tile pair (I, J <= I), mma.sync, on all
        //      16 warps: warp = (row tile I, 8-column half, half of the column tiles J),
        //      the row operand's fragments loaded once per warp. X is K^ on the diagonal and
        //      K' scaled by the decays of the tiles in between off it.
        auto col_tile = [&](int Ii, int Jj) -> uint32_t {
            int ct;
            if (Jj == Ii) ct = T_KH + Ii;
            else if (Ii - Jj == 1) ct = T_KP + Jj;
            else if (Ii == 2) ct = T_KX + 0;
            else ct = T_KX + (Jj == 0 ? 1 : 2);
            return tile(ct);
        };
        // rows of tile Ii times X^T for column tiles [j_lo, j_hi], 8-column half nh; the
        // epilogue gets (Jj, r, j0, v0, v1) for this lane's two adjacent columns
        auto pair_products = [&](uint32_t rowt, int Ii, int nh, int j_lo, int j_hi, auto &&epi) {
            uint32_t a[D / 16][4];
#pragma unroll
            for (int kt = 0; kt < D / 16; ++kt)
                ldsm_x4_t(rowt + cmaj(kt * 16 + (i8 >> 1) * 8 + r8, (i8 & 1) * 8), a[kt][0], a[kt][1], a[kt][2], a[kt][3]);
            for (int Jj = j_lo; Jj <= j_hi; ++Jj) {
                const uint32_t colt = col_tile(Ii, Jj);
                float acc[2][4] = {};
#pragma unroll
                for (int kp = 0; kp < D / 32; ++kp) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(colt + cmaj(kp * 32 + i8 * 8 + r8, nh * 8), b0, b1, b2, b3);
                    mma16816(acc[0], a[2 * kp], b0, b1);
                    mma16816(acc[1], a[2 * kp + 1], b2, b3);
                }
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
                    epi(Jj, g + 8 * hh, nh * 8 + 2 * t4, acc[0][2 * hh] + acc[1][2 * hh],
                        acc[0][2 * hh + 1] + acc[1][2 * hh + 1]);
            }
        };
        {
            const int Ii = warp >> 2, nh = (warp >> 1) & 1, hf = warp & 1;
            const int sp = (Ii + 2) >> 1;
            const int j_lo = hf ? sp : 0, j_hi = hf ? Ii : sp - 1;
            if (j_lo <= j_hi)
                pair_products(tile(T_KT + Ii), Ii, nh, j_lo, j_hi, [&](int Jj, int r, int j0, float v0, float v1) {
                    const bool diag = Jj == Ii;
                    const float bb = bet[TL * Ii + r];
                    *reinterpret_cast<float2 *>(AT + (TL * Ii + r) * BT + TL * Jj + j0) =
                        make_float2((!diag || j0 < r) ? bb * v0 : 0.f, (!diag || j0 + 1 < r) ? bb * v1 : 0.f);
                });
        }
        __syncthreads();
        if (tid == 0) F64_TRACE(m, 12);
        // ---- P4, two groups at once.
        //  Warps 0-5: T = (I + A)^-1, A strictly lower, in 16 x 16 tiles. L = the diagonal
        //   tiles of I + A, N = the rest, M = L^-1 N (M_IJ = T_II A_IJ, I > J; nilpotent,
        //   M^4 = 0), so T = (I + M)^-1 L^-1 = (I - M)(I + M^2) L^-1. Diagonal tiles T_II:
        //   fp32 forward substitution, one column per thread. Products of tiles: tensor
        //   cores, operands rounded to bf16. TB = T diag(beta) goes to rows 0..63 of B1 as
        //   each tile is done (the tiles above the diagonal stay 0).
        //  Warps 6-15: the next step's raw tiles requested; P = lower(Q~ X^T) into rows
        //   64..127 of B1 (zero above the diagonal tiles); then K~B = K~^I Gamma_I and
        //   Q~B = Q~^I Gamma_I ([c][64 t], 128-byte swizzle) over the K^ / K' tiles.
        if (warp < 6) {
            constexpr int kSolveThreads = 192;
            if (tid < 64) {
                const int Id = tid >> 4, j = tid & 15;
                const float *Ar = AT + (TL * Id) * BT + TL * Id;
                float x[TL];
#pragma unroll
                for (int r = 0; r < TL; ++r) {
                    // row r of A_II as four 16-byte loads, independent of the solve so far
                    float ar[TL];
#pragma unroll
                    for (int q = 0; q < (r + 3) / 4; ++q) {
                        const float4 v4 = *reinterpret_cast<const float4 *>(Ar + r * BT + 4 * q);
                        ar[4 * q] = v4.x; ar[4 * q + 1] = v4.y; ar[4 * q + 2] = v4.z; ar[4 * q + 3] = v4.w;
                    }
                    float a0 = r == j ? 1.f : 0.f, a1 = 0.f;
#pragma unroll
                    for (int i = 0; i < r; i += 2) {
                        a0 = fmaf(-ar[i], x[i], a0);
                        if (i + 1 < r) a1 = fmaf(-ar[i + 1], x[i + 1], a1);
                    }
                    x[r] = a0 + a1;
                }
                const float bj = bet[TL * Id + j];
#pragma unroll
                for (int r = 0; r < TL; ++r) {
                    TD[(Id * TL + r) * TL + j] = x[r];
                    *reinterpret_cast<__nv_bfloat16 *>(sm + PR_STG + SL_B1 + sw128(TL * Id + r, TL * Id + j)) =
                        __float2bfloat16_rn(x[r] * bj);
                }
            }
            named_sync(2, kSolveThreads);
            if (tid == 0) F64_TRACE(m, 16);
            {   // M_IJ = T_II A_IJ for the six pairs I > J (one warp each)
                const int Ir = kOffI[warp], Jc = kOffJ[warp];
                float acc[2][4] = {};
                mma16_f32(acc, TD + Ir * 256, TL, AT + (TL * Ir) * BT + TL * Jc, BT, g, t4);
                store16(MM + warp * 256, acc, 1.f, g, t4);
            }
            named_sync(2, kSolveThreads);
            if (tid == 0) F64_TRACE(m, 17);
            // M^2: (2,0) = M21 M10, (3,1) = M32 M21, (3,0) = M31 M10 + M32 M20; meanwhile warps
            // 3-5 write the constant [0; -I] operand tile over A (no longer read)
            if (warp < 3) {
                float acc[2][4] = {};
                if (warp == 0) mma16_f32(acc, MM + 1 * 256, TL, MM + 0 * 256, TL, g, t4);
                if (warp == 1) mma16_f32(acc, MM + 2 * 256, TL, MM + 1 * 256, TL, g, t4);
                if (warp == 2) {
                    mma16_f32(acc, MM + 4 * 256, TL, MM + 0 * 256, TL, g, t4);
                    mma16_f32(acc, MM + 2 * 256, TL, MM + 3 * 256, TL, g, t4);
                }
                store16(M2 + warp * 256, acc, 1.f, g, t4);
            } else {
                // 128 rows x 64 k, row n >= 64 holds -1 at k = n - 64; 32 bytes per slot
                for (int e = tid - 96; e < 512; e += 96) {
                    const int n = e >> 2, q0 = 2 * (e & 3);
#pragma unroll
                    for (int q = q0; q < q0 + 2; ++q) {
                        uint32_t w[4];
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const int k0 = 8 * q + 2 * h;
                            w[h] = pack_bf16(n - 64 == k0 ? -1.f : 0.f, n - 64 == k0 + 1 ? -1.f : 0.f);
                        }
                        *reinterpret_cast<uint4 *>(sm + PR_AT + sw128(n, 8 * q)) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            named_sync(2, kSolveThreads);
            if (tid == 0) F64_TRACE(m, 18);
            {   // T_IJ = [-(M)_IJ + (M^2)_IJ - (M^3)_IJ] T_JJ, M^3 only at (3,0) = M32 (M^2)_20;
                // TB_IJ = T_IJ diag(beta_J) straight into B1
                const int Ir = kOffI[warp], Jc = kOffJ[warp];
                float *ls = XS + warp * 256;  // this warp's left operand
                const int q2 = (Ir == 2 && Jc == 0) ? 0 : (Ir == 3 && Jc == 1) ? 1 : (Ir == 3 && Jc == 0) ? 2 : -1;
                float c3[2][4] = {};
                if (q2 == 2) mma16_f32(c3, MM + 2 * 256, TL, M2 + 0 * 256, TL, g, t4);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int row = g + 8 * h, col = 8 * nt + 2 * t4;
                        float2 v2 = *reinterpret_cast<const float2 *>(MM + warp * 256 + row * TL + col);
                        v2.x = -v2.x;
                        v2.y = -v2.y;
                        if (q2 >= 0) {
                            const float2 w2 = *reinterpret_cast<const float2 *>(M2 + q2 * 256 + row * TL + col);
                            v2.x += w2.x;
                            v2.y += w2.y;
                        }
                        v2.x -= c3[nt][2 * h];
                        v2.y -= c3[nt][2 * h + 1];
                        *reinterpret_cast<float2 *>(ls + row * TL + col) = v2;
                    }
                __syncwarp();
                float acc[2][4] = {};
                mma16_f32(acc, ls, TL, TD + Jc * 256, TL, g, t4);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int col = TL * Jc + 8 * nt + 2 * t4;
                    const float b0 = bet[col], b1 = bet[col + 1];
                    *reinterpret_cast<uint32_t *>(sm + PR_STG + SL_B1 + sw128(TL * Ir + g, col)) =
                        pack_bf16(acc[nt][0] * b0, acc[nt][1] * b1);
                    *reinterpret_cast<uint32_t *>(sm + PR_STG + SL_B1 + sw128(TL * Ir + g + 8, col)) =
                        pack_bf16(acc[nt][2] * b0, acc[nt][3] * b1);
                }
            }
        } else {
            constexpr int kAuxThreads = 320;
            if (warp == 15) fetch(m + kPro, (k + 1) & 1);  // the raw tiles have been consumed
            // P in 14 units of at most two column tiles on warps 6-15 (unit = row tile I,
            // 8-column half, part of the column tiles); warps 6-11 take one two-tile unit,
            // warps 12-15 two one-tile units
            auto p_unit = [&](int Ii, int nh, int j_lo, int j_hi) {
                pair_products(tile(T_QT + Ii), Ii, nh, j_lo, j_hi, [&](int Jj, int r, int j0, float v0, float v1) {
                    const bool diag = Jj == Ii;
                    *reinterpret_cast<uint32_t *>(sm + PR_STG + SL_B1 + sw128(BT + TL * Ii + r, TL * Jj + j0)) =
                        pack_bf16((!diag || j0 <= r) ? v0 : 0.f, (!diag || j0 + 1 <= r) ? v1 : 0.f);
                });
            };
            const int w6 = warp - 6;
            if (w6 < 6) {  // (3, nh, J 0-1), (3, nh, J 2-3), (2, nh, J 0-1)
                const int nh = w6 & 1, u = w6 >> 1;
                if (u == 0) p_unit(3, nh, 0, 1);
                else if (u == 1) p_unit(3, nh, 2, 3);
                else p_unit(2, nh, 0, 1);
            } else {       // (2, nh, J 2) + (0, nh, J 0), (1, nh, J 0) + (1, nh, J 1)
                const int nh = w6 & 1, u = (w6 - 6) >> 1;
                if (u == 0) {
                    p_unit(2, nh, 2, 2);
                    p_unit(0, nh, 0, 0);
                } else {
                    p_unit(1, nh, 0, 0);
                    p_unit(1, nh, 1, 1);
                }
            }
            // tiles above the diagonal: zero (rows of tile I = w6 >> 1 for w6 < 8, both halves)
            if (w6 < 8) {
                const int Ii = w6 >> 1, nh = w6 & 1;
                for (int Jj = Ii + 1; Jj < NT; ++Jj)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh)
                        *reinterpret_cast<uint32_t *>(sm + PR_STG + SL_B1 +
                                                      sw128(BT + TL * Ii + g + 8 * hh, TL * Jj + nh * 8 + 2 * t4)) = 0u;
            }
            named_sync(3, kAuxThreads);  // every read of the K^ / K' tiles is done
            // K~B and Q~B over the K^ and K' tiles
            for (int e = tid - 192; e < NT * D; e += kAuxThreads) {
                const int cc = e & (D - 1), Ie = e >> 7;
                const float gpre = PRE[Ie * D + cc];
#pragma unroll
                for (int which = 0; which < 2; ++which) {
                    const unsigned char *src = sm + PR_TILES + ((which ? T_QT : T_KT) + Ie) * TILE_BYTES;
                    unsigned char *dst = sm + (which ? PR_QB : PR_KB);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint4 u = *reinterpret_cast<const uint4 *>(src + cmaj(cc, 8 * h));
                        const uint32_t in[4] = {u.x, u.y, u.z, u.w};
                        uint32_t o[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const __nv_bfloat162 b2v = *reinterpret_cast<const __nv_bfloat162 *>(&in[q]);
                            o[q] = pack_bf16(__low2float(b2v) * gpre, __high2float(b2v) * gpre);
                        }
                        *reinterpret_cast<uint4 *>(dst + sw128(cc, TL * Ie + 8 * h)) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
            }
        }
        fence_proxy_async();  // B1, K~B, Q~B and [0; -I]: generic writes -> tensor-core reads
        tc_fence_before();
        __syncthreads();
        if (tid == 0) F64_TRACE(m, 13);
        // ---- P5: P' = P TB on this CTA's tensor core: A = B1 ([TB; P], K = 64 tokens),
        //      B = TB read MN-major from the same rows 0..63; rows 64..127 of the result
        //      go back into rows 64..127 of B1
        if (tid == 0) {
            tc_fence_after();
            const uint64_t da = sdesc_sw128(stg + SL_B1, 16, 1024), db = sdesc_sw128(stg + SL_B1, 8192, 1024);
            const uint32_t idp = idesc_bf16(128, 64, 0, 1);
#pragma unroll
            for (int kk2 = 0; kk2 < 4; ++kk2) umma_ss(ptmem + 128u, da + 2 * kk2, db + 128 * kk2, idp, kk2 > 0);
            umma_commit(mmabar);
        }
        if ((warp & 3) >= 2 && warp < 8) {  // lane quarters 2 and 3: rows 64..127
            const bool got = wait_bar(mmabar, 0);
            if (__all_sync(0xffffffffu, got)) {
                tc_fence_after();
                const int n = ((warp & 3) << 5) + lane, ch = warp >> 2;  // row, 32-column half
                uint32_t r[32];
                tmem_ld32(ptmem + 128u + ((uint32_t)((warp & 3) * 32) << 16) + 32u * ch, r);
                tmem_ld_wait();
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    uint32_t w[4];
#pragma unroll
                    for (int h = 0; h < 4; ++h)
                        w[h] = pack_bf16(__uint_as_float(r[8 * c8 + 2 * h]), __uint_as_float(r[8 * c8 + 2 * h + 1]));
                    *reinterpret_cast<uint4 *>(sm + PR_STG + SL_B1 + sw128(n, 32 * ch + 8 * c8)) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            tc_fence_before();
        }
        fence_proxy_async();
        __syncthreads();
        if (tid == 0) F64_TRACE(m, 14);
        // ---- P6: [W; -Q'] = [TB | 0; P' | -I] [K~B; Q~B] (M = 128, N = 128 channels, K = 128)
        //      on this CTA's tensor core; B2 = -(that), rows 0..63 -W, 64..127 Q'.
        if (tid == 0) {
            tc_fence_after();
            const uint64_t da1 = sdesc_sw128(stg + SL_B1, 16, 1024), da2 = sdesc_sw128(sbase + PR_AT, 16, 1024);
            const uint64_t db1 = sdesc_sw128(sbase + PR_KB, 16, 1024), db2 = sdesc_sw128(sbase + PR_QB, 16, 1024);
            const uint32_t idk = idesc_bf16(128, 128, 0, 0);
#pragma unroll
            for (int kk2 = 0; kk2 < 4; ++kk2) umma_ss(ptmem, da1 + 2 * kk2, db1 + 2 * kk2, idk, kk2 > 0);
#pragma unroll
            for (int kk2 = 0; kk2 < 4; ++kk2) umma_ss(ptmem, da2 + 2 * kk2, db2 + 2 * kk2, idk, 1);
            umma_commit(mmabar);
        }
        if (warp < 8) {
            const bool got = wait_bar(mmabar, 1);
            if (__all_sync(0xffffffffu, got)) {
                tc_fence_after();
                const int n = ((warp & 3) << 5) + lane, ch = warp >> 2;  // row, 64-channel half
                const uint32_t ta = ptmem + ((uint32_t)((warp & 3) * 32) << 16) + 64u * ch;
                unsigned char *dst = sm + PR_STG + SL_B2 + ch * 16384;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t r[32];
                    tmem_ld32(ta + 32u * q, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) {
                        uint32_t w[4];
#pragma unroll
                        for (int h = 0; h < 4; ++h)
                            w[h] = pack_bf16(-__uint_as_float(r[8 * c8 + 2 * h]), -__uint_as_float(r[8 * c8 + 2 * h + 1]));
                        *reinterpret_cast<uint4 *>(dst + sw128(n, 32 * q + 8 * c8)) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            tc_fence_before();
        }
        fence_proxy_async();  // generic writes of the staging slot -> the bulk copy's reads
        __syncthreads();
        if (tid == 0) F64_TRACE(m, 15);
        // ---- P8: into the chain CTA's slot m % NSLOT once step m - NSLOT has consumed it
        if (tid == 0 && !bad) {
            if (m >= NSLOT) {
                bad = !wait_bar(slotfree, nfree & 1);
                ++nfree;
            }
            if (!bad) copy_out(m);
            F64_TRACE(m, 7);
        }
    }
    if (tid == 0) {
        bulk_wait_read0();  // no copy may still read this CTA's memory at exit
        umma_commit(mmabar);  // and every product has completed before the tensor memory goes
        wait_bar(mmabar, 0);    // two commits per step: this is an even-numbered phase
    }
    if (warp == 15) cp_async_wait0();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(ptmem, kProTmemCols);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    kda_fwd64_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_v,
                     const F64Params p) {
    extern __shared__ unsigned char smraw[];
    __shared__ int item[2];
    __shared__ uint32_t tmem_slot;
    unsigned char *sm = reinterpret_cast<unsigned char *>(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(sm);
    const uint32_t rank = cluster_rank();
    resolve_item(p, (int)(blockIdx.x / kCluster), &item[0], &item[1]);
    const int seq = item[0], head = item[1];
    const int t0 = p.cu[seq], t1 = p.cu[seq + 1];
    if (threadIdx.x == 0) {
        if (rank == 0) {
            for (int s = 0; s < NSLOT; ++s) {
                mbar_init(sbase + CH_BAR + 8u * (B_FULL + s), 1);
                mbar_init(sbase + CH_BAR + 8u * (B_FREE + s), 2);
            }
            for (int b = 0; b < 2; ++b) {
                mbar_init(sbase + CH_BAR + 8u * (B_D1FULL + b), 1);
                mbar_init(sbase + CH_BAR + 8u * (B_D1FREE + b), 4);
            }
            mbar_init(sbase + CH_BAR + 8u * B_D2FULL, 1);
            mbar_init(sbase + CH_BAR + 8u * B_DRAIN, 1);
        } else {
            mbar_init(sbase + PR_BAR, 1);
            mbar_init(sbase + PR_BAR + 8, 1);
            mbar_init(sbase + PR_BAR + 16, 1);
        }
        mbar_init_fence();
    }
    cluster_sync();  // every barrier of the cluster is initialised before any remote use
    if (rank == 0)
        chain_cta(sm, sbase, &tm_v, p, seq, head, t0, t1, &tmem_slot);
    else
        prologue_cta(sm, sbase, &tm_q, &tm_k, &tm_a, p, head, t0, t1, (int)rank - 1, &tmem_slot);
    __syncwarp();
    cluster_sync();  // no CTA leaves while a peer may still write into its shared memory
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

// [n_tok][H][128] viewed as (channel, head, token); boxes of box_x channels x 1 head x
// 64 tokens; tokens past n_tok read as zero
bool encode(CUtensorMap *m, const void *base, bool f32, int64_t n_tok, int H, int box_x,
            CUtensorMapSwizzle sw) {
    auto enc = encoder();
    if (!enc) return false;
    const cuuint64_t es = f32 ? 4 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)n_tok};
    cuuint64_t strides[2] = {D * es, (cuuint64_t)H * D * es};
    cuuint32_t box[3] = {(cuuint32_t)box_x, 1, (cuuint32_t)BT};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
               const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool fwd64_supported(const FwdArgs &a) {
    return a.bf16 && a.d_k == D && a.d_v == D && a.n_tok > 0 &&
           (int64_t)a.n_seq * a.n_heads * kCluster < 0x7fffffffLL && a.n_tok < 0x7fffffffLL;
}

cudaError_t launch_fwd64(const FwdArgs &a, cudaStream_t stream) {
    CUtensorMap mq, mk, ma, mv;
    if (!encode(&mq, a.q, false, a.n_tok, a.n_heads, D, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode(&mk, a.k, false, a.n_tok, a.n_heads, D, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode(&ma, a.a, true, a.n_tok, a.n_heads, D, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode(&mv, a.v, false, a.n_tok, a.n_heads, 64, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kda_fwd64_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES);
    if (e != cudaSuccess) return e;
    // the warpgroups' register increase is covered only when the block is launched with
    // exactly kRegsLaunch registers per thread
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kda_fwd64_kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kRegsLaunch) return cudaErrorInvalidConfiguration;
    F64Params p;
    p.beta = a.beta; p.h0 = a.h0; p.cu = a.cu_seqlens;
    p.out = reinterpret_cast<__nv_bfloat16 *>(a.out); p.h_final = a.h_final;
    p.n_seq = a.n_seq; p.H = a.n_heads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((int64_t)a.n_seq * a.n_heads * kCluster));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kda_fwd64_kernel, mq, mk, ma, mv, p);
    if (e == cudaSuccess) count_launches(1);
    return e;
}

cudaError_t read_fwd64_flags(unsigned int *flags, bool reset, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(flags, g_fwd64_flags, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess || !reset) return e;
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_fwd64_flags, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}

#ifdef KDA_FWD64_TRACE
extern "C" int kda_debug_f64_trace_dump(long long *host) {
    return (int)cudaMemcpyFromSymbol(host, g_f64_trace, sizeof(g_f64_trace));
}
#endif

}  // namespace kda
