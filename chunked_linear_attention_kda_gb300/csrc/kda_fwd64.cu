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
//   TB = (I + A)^-1 diag(beta),   K~B = K exp(G^B),   K'B = K exp(G^B_end - G^B)
//   W  = TB K~B,   U = TB (V - K~B S) = TB V - W S,   O = d_k^-1/2 (Q~B S + P U),
//   S <- Diag(exp G^B_end) S + K'B^T U
//
// Work decomposition: one cluster of 1 + kPro CTAs per (sequence, head).
//  * rank 0, the chain CTA, runs the serial recurrence. Transposed, with the state S^T
//    (d_v x d_k) as the A operand of the tensor core, per step:
//        W^T       = K~B^T TB^T                  (issued a step ahead)
//        [U | O]  += S^T [-W^T | Q~B^T]          (U started a step ahead as V^T TB^T)
//        [O | D2] += U^T [P^T | K'B]             (O^T / scale, and the state increment)
//    A tcgen05.mma costs about the same to issue whatever its N, so products sharing an A
//    operand go out as one MMA. Only the two S^T / U^T groups lie on the state's
//    critical path; the next step's W and V^T TB^T products run while the state is
//    updated. S^T lives in fp32 registers of eight "state" warps (two warpgroups; one
//    value row and 64 keys per thread) and is mirrored as bf16 into tensor memory as the
//    next A operand; U^T likewise. One issuer thread (its own warp) issues every
//    tcgen05.mma; the state warps signal it per warp through mbarriers. Four "output"
//    warps write -W^T in bf16 over the K~B rows of the step's slot (the B operand of
//    S^T W^T), read O^T, zero it for the next step's products and store O. A producer warp
//    loads each step's V tile by TMA into one of two buffers; the products arrive in one
//    of three operand slots.
//  * ranks 1..kPro, the prologue CTAs, each compute every kPro-th step's operands (the
//    gate, the four tiles' scaled operands, [A; P] as one tcgen05 product, the 64 x 64
//    solve for TB) into a staging buffer laid out exactly as the chain CTA's operand
//    slot, and copy it there with bulk copies (shared::cta -> shared::cluster) once the
//    chain CTA has freed the slot (with three slots and three prologue CTAs, each
//    prologue CTA always fills the same slot).
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
// compiled only with -DKDA_FWD64_TRACE. Chain CTA, per step: 0 state-warp loop top,
// 1 [U | O] products issued, 2 U^T complete, 3 U^T stored, 4 [O | D2] products issued,
// 5 D2 complete, 6 state stored. The prologue CTA owning the step:
// 8 loop top, 9 raw tiles in, 20 / 26 gate pass done (first / last thread), 10 next
// fetch issued, 11 operands written, 21 [A; P] issued, 22 / 24 [A; P] complete, 23 A
// and P read out, 12 read-out barrier, 16 diagonal T tiles, 17 M, 18 M^2, 27 TB tiles,
// 13 staging slot complete, 7 copy issued.
#ifdef KDA_FWD64_TRACE
__device__ long long g_f64_trace[64][32];
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
// B1: [n][j] K-major rows, 128-byte swizzle (K = tokens): rows 0..63 = TB, rows 64..127 = P,
//     rows 128..255 = K'B^T ([c][t]); rows 64..255 are one 192-row operand [P; K'B^T]
// B2: bytes 0..16383: K~B, bytes 16384..32767: Q~B, each [c][t] (128 channel rows of 64
//     tokens). K~B is read K-major as the A operand of W^T = K~B^T TB^T and then
//     overwritten in the chain CTA by -W^T; [-W^T | Q~B^T] is then read as one MN-major
//     operand (tokens along N, channels along K)
// G : gamma^B[c] = exp(G^B_end), fp32
constexpr int SL_B1 = 0, SL_B3 = 16384, SL_B2 = 32768, SL_G = 65536;
constexpr int B2_QB = 16384;  // offset of Q~B inside B2
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
constexpr int B_FREE = 3;     // [NSLOT] slot s: its MMAs completed and gamma read (1 + 8 arrivals)
constexpr int B_UFULL = 6;    // [U | O] += S^T [-W^T | Q~B^T] complete
constexpr int B_WFULL = 7;    // W^T = K~B^T TB^T complete
constexpr int B_OFREE = 8;    // O read out and zeroed (4 output-warp arrivals)
constexpr int B_OFULL = 9;    // O^T complete
constexpr int B_D2FULL = 10;  // D2 complete
constexpr int B_DRAIN = 11;   // every MMA complete (before the tensor memory is released)
constexpr int B_SREADY = 12;  // the state's keys 0..63 in bf16 are in tensor memory (8 warp arrivals)
constexpr int B_SREADY2 = 13; // the state's keys 64..127 in bf16
constexpr int B_UREADY = 14;  // U^T's bf16 copy is in tensor memory (8 warp arrivals)
constexpr int B_WREADY = 15;  // -W^T in bf16 is in the step's slot (4 output-warp arrivals)
constexpr int NBARS = 16;
static_assert(NSLOT == 3 && B_FREE == NSLOT, "barrier table");
// tensor-memory columns: [U | O] and [O | D2] are each one contiguous MMA destination
constexpr uint32_t TM_U = 0;      // U^T fp32: 64 columns (64 tokens)
constexpr uint32_t TM_O = 64;     // O^T fp32: 64 columns
constexpr uint32_t TM_D2 = 128;   // D2 fp32: 128 columns (keys)
constexpr uint32_t TM_W = 256;    // W^T fp32: 64 columns (keys on the lanes)
constexpr uint32_t TM_AS = 320;   // S^T bf16: 64 columns (128 keys)
constexpr uint32_t TM_AU = 384;   // U^T bf16: 32 columns (64 tokens)
constexpr uint32_t kTmemCols = 512;

// ---- prologue CTA shared memory
constexpr int PR_Q = 0, PR_K = 16384, PR_A = 32768;  // raw tiles [64 t][128 c] (TMA)
// X: the operands of the [A; P] product, then the solve's fp32 scratch tiles. Every operand
// here is a set of 128 channel rows of 64 tokens (128-byte rows, 128-byte swizzle), which
// the tensor core reads MN-major (tokens along M or N, channels along K) or K-major
// (channels along N, tokens along K).
constexpr int PR_X = 65536;
constexpr int X_R = 0;       // [K~ | Q~] of the step's 64 tokens: two 16 KB halves (A operand)
constexpr int X_C = 32768;   // column tiles: [K^_0..3 | K'_0..2, Kx_20 | Kx_30, Kx_31, -] (B)
constexpr int X_BYTES = 81920;
constexpr int PR_AD = PR_X + X_BYTES;             // diagonal A tiles, fp32 [4][16][16]
constexpr int PR_AO = PR_AD + NT * TL * TL * 4;   // off-diagonal A tiles, bf16 [6][16][16]
constexpr int PR_GAM = PR_AO + 6 * TL * TL * 2;   // gamma_I[c] fp32 [4][128]
constexpr int PR_BETA = PR_GAM + NT * D * 4;      // beta [2][64]
constexpr int PR_BAR = PR_BETA + 2 * BT * 4;      // RAWFULL, SLOTFREE, MMA done, A / P done
constexpr int PR_STG = (PR_BAR + 32 + 1023) & ~1023;  // staging slot
constexpr int PR_END = PR_STG + SLOT_BYTES;
static_assert(PR_X % 1024 == 0 && (PR_X + X_C) % 1024 == 0 && PR_STG % 1024 == 0, "swizzled tiles");
// tensor-memory columns of a prologue CTA
constexpr uint32_t TP_AP = 0;    // [A; P] before masking (192 columns)
constexpr uint32_t kProTmemCols = 256;
constexpr int SMEM_USED = (PR_END > CH_BAR + NBARS * 8 ? PR_END : CH_BAR + NBARS * 8);
constexpr int SMEM_BYTES = SMEM_USED + 1024;  // + alignment slack of the dynamic base
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
// fp32 16 x 16 scratch tiles of the solve in X (free once the [A; P] product has read it):
// M = L^-1 N (6 tiles), M^2 (3), the diagonal T tiles (4)
constexpr int STG_MM = PR_X;
constexpr int STG_M2 = STG_MM + 6 * 1024;
constexpr int STG_TD = STG_M2 + 3 * 1024;
static_assert(STG_TD + 4 * 1024 <= PR_X + X_BYTES, "solve scratch stays in X");

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
// two fp32 values -> bf16x2 (x in the lower half)
__device__ __forceinline__ uint32_t pk2(float2 v) { return pack_bf16(v.x, v.y); }

// the thread that records the chain CTA's state-warp trace points
__device__ __forceinline__ bool elect_trace(int warp, int lane) { return warp == 4 && lane == 0; }

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
            // step m's V goes to buffer m & 1; its last reader, the V^T TB^T product of step
            // m - 2, completes before slot m - 2 is released
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
        } else if (warp == 2 && lane == 0) {
            // ---------------------------------------------- MMA issuer
            // A tcgen05.mma costs about the same to issue whatever its N, so products that
            // share an A operand go out as one wide MMA. Per step n (slot s):
            //   [U | O]  += S^T [-W^T | Q~B^T]      N = 128, keys 0..63 as soon as they are
            //                                       in, then 64..127; commit UFULL
            //   [O | D2] += U^T [P^T | K'B]          N = 192; commit D2FULL, OFULL, FREE
            //   W of step n + 1: K~B^T TB^T          N = 64 (once its slot is in); commit WFULL
            //   U of step n + 1: V^T TB^T            N = 64 (starts the next U)
            // W and U of the next step go out while the state warps update the state; issued
            // earlier (between the U^T hand-off and D2) they delayed D2.
            // O and D2 are zeroed by the warps that read them, so every product after the
            // first of U accumulates.
            const uint32_t id_w = idesc_bf16(128, 64, 0, 0);    // A and B K-major
            const uint32_t id_v = idesc_bf16(128, 64, 1, 0);    // A MN-major (V^T)
            const uint32_t id_1 = idesc_bf16(128, 128, 0, 1);   // B MN-major [-W^T | Q~B^T]
            const uint32_t id_2 = idesc_bf16(128, 192, 0, 0);   // B K-major [P; K'B^T]
            // slot s's descriptors are slot 0's plus s x the slot stride (16-byte units)
            const uint64_t dTB0 = sdesc_sw128(sbase + CH_SLOT + SL_B1, 16, 1024);
            const uint64_t dPK0 = sdesc_sw128(sbase + CH_SLOT + SL_B1 + BT * 128, 16, 1024);
            const uint64_t dWQ0 = sdesc_sw128(sbase + CH_SLOT + SL_B2, B2_QB, 1024);   // MN-major
            const uint64_t dKA0 = sdesc_sw128(sbase + CH_SLOT + SL_B2, 16, 1024);      // K-major
            const uint64_t dV0 = sdesc_sw128(sbase + CH_V, V_BYTES / 2, 1024);       // V^T, MN-major
            constexpr uint64_t kSlotStep = SLOT_STRIDE >> 4;
            constexpr uint64_t kVStep = V_BYTES >> 4;
            auto issue_w = [&](int m) {  // W^T of step m
                const uint64_t so = (uint64_t)(m % NSLOT) * kSlotStep;
#pragma unroll
                for (int j = 0; j < 4; ++j)  // K = 16 tokens per MMA
                    umma_ss(tmem + TM_W, dKA0 + so + (uint64_t)(2 * j), dTB0 + so + (uint64_t)(2 * j), id_w, j > 0);
                umma_commit(bar(B_WFULL));
            };
            auto issue_vtb = [&](int m) {  // U of step m starts as V^T TB^T
                const uint64_t so = (uint64_t)(m % NSLOT) * kSlotStep;
                const uint64_t vo = (uint64_t)(m & 1) * kVStep;
#pragma unroll
                for (int j = 0; j < 4; ++j)  // 16 token rows (2048 bytes) of V per MMA
                    umma_ss(tmem + TM_U, dV0 + vo + (uint64_t)(128 * j), dTB0 + so + (uint64_t)(2 * j), id_v, j > 0);
            };
            bool ok = true;
            if (nblocks > 0) {
                ok = wait_bar(bar(B_FULL), 0);
                if (ok) {
                    tc_fence_after();
                    issue_w(0);
                    issue_vtb(0);
                }
            }
            for (int n = 0; ok && n < nblocks; ++n) {
                const int s = n % NSLOT;
                const uint64_t so = s * kSlotStep;
                if (!wait_bar(bar(B_WREADY), n & 1)) break;  // -W^T of step n is in slot s
                if (!wait_bar(bar(B_OFREE), n & 1)) break;   // O read out and zeroed
                if (!wait_bar(bar(B_SREADY), n & 1)) break;  // S^T keys 0..63 (bf16) of step n
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; ++k)  // 16 channel rows (2048 bytes) per MMA
                    umma_ts(tmem + TM_U, tmem + TM_AS + 8u * k, dWQ0 + so + (uint64_t)(128 * k), id_1, 1);
                if (!wait_bar(bar(B_SREADY2), n & 1)) break;  // keys 64..127
                tc_fence_after();
#pragma unroll
                for (int k = 4; k < 8; ++k)
                    umma_ts(tmem + TM_U, tmem + TM_AS + 8u * k, dWQ0 + so + (uint64_t)(128 * k), id_1, 1);
                umma_commit(bar(B_UFULL));
                F64_TRACE(n, 1);
                if (!wait_bar(bar(B_UREADY), n & 1)) break;  // U^T (bf16) of step n is in
                tc_fence_after();
#pragma unroll
                for (int j = 0; j < 4; ++j)  // K = 16 tokens per MMA
                    umma_ts(tmem + TM_O, tmem + TM_AU + 8u * j, dPK0 + so + (uint64_t)(2 * j), id_2, 1);
                umma_commit(bar(B_D2FULL));
                umma_commit(bar(B_OFULL));
                umma_commit(bar(B_FREE + s));
                F64_TRACE(n, 4);
                if (n + 1 < nblocks) {  // the next step's W and U while the state is updated
                    if (!wait_bar(bar(B_FULL + (n + 1) % NSLOT), ((n + 1) / NSLOT) & 1)) break;
                    tc_fence_after();
                    issue_w(n + 1);
                    issue_vtb(n + 1);  // U of step n has been read (UREADY above)
                }
            }
            // every MMA has completed before the tensor memory is released
            umma_commit(bar(B_DRAIN));
            wait_bar(bar(B_DRAIN), 0);
        }
    } else if (warp < 12) {
        regs_set<kRegsState>();
        // -------------------------------------------------- state warps (two warpgroups)
        // Thread (value row v = TMEM lane, warpgroup wg) holds S^T[v][k] in fp32 registers
        // for the keys k = 64 h + 32 wg + j (h = 0, 1; j < 32): each half of the keys is
        // split over both warpgroups, so that each half is updated, converted and handed to
        // the issuer (SREADY, SREADY2) while the other is still being updated. Each warp
        // signals the issuer on its own (8 arrivals per barrier).
        const int wg = (warp - 4) >> 2;
        const int v = ((warp & 3) << 5) + lane;                 // value row = TMEM lane
        const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;  // lane quarter
        uint32_t zero[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) zero[j] = 0u;
        float S[64];  // S[32 h + j] = S^T[v][64 h + 32 wg + j]
        {
            const float *h0 = p.h0 ? p.h0 + ((size_t)seq * H + head) * D * D : nullptr;
#pragma unroll
            for (int c = 0; c < 64; ++c) S[c] = h0 ? h0[(size_t)(64 * (c >> 5) + 32 * wg + (c & 31)) * D + v] : 0.f;
        }
        auto store_half = [&](int h) {  // bf16 copy of this thread's keys of half h -> A operand
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) w[j] = pack_bf16(S[32 * h + 2 * j], S[32 * h + 2 * j + 1]);
            tmem_st16(tmem + lb + TM_AS + 32 * h + 16 * wg, w);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(h ? B_SREADY2 : B_SREADY));
        };
        tmem_st32(tmem + lb + TM_D2 + 32u * wg, zero);        // D2 starts at zero
        tmem_st32(tmem + lb + TM_D2 + 64u + 32u * wg, zero);
        store_half(0);
        store_half(1);
        for (int n = 0; n < nblocks; ++n) {
            const int s = n % NSLOT;
            if (elect_trace(warp, lane)) F64_TRACE(n, 0);
            // ---- the slot's FULL phase is observed first: it makes gamma^B (landed by bulk
            //      copy) visible to this thread's loads
            if (!wait_bar(bar(B_FULL + s), (n / NSLOT) & 1)) break;
            // ---- U^T = V^T TB^T - S^T W^T -> bf16 A operand, 32 tokens per warpgroup
            if (!wait_bar(bar(B_UFULL), n & 1)) break;
            if (elect_trace(warp, lane)) F64_TRACE(n, 2);
            tc_fence_after();
            {
                uint32_t r[32], w[16];
                tmem_ld32(tmem + lb + TM_U + 32u * wg, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    w[j] = pack_bf16(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
                tmem_st16(tmem + lb + TM_AU + 16 * wg, w);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_UREADY));
            if (elect_trace(warp, lane)) F64_TRACE(n, 3);
            // ---- S^T <- S^T diag(gamma^B) + D2, one key half at a time (D2 zeroed behind
            //      the read), then bf16
            if (!wait_bar(bar(B_D2FULL), n & 1)) break;
            if (elect_trace(warp, lane)) F64_TRACE(n, 5);
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float4 *gam = reinterpret_cast<const float4 *>(sm + CH_G + s * D * 4 + (64 * h + 32 * wg) * 4);
                uint32_t r[32];
                const uint32_t col = tmem + lb + TM_D2 + 64u * h + 32u * wg;
                tmem_ld32(col, r);
                tmem_ld_wait();
                tmem_st32(col, zero);
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const float4 g = gam[j4];
                    const int c = 32 * h + 4 * j4;
                    S[c] = fmaf(g.x, S[c], __uint_as_float(r[4 * j4]));
                    S[c + 1] = fmaf(g.y, S[c + 1], __uint_as_float(r[4 * j4 + 1]));
                    S[c + 2] = fmaf(g.z, S[c + 2], __uint_as_float(r[4 * j4 + 2]));
                    S[c + 3] = fmaf(g.w, S[c + 3], __uint_as_float(r[4 * j4 + 3]));
                }
                if (h == 1) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_FREE + s));  // this warp has read gamma^B
                }
                store_half(h);
            }
            if (elect_trace(warp, lane)) F64_TRACE(n, 6);
        }
        if (p.h_final) {
            float *hf = p.h_final + ((size_t)seq * H + head) * D * D;
#pragma unroll
            for (int c = 0; c < 64; ++c) hf[(size_t)(64 * (c >> 5) + 32 * wg + (c & 31)) * D + v] = S[c];
        }
    } else {
        regs_set<kRegsOut>();
        // -------------------------------------------------- output warps
        // Each step: -W^T of the next step from tensor memory into that step's slot (over
        // its K~B rows, which the W product has finished reading), then this step's O^T,
        // which is zeroed behind the read for the next step's products.
        const int v = threadIdx.x - 384;  // TMEM lane: a value row of O^T, a key row of W^T
        const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
        const size_t tstride = (size_t)H * D;
        uint32_t zero[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) zero[j] = 0u;
        auto release_o = [&]() {  // O zeroed, then free for the next step's products
            tmem_st32(tmem + lb + TM_O, zero);
            tmem_st32(tmem + lb + TM_O + 32u, zero);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_OFREE));
        };
        auto convert_w = [&](int m) -> bool {  // -W^T of step m -> slot m % NSLOT, [c][t] bf16
            const bool got = wait_bar(bar(B_WFULL), m & 1);
            if (!__all_sync(0xffffffffu, got)) return false;
            tc_fence_after();
            uint32_t r0[32], r1[32];
            tmem_ld32(tmem + lb + TM_W, r0);
            tmem_ld32(tmem + lb + TM_W + 32u, r1);
            tmem_ld_wait();
            unsigned char *row = sm + CH_SLOT + (m % NSLOT) * SLOT_STRIDE + SL_B2;
#pragma unroll
            for (int q = 0; q < 4; ++q) {  // 8 tokens (16 bytes) per store
                uint4 w0, w1;
                w0.x = pack_bf16(-__uint_as_float(r0[8 * q]), -__uint_as_float(r0[8 * q + 1]));
                w0.y = pack_bf16(-__uint_as_float(r0[8 * q + 2]), -__uint_as_float(r0[8 * q + 3]));
                w0.z = pack_bf16(-__uint_as_float(r0[8 * q + 4]), -__uint_as_float(r0[8 * q + 5]));
                w0.w = pack_bf16(-__uint_as_float(r0[8 * q + 6]), -__uint_as_float(r0[8 * q + 7]));
                w1.x = pack_bf16(-__uint_as_float(r1[8 * q]), -__uint_as_float(r1[8 * q + 1]));
                w1.y = pack_bf16(-__uint_as_float(r1[8 * q + 2]), -__uint_as_float(r1[8 * q + 3]));
                w1.z = pack_bf16(-__uint_as_float(r1[8 * q + 4]), -__uint_as_float(r1[8 * q + 5]));
                w1.w = pack_bf16(-__uint_as_float(r1[8 * q + 6]), -__uint_as_float(r1[8 * q + 7]));
                *reinterpret_cast<uint4 *>(row + sw128(v, 8 * q)) = w0;
                *reinterpret_cast<uint4 *>(row + sw128(v, 32 + 8 * q)) = w1;
            }
            fence_proxy_async();  // generic writes -> the tensor core's reads of the slot
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_WREADY));
            return true;
        };
        release_o();
        bool ok = nblocks == 0 || convert_w(0);
        for (int n = 0; ok && n < nblocks; ++n) {
            if (n + 1 < nblocks && !convert_w(n + 1)) break;
            const bool got = wait_bar(bar(B_OFULL), n & 1);
            if (!__all_sync(0xffffffffu, got)) break;
            tc_fence_after();
            uint32_t r0[32], r1[32];
            tmem_ld32(tmem + lb + TM_O, r0);
            tmem_ld32(tmem + lb + TM_O + 32u, r1);
            tmem_ld_wait();
            release_o();
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
// the six off-diagonal tile pairs (I, J), in the order of the off-diagonal A tiles
__device__ __constant__ int kOffI[6] = {1, 2, 3, 2, 3, 3};
__device__ __constant__ int kOffJ[6] = {0, 1, 2, 0, 1, 0};
// column of the A / P product holding X_IJ, the column tile of pair (I, J <= I): K^_I on
// the diagonal, K'_J next to it, K'_J scaled by the decays of the tiles in between
// further out
__device__ __forceinline__ int ap_column(int I, int J) {
    if (I == J) return TL * I;
    if (I - J == 1) return 64 + TL * J;
    if (I == 2) return 112;
    return J == 0 ? 128 : 144;
}
// a 16 x 16 accumulator (two m16n8 fragments) into a row-major fp32 tile, scaled
__device__ __forceinline__ void store16(float *dst, const float (&acc)[2][4], float sc, int g, int t4) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        *reinterpret_cast<float2 *>(dst + g * 16 + 8 * nt + 2 * t4) = make_float2(sc * acc[nt][0], sc * acc[nt][1]);
        *reinterpret_cast<float2 *>(dst + (g + 8) * 16 + 8 * nt + 2 * t4) = make_float2(sc * acc[nt][2], sc * acc[nt][3]);
    }
}
// the A fragment of a row-major fp32 16 x 16 tile (row pitch lp), rounded to bf16
__device__ __forceinline__ void frag_a_f32(uint32_t (&a)[4], const float *L, int lp, int g, int t4) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int row = g + 8 * (q & 1), col = 2 * t4 + 8 * (q >> 1);
        const float2 v = *reinterpret_cast<const float2 *>(L + row * lp + col);
        a[q] = pack_bf16(v.x, v.y);
    }
}
// acc (16 x 16 as two m16n8 fragments) += L (16 x 16 fp32, row pitch lp) x R (16 x 16
// fp32, row pitch rp), the operands rounded to bf16 (one mma.sync per 8-column tile).
// Used inside the 64 x 64 solve, whose result is itself rounded to bf16: the products'
// rounding is about two orders of magnitude below that.
__device__ __forceinline__ void mma16_f32(float (&acc)[2][4], const float *L, int lp, const float *R,
                                          int rp, int g, int t4) {
    uint32_t a[4];
    frag_a_f32(a, L, lp, g, t4);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int n = 8 * nt + g;
        const uint32_t b0 = pack_bf16(R[(2 * t4) * rp + n], R[(2 * t4 + 1) * rp + n]);
        const uint32_t b1 = pack_bf16(R[(2 * t4 + 8) * rp + n], R[(2 * t4 + 9) * rp + n]);
        mma16816(acc[nt], a, b0, b1);
    }
}
// acc += (A fragment a) x R (16 x 16 fp32, row pitch rp, rounded to bf16)
__device__ __forceinline__ void mma16_ar(float (&acc)[2][4], const uint32_t (&a)[4], const float *R, int rp,
                                         int g, int t4) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int n = 8 * nt + g;
        const uint32_t b0 = pack_bf16(R[(2 * t4) * rp + n], R[(2 * t4 + 1) * rp + n]);
        const uint32_t b1 = pack_bf16(R[(2 * t4 + 8) * rp + n], R[(2 * t4 + 9) * rp + n]);
        mma16816(acc[nt], a, b0, b1);
    }
}
// the same with R a row-major bf16 16 x 16 tile
__device__ __forceinline__ void mma16_fb(float (&acc)[2][4], const float *L, int lp,
                                         const unsigned short *R, int g, int t4) {
    uint32_t a[4];
    frag_a_f32(a, L, lp, g, t4);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int n = 8 * nt + g;
        const uint32_t b0 = (uint32_t)R[(2 * t4) * TL + n] | ((uint32_t)R[(2 * t4 + 1) * TL + n] << 16);
        const uint32_t b1 = (uint32_t)R[(2 * t4 + 8) * TL + n] | ((uint32_t)R[(2 * t4 + 9) * TL + n] << 16);
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
    const uint32_t rawfull = sbase + PR_BAR, slotfree = sbase + PR_BAR + 8, mmabar = sbase + PR_BAR + 16,
                   apbar = sbase + PR_BAR + 24;
    const uint32_t stg = sbase + PR_STG;
    const int g = lane >> 2, t4 = lane & 3;
    unsigned char *X = sm + PR_X;
    float *AD = reinterpret_cast<float *>(sm + PR_AD);
    const unsigned short *AO = reinterpret_cast<const unsigned short *>(sm + PR_AO);
    float *MM = reinterpret_cast<float *>(sm + STG_MM);   // M = L^-1 N, 6 tiles
    auto M2 = [&](int q) {                                // M^2: (2,0), (3,1), (3,0)
        return reinterpret_cast<float *>(sm + STG_M2 + 1024 * q);
    };
    float *TD = reinterpret_cast<float *>(sm + STG_TD);   // T_II, 4 tiles
    float *GAM = reinterpret_cast<float *>(sm + PR_GAM);

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
    // exp(g) = exp(-5 sigmoid(a)) in place over the raw gate-logit tile, by the threads
    // [first, first + count): the gate pass of a step then reads exp(g) directly. The
    // MUFU-bound exponentials of the next owned step run on the warps the solve leaves
    // idle.
    auto exp_gate_inplace = [&](int first, int count) {
        float4 *ra4 = reinterpret_cast<float4 *>(sm + PR_A);
#pragma unroll 4
        for (int i = tid - first; i < BT * D / 4; i += count) {
            float4 v = ra4[i];
            v.x = __expf(kGMin * __fdividef(1.f, 1.f + __expf(-v.x)));
            v.y = __expf(kGMin * __fdividef(1.f, 1.f + __expf(-v.y)));
            v.z = __expf(kGMin * __fdividef(1.f, 1.f + __expf(-v.z)));
            v.w = __expf(kGMin * __fdividef(1.f, 1.f + __expf(-v.w)));
            ra4[i] = v;
        }
    };
    fetch(prank, 0);
    // tensor memory for the products. B1 starts at zero: the tiles of TB and of P above
    // the diagonal are never written, so they stay zero in every step's slot. The unused
    // last 32 columns of the column tiles are zeroed once (their products are never read).
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kProTmemCols);
    for (int i = tid; i < 16384 / 16; i += kThreads) {
        reinterpret_cast<uint4 *>(sm + PR_STG + SL_B1)[i] = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint4 *>(X + X_C + 32768)[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t ptmem = *tmem_slot;
    bool bad = false;   // a wait of this thread gave up (thread 0: slots; warps 8-15: raw tiles)
    int nfree = 0;      // slot-free signals consumed (thread 0)
    if (prank < nblocks) {  // the first owned step's raw tiles, exp(g) by every thread
        bad = !wait_bar(rawfull, 0);
        if (!bad) exp_gate_inplace(0, kThreads);
        fence_proxy_async();  // generic writes of the raw tile -> the next TMA into it
    }
    int k = 0;
    for (int m = prank; m < nblocks; m += kPro, ++k) {
        const int L = min(BT, t1 - (t0 + m * BT));
        const float *bet = reinterpret_cast<const float *>(sm + PR_BETA) + (k & 1) * BT;
        // ---- P0: this step's raw tiles are in, exp(g) already formed over the gate tile
        //      (before the loop, or by warps 8-15 during the previous owned step's solve)
        if (tid == 0) F64_TRACE(m, 8);
        if (warp == 15) cp_async_wait0();
        if (__syncthreads_or(bad)) break;
        mbar_try(rawfull, k & 1);  // observe the completed phase (the q and k tiles)
        if (tid == 0) F64_TRACE(m, 9);
        // ---- P1: gate pass, one (key channel c, tile I) per thread: exp(g) of its 16
        //      tokens and the inclusive within-tile decay Gamma_r = exp(G_r)
        const int c = tid & (D - 1), I = tid >> 7, rb = TL * I;
        float eg[TL], gm[TL];
        uint32_t kq[TL];  // k_r (low half) and q_r (high half), bf16
        {
            const float *ra = reinterpret_cast<const float *>(sm + PR_A);
            const unsigned short *rq = reinterpret_cast<const unsigned short *>(sm + PR_Q);
            const unsigned short *rk = reinterpret_cast<const unsigned short *>(sm + PR_K);
#pragma unroll
            for (int r = 0; r < TL; ++r) eg[r] = ra[(rb + r) * D + c];  // exp(g), g = -5 sigmoid(a)
            float gam = 1.f;
#pragma unroll
            for (int r = 0; r < TL; ++r) {
                const bool in = rb + r < L;
                const float e = eg[r];
                eg[r] = in ? e : 1.f;
                kq[r] = in ? ((uint32_t)rk[(rb + r) * D + c] | ((uint32_t)rq[(rb + r) * D + c] << 16)) : 0u;
                gam *= eg[r];
                gm[r] = gam;
            }
            GAM[I * D + c] = gam;  // gamma_I = exp(G_end), >= exp(-80)
        }
        if (tid == 0) F64_TRACE(m, 20);
        if (tid == 511) F64_TRACE(m, 26);
        __syncthreads();
        fetch(m + kPro, (k + 1) & 1);  // the raw tiles have been consumed
        if (tid == 0) F64_TRACE(m, 10);
        // ---- P2: every scaled operand of this (channel, tile), from fp32 values:
        //   R = [K~ | Q~] (K~ = K Gamma), the column tiles K^ = K / Gamma and
        //   K' = K gamma / Gamma (and K' scaled by the decays of the tiles after it: Kx),
        //   K'B = K' prod_{J > I} gamma_J, gamma^B, K~B and Q~B (x prod_{J < I} gamma_J) stay
        //   in registers until the staging slot may be written.
        uint32_t wkb[TL / 2], wqb[TL / 2], wkp[TL / 2];
        float gB = 0.f;
        {
            float pre = 1.f, post = 1.f, gj[NT];
#pragma unroll
            for (int J = 0; J < NT; ++J) {
                gj[J] = GAM[J * D + c];
                if (J < I) pre *= gj[J];
                if (J > I) post *= gj[J];
            }
            const float inv = __frcp_rn(gm[TL - 1]);  // exp(-G_end) <= exp(80)
            auto put2 = [&](unsigned char *base, int col, const uint32_t (&w)[TL / 2]) {
                *reinterpret_cast<uint4 *>(base + sw128(c, col)) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4 *>(base + sw128(c, col + 8)) = make_uint4(w[4], w[5], w[6], w[7]);
            };
            // token pairs (r, r + 1) as float2: the products below are packed fp32x2 multiplies
            float2 k2[TL / 2], kp[TL / 2];   // K, and K' = K exp(G_end - G_r) (suffix product of exp(g))
            {
                float sf[TL];
                float acc = 1.f;
#pragma unroll
                for (int r = TL - 1; r >= 0; --r) {
                    sf[r] = acc;
                    acc *= eg[r];
                }
#pragma unroll
                for (int i = 0; i < TL / 2; ++i) {
                    k2[i] = make_float2(__uint_as_float(kq[2 * i] << 16), __uint_as_float(kq[2 * i + 1] << 16));
                    kp[i] = __fmul2_rn(k2[i], make_float2(sf[2 * i], sf[2 * i + 1]));
                }
            }
            const float2 pre2 = make_float2(pre, pre);
            uint32_t w[TL / 2];
#pragma unroll
            for (int i = 0; i < TL / 2; ++i) {
                const float2 a = __fmul2_rn(k2[i], make_float2(gm[2 * i], gm[2 * i + 1]));  // K~
                w[i] = pk2(a);
                wkb[i] = pk2(__fmul2_rn(a, pre2));
            }
            put2(X + X_R, rb, w);                                  // K~
#pragma unroll
            for (int i = 0; i < TL / 2; ++i) {
                const float2 q2 = make_float2(__uint_as_float(kq[2 * i] & 0xffff0000u),
                                              __uint_as_float(kq[2 * i + 1] & 0xffff0000u));
                const float2 b = __fmul2_rn(q2, make_float2(gm[2 * i], gm[2 * i + 1]));  // Q~
                w[i] = pk2(b);
                wqb[i] = pk2(__fmul2_rn(b, pre2));
            }
            put2(X + X_R + 16384, rb, w);                          // Q~
            auto scaled = [&](float sc) {
                const float2 s2 = make_float2(sc, sc);
#pragma unroll
                for (int i = 0; i < TL / 2; ++i) w[i] = pk2(__fmul2_rn(kp[i], s2));
            };
            scaled(inv);
            put2(X + X_C, rb, w);                                  // K^_I
            if (I < NT - 1) {
#pragma unroll
                for (int i = 0; i < TL / 2; ++i) w[i] = pk2(kp[i]);
                put2(X + X_C + 16384, rb, w);                      // K'_I
            }
            {
                const float2 s2 = make_float2(post, post);
#pragma unroll
                for (int i = 0; i < TL / 2; ++i) wkp[i] = pk2(__fmul2_rn(kp[i], s2));  // K'B
            }
            if (I == 0) {
                scaled(gj[1]);
                put2(X + X_C + 16384, 48, w);                      // Kx_20 = K'_0 gamma_1
                scaled(gj[1] * gj[2]);
                put2(X + X_C + 32768, 0, w);                       // Kx_30 = K'_0 gamma_1 gamma_2
                gB = gj[0] * gj[1] * gj[2] * gj[3];  // gamma^B = exp(G^B_end)
            } else if (I == 1) {
                scaled(gj[2]);
                put2(X + X_C + 32768, 16, w);                      // Kx_31 = K'_1 gamma_2
            }
        }
        if (tid == 0) bulk_wait_read0();  // the previous step's copies have read the staging slot
        fence_proxy_async();  // generic writes of X -> the tensor core's reads
        tc_fence_before();
        __syncthreads();
        if (tid == 0) F64_TRACE(m, 11);
        // ---- P3: [A; P] before masking = [K~; Q~] [column tiles]^T on this CTA's tensor
        //      core (M = 128 tokens, N = 192 columns, K = 128 channels)
        if (tid == 0) {
            tc_fence_after();
            const uint64_t da = sdesc_sw128(sbase + PR_X + X_R, 16384, 1024);
            const uint64_t db = sdesc_sw128(sbase + PR_X + X_C, 16384, 1024);
            const uint32_t idap = idesc_bf16(128, 192, 1, 1);
#pragma unroll
            for (int kk2 = 0; kk2 < 8; ++kk2)  // K = 16 channels per MMA (+2048 bytes)
                umma_ss(ptmem + TP_AP, da + 128 * kk2, db + 128 * kk2, idap, kk2 > 0);
            umma_commit(apbar);
            F64_TRACE(m, 21);
        }
        {   // while the product runs: K'B, K~B and Q~B ([c][64 t]) and gamma^B into the staging
            // slot (the previous copy out of it has completed: checked before the barrier above)
            unsigned char *kb = sm + PR_STG + SL_B2;
            *reinterpret_cast<uint4 *>(kb + sw128(c, rb)) = make_uint4(wkb[0], wkb[1], wkb[2], wkb[3]);
            *reinterpret_cast<uint4 *>(kb + sw128(c, rb + 8)) = make_uint4(wkb[4], wkb[5], wkb[6], wkb[7]);
            unsigned char *b3 = sm + PR_STG + SL_B3;
            *reinterpret_cast<uint4 *>(b3 + sw128(c, rb)) = make_uint4(wkp[0], wkp[1], wkp[2], wkp[3]);
            *reinterpret_cast<uint4 *>(b3 + sw128(c, rb + 8)) = make_uint4(wkp[4], wkp[5], wkp[6], wkp[7]);
            unsigned char *qb = sm + PR_STG + SL_B2 + B2_QB;
            *reinterpret_cast<uint4 *>(qb + sw128(c, rb)) = make_uint4(wqb[0], wqb[1], wqb[2], wqb[3]);
            *reinterpret_cast<uint4 *>(qb + sw128(c, rb + 8)) = make_uint4(wqb[4], wqb[5], wqb[6], wqb[7]);
            if (I == 0) reinterpret_cast<float *>(sm + PR_STG + SL_G)[c] = gB;
        }
        {
            const bool got = wait_bar(apbar, k & 1);
            if (tid == 0) F64_TRACE(m, 22);
            if (__all_sync(0xffffffffu, got)) {
                tc_fence_after();
                if (tid == 0) F64_TRACE(m, 24);
                // A (rows 0..63: beta-scaled, strictly lower on the diagonal tiles) and P
                // (rows 64..127: lower on the diagonal tiles) out of the product's columns.
                // Warp = (lane quarter q, part); each part takes whole 16-column chunks.
                const int q = warp & 3, part = warp >> 2;
                const bool prow = q >= 2;
                const int Il = 2 * (q & 1) + (lane >> 4), r = lane & 15;
                int n_ch, I0, J0, I1 = 0, J1 = 0;
                if ((q & 1) == 0) {  // row tiles 0, 1: chunks (0,0), (1,1), (1,0)
                    n_ch = part < 3 ? 1 : 0;
                    I0 = part == 0 ? 0 : 1;
                    J0 = part == 1 ? 1 : 0;
                } else {             // row tiles 2, 3: seven chunks over four parts
                    n_ch = part < 3 ? 2 : 1;
                    I0 = 2;
                    J0 = part == 0 ? 2 : (part == 1 ? 1 : (part == 2 ? 0 : 1));
                    if (part == 3) I0 = 3;
                    I1 = 3;
                    J1 = part == 0 ? 3 : (part == 1 ? 2 : 0);
                }
                const uint32_t trow = ptmem + TP_AP + ((uint32_t)(32 * q) << 16);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    if (u < n_ch) {
                        const int Ic = u == 0 ? I0 : I1, Jc = u == 0 ? J0 : J1;
                        uint32_t v[16];
                        tmem_ld16(trow + (uint32_t)ap_column(Ic, Jc), v);
                        tmem_ld_wait();
                        if (Il == Ic) {
                            const bool diag = Ic == Jc;
                            if (!prow) {
                                const float b = bet[TL * Ic + r];
                                auto av = [&](int j) { return (!diag || j < r) ? b * __uint_as_float(v[j]) : 0.f; };
                                if (diag) {  // column j of A_II, rows p + 4 q at [j][p][q]
#pragma unroll
                                    for (int j = 0; j < 16; ++j) AD[(Ic * TL + j) * TL + 4 * (r & 3) + (r >> 2)] = av(j);
                                } else {
                                    uint32_t w[8];
#pragma unroll
                                    for (int j = 0; j < 8; ++j) w[j] = pack_bf16(av(2 * j), av(2 * j + 1));
                                    uint4 *dst = reinterpret_cast<uint4 *>(sm + PR_AO + (off_blk(Ic, Jc) * 256 + r * TL) * 2);
                                    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                                    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                                }
                            } else {
                                uint32_t w[8];
#pragma unroll
                                for (int j = 0; j < 16; j += 2)
                                    w[j >> 1] = pack_bf16((!diag || j <= r) ? __uint_as_float(v[j]) : 0.f,
                                                          (!diag || j + 1 <= r) ? __uint_as_float(v[j + 1]) : 0.f);
                                const int row = BT + TL * Ic + r;
                                unsigned char *b1 = sm + PR_STG + SL_B1;
                                *reinterpret_cast<uint4 *>(b1 + sw128(row, TL * Jc)) = make_uint4(w[0], w[1], w[2], w[3]);
                                *reinterpret_cast<uint4 *>(b1 + sw128(row, TL * Jc + 8)) = make_uint4(w[4], w[5], w[6], w[7]);
                            }
                        }
                    }
                }
            }
            if (tid == 160) F64_TRACE(m, 23);
            tc_fence_before();
        }
        __syncthreads();
        if (tid == 0) F64_TRACE(m, 12);
        // ---- P4 (warps 0-5): T = (I + A)^-1, A strictly lower, in 16 x 16 tiles. L = the
        //   diagonal tiles of I + A, N = the rest, M = L^-1 N (M_IJ = T_II A_IJ, I > J;
        //   nilpotent, M^4 = 0), so T = (I + M)^-1 L^-1 = (I - M)(I + M^2) L^-1. Diagonal
        //   tiles T_II: fp32 forward substitution, one column per thread. Products of
        //   tiles: tensor cores, operands rounded to bf16. TB = T diag(beta) goes to rows
        //   0..63 of B1 as each tile is done (the tiles above the diagonal stay 0).
        if (warp < 8) {
            constexpr int kSolveThreads = 256;
            {
                // column j of T_II = (I + A_II)^-1, right-looking: once x_i is final (in the
                // thread owning row i) it is broadcast to the column's four threads, each of
                // which folds it into its rows p, p + 4, p + 8, p + 12
                const int Id = tid >> 6, j = (tid >> 2) & 15, pr = tid & 3;
                const float *Ac = AD + Id * TL * TL + 4 * pr;  // column i: Ac[16 i + q] = A[pr + 4q][i]
                float x[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) x[q] = pr + 4 * q == j ? 1.f : 0.f;
#pragma unroll
                for (int i = 0; i < TL - 1; ++i) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(Ac + TL * i);
                    const float xi = __shfl_sync(0xffffffffu, x[i >> 2], (lane & ~3) | (i & 3));
                    const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (4 * q + 3 >= i + 1)  // some of this q's rows can lie below i
                            x[q] = pr + 4 * q > i ? fmaf(-av[q], xi, x[q]) : x[q];
                }
                const float bj = bet[TL * Id + j];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int r = pr + 4 * q;
                    TD[(Id * TL + r) * TL + j] = x[q];
                    *reinterpret_cast<__nv_bfloat16 *>(sm + PR_STG + SL_B1 + sw128(TL * Id + r, TL * Id + j)) =
                        __float2bfloat16_rn(x[q] * bj);
                }
            }
            named_sync(2, kSolveThreads);
            if (tid == 0) F64_TRACE(m, 16);
            if (warp < 6) {   // M_IJ = T_II A_IJ for the six pairs I > J (one warp each)
                const int Ir = kOffI[warp];
                float acc[2][4] = {};
                mma16_fb(acc, TD + Ir * 256, TL, AO + warp * 256, g, t4);
                store16(MM + warp * 256, acc, 1.f, g, t4);
            }
            named_sync(2, kSolveThreads);
            if (tid == 0) F64_TRACE(m, 17);
            // M^2: (2,0) = M21 M10, (3,1) = M32 M21, (3,0) = M31 M10 + M32 M20
            if (warp < 3) {
                float acc[2][4] = {};
                if (warp == 0) mma16_f32(acc, MM + 1 * 256, TL, MM + 0 * 256, TL, g, t4);
                if (warp == 1) mma16_f32(acc, MM + 2 * 256, TL, MM + 1 * 256, TL, g, t4);
                if (warp == 2) {
                    mma16_f32(acc, MM + 4 * 256, TL, MM + 0 * 256, TL, g, t4);
                    mma16_f32(acc, MM + 2 * 256, TL, MM + 3 * 256, TL, g, t4);
                }
                store16(M2(warp), acc, 1.f, g, t4);
            }
            named_sync(2, kSolveThreads);
            if (tid == 0) F64_TRACE(m, 18);
            if (warp < 6) {   // T_IJ = [-(M)_IJ + (M^2)_IJ - (M^3)_IJ] T_JJ, M^3 only at (3,0) = M32 (M^2)_20;
                // TB_IJ = T_IJ diag(beta_J) straight into B1. The left factor is formed in
                // the accumulator layout, which is also the A-fragment layout of a 16 x 16.
                const int Ir = kOffI[warp], Jc = kOffJ[warp];
                const int q2 = (Ir == 2 && Jc == 0) ? 0 : (Ir == 3 && Jc == 1) ? 1 : (Ir == 3 && Jc == 0) ? 2 : -1;
                float c3[2][4] = {};
                if (q2 == 2) mma16_f32(c3, MM + 2 * 256, TL, M2(0), TL, g, t4);
                uint32_t la[4];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int row = g + 8 * h, col = 8 * nt + 2 * t4;
                        float2 v2 = *reinterpret_cast<const float2 *>(MM + warp * 256 + row * TL + col);
                        v2.x = -v2.x;
                        v2.y = -v2.y;
                        if (q2 >= 0) {
                            const float2 w2 = *reinterpret_cast<const float2 *>(M2(q2) + row * TL + col);
                            v2.x += w2.x;
                            v2.y += w2.y;
                        }
                        v2.x -= c3[nt][2 * h];
                        v2.y -= c3[nt][2 * h + 1];
                        la[2 * nt + h] = pack_bf16(v2.x, v2.y);
                    }
                float acc[2][4] = {};
                mma16_ar(acc, la, TD + Jc * 256, TL, g, t4);
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
            if (tid == 0) F64_TRACE(m, 27);
        } else if (m + kPro < nblocks) {
            // warps 8-15: the next owned step's raw tiles (fetched after this step's gate
            // pass) and exp(g) in place over its gate tile
            bad = !wait_bar(rawfull, (k + 1) & 1);
            if (!bad) exp_gate_inplace(8 * 32, kThreads - 8 * 32);
            if (tid == 256) F64_TRACE(m, 28);
        }
        fence_proxy_async();  // generic writes of the staging slot (and of the gate tile) -> the
                              // bulk copy's reads (and the next TMA into the tile)
        tc_fence_before();
        __syncthreads();
        if (tid == 0) F64_TRACE(m, 13);
        // ---- P5: into the chain CTA's slot m % NSLOT once step m - NSLOT has consumed it
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
        wait_bar(mmabar, 0);      // the only commit on this barrier
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
                mbar_init(sbase + CH_BAR + 8u * (B_FREE + s), 1 + 8);
            }
            mbar_init(sbase + CH_BAR + 8u * B_UFULL, 1);
            mbar_init(sbase + CH_BAR + 8u * B_WFULL, 1);
            mbar_init(sbase + CH_BAR + 8u * B_OFREE, 4);
            mbar_init(sbase + CH_BAR + 8u * B_OFULL, 1);
            mbar_init(sbase + CH_BAR + 8u * B_D2FULL, 1);
            mbar_init(sbase + CH_BAR + 8u * B_DRAIN, 1);
            mbar_init(sbase + CH_BAR + 8u * B_SREADY, 8);
            mbar_init(sbase + CH_BAR + 8u * B_SREADY2, 8);
            mbar_init(sbase + CH_BAR + 8u * B_UREADY, 8);
            mbar_init(sbase + CH_BAR + 8u * B_WREADY, 4);
        } else {
            mbar_init(sbase + PR_BAR, 1);
            mbar_init(sbase + PR_BAR + 8, 1);
            mbar_init(sbase + PR_BAR + 16, 1);
            mbar_init(sbase + PR_BAR + 24, 1);
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
