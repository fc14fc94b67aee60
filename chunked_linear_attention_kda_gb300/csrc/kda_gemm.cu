// kda_gemm.cu -- the gate projection a = x W^T + b that produces the gate logits from
// the layer input ("projection(x)" inside the bounded gate -5 sigmoid(projection(x)):
// "Architecture Analysis of Ultra-Long Context Sparse MoE Models", §2.2; "From Numerical
// Stability to Load Balancing", §2.2). x [M, K] and W [N, K] bf16 (both K-major, W as a
// linear layer stores it), b [N] fp32 or none, a [M, N] fp32 = [tokens, heads x d_k].
//
// A persistent tcgen05 GEMM, one CTA per SM, 192 threads:
//   warp 0     TMA producer: 128 x 64 tiles of x and 256 x 64 tiles of W, 128-byte
//              swizzled, into a 4-stage ring (48 KB per stage), mbarrier-tracked;
//   warp 1     owns the tensor memory (512 columns: two 128 x 256 fp32 accumulators) and
//              its lane 0 issues tcgen05.mma (M = 128, N = 256, K = 16; four per stage),
//              committing each stage back to the producer and each finished tile to the
//              epilogue;
//   warps 2-5  epilogue: tcgen05.ld of their 32 accumulator lanes, + b, fp32 stores (or
//              bf16, rounded to nearest even, when the caller asks for bf16 output);
//              tile i's epilogue overlaps tile i + 1's main loop (the second accumulator).
// Tiles run n-fastest so that a 128-row slab of x is reused from L2 by every n tile while
// W stays L2-resident. Out-of-range rows and the K tail are zero-filled by TMA and
// masked on store. Every wait is bounded; one that gives up sets bit 1 of the status word
// (kda_read_device_flags) and the kernel drains.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "kda_internal.h"

namespace kda {

__device__ unsigned int g_gemm_flags;  // bit 1: a GEMM pipeline wait exceeded its limit

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2, STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr long long kWaitLimit = 4000000000LL;  // cycles (~2 s)
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024;  // + alignment slack for 1024-B tiles

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t a, uint32_t c) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(c));
}
__device__ __forceinline__ void mbar_arrive(uint32_t a) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t a, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes)
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
// Bounded wait; false when this or another wait of the grid gave up.
__device__ bool mbar_wait(uint32_t a, uint32_t parity) {
    if (mbar_try(a, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try(a, parity)) return true;
        if ((it & 63u) == 0) {
            if (*(volatile unsigned int *)&g_gemm_flags != 0u) return false;
            if (clock64() - t0 > kWaitLimit) {
                atomicOr(&g_gemm_flags, 2u);
                return false;
            }
        }
    }
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *m, int x, int y,
                                            uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(m), "r"(x), "r"(y), "r"(mbar) : "memory");
}
// Shared-memory matrix descriptor of a K-major tile written by TMA with 128-byte swizzle:
// start address, 8-row groups 1024 bytes apart, descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t addr) {
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B (both K-major), N, M.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);
__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, "
        "%3, p; }" ::"r"(d), "l"(a), "l"(b), "r"(kIdesc), "r"(acc));
}
__device__ __forceinline__ void commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(mbar) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t ta, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(ta));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

template <typename OutT>
__device__ __forceinline__ void store_row32(OutT *dst, const uint32_t (&r)[32], const float *bias, int col0,
                                            int N);
// 32 consecutive outputs of one row: + bias, fp32
template <>
__device__ __forceinline__ void store_row32<float>(float *dst, const uint32_t (&r)[32], const float *bias,
                                                   int col0, int N) {
    if (col0 + 32 <= N && (N & 3) == 0) {
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            float4 v = make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]), __uint_as_float(r[j + 2]),
                                   __uint_as_float(r[j + 3]));
            if (bias) {
                v.x += bias[col0 + j];
                v.y += bias[col0 + j + 1];
                v.z += bias[col0 + j + 2];
                v.w += bias[col0 + j + 3];
            }
            *reinterpret_cast<float4 *>(dst + j) = v;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (col0 + j < N) dst[j] = __uint_as_float(r[j]) + (bias ? bias[col0 + j] : 0.f);
    }
}
// the same rounded to bf16 (nearest even) after the bias is added in fp32
template <>
__device__ __forceinline__ void store_row32<__nv_bfloat16>(__nv_bfloat16 *dst, const uint32_t (&r)[32],
                                                           const float *bias, int col0, int N) {
    auto val = [&](int j) { return __uint_as_float(r[j]) + (bias ? bias[col0 + j] : 0.f); };
    if (col0 + 32 <= N && (N & 7) == 0) {
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                __nv_bfloat162 p2 = __floats2bfloat162_rn(val(j + 2 * h), val(j + 2 * h + 1));
                w[h] = *reinterpret_cast<uint32_t *>(&p2);
            }
            *reinterpret_cast<uint4 *>(dst + j) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (col0 + j < N) dst[j] = __float2bfloat16_rn(val(j));
    }
}

template <typename OutT>
__global__ void __launch_bounds__(kThreads, 1)
    gate_proj_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                     const float *__restrict__ bias, OutT *__restrict__ out, int M, int N, int K) {
    extern __shared__ unsigned char smraw[];
    __shared__ __align__(8) unsigned long long bars[2 * STAGES + 5];
    __shared__ uint32_t tmem_base;
    unsigned char *sm = reinterpret_cast<unsigned char *>(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto full = [&](int s) { return smem_u32(&bars[s]); };
    auto empty = [&](int s) { return smem_u32(&bars[STAGES + s]); };
    auto tfull = [&](int b) { return smem_u32(&bars[2 * STAGES + b]); };
    auto tempty = [&](int b) { return smem_u32(&bars[2 * STAGES + 2 + b]); };
    const uint32_t drained = smem_u32(&bars[2 * STAGES + 4]);
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull(b), 1);
            mbar_init(tempty(b), 4);  // one arrival per epilogue warp
        }
        mbar_init(drained, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&tmem_base)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    const int m_tiles = (M + BM - 1) / BM, n_tiles = (N + BN - 1) / BN;
    const int tiles = m_tiles * n_tiles, kblocks = (K + BK - 1) / BK;
    const uint32_t sbase = smem_u32(sm);

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
                const int m0 = (t / n_tiles) * BM, n0 = (t % n_tiles) * BN;
                bool ok = true;
                for (int kb = 0; kb < kblocks && ok; ++kb) {
                    ok = mbar_wait(empty(s), ph ^ 1);
                    if (!ok) break;
                    mbar_arrive_tx(full(s), STAGE_BYTES);
                    const uint32_t a_s = sbase + s * STAGE_BYTES;
                    tma_load_2d(a_s, &tm_x, kb * BK, m0, full(s));
                    tma_load_2d(a_s + A_BYTES, &tm_w, kb * BK, n0, full(s));
                    if (++s == STAGES) { s = 0; ph ^= 1; }
                }
                if (!ok) break;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int it = 0;
            for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
                const int b = it & 1;
                if (!mbar_wait(tempty(b), ((it >> 1) & 1) ^ 1)) break;  // accumulator b drained
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(b * BN);
                bool ok = true;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!(ok = mbar_wait(full(s), ph))) break;
                    tc_fence_after();
                    const uint32_t a_s = sbase + s * STAGE_BYTES, b_s = a_s + A_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)  // 16 bf16 = 32 bytes along the swizzled row
                        mma_bf16(d, sdesc_sw128(a_s + 32 * k), sdesc_sw128(b_s + 32 * k),
                                 (kb | k) != 0);
                    commit(empty(s));  // the stage is free once these products have read it
                    if (++s == STAGES) { s = 0; ph ^= 1; }
                }
                if (!ok) break;
                commit(tfull(b));      // the tile's accumulator is complete
            }
            // every product issued has completed before the tensor memory is released
            commit(drained);
            mbar_wait(drained, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;  // tensor-memory lane quarter of this warp
        int it = 0;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
            const int b = it & 1;
            const bool ok = mbar_wait(tfull(b), (it >> 1) & 1);
            if (__any_sync(0xffffffffu, !ok)) break;
            tc_fence_after();
            const int m0 = (t / n_tiles) * BM, n0 = (t % n_tiles) * BN;
            const int row = m0 + q * 32 + lane;
            const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN);
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(ta + c * 32, r);
                const int col0 = n0 + c * 32;
                if (row < M) store_row32<OutT>(out + (size_t)row * N + col0, r, bias, col0, N);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty(b));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// [rows][K] bf16 row-major, boxes of box_rows x 64, 128-byte swizzle, zero fill outside
bool encode_kmajor(CUtensorMap *m, const void *base, int rows, int K, int box_rows) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

template <typename OutT>
cudaError_t launch_gate_proj_t(const void *x, const void *w, const float *bias, OutT *out, int M, int N,
                               int K, cudaStream_t stream) {
    if (M == 0 || N == 0) return cudaSuccess;
    CUtensorMap mx, mw;
    if (!encode_kmajor(&mx, x, M, K, BM) || !encode_kmajor(&mw, w, N, K, BN))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gate_proj_kernel<OutT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    const int tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const int grid = tiles < sms ? tiles : sms;
    gate_proj_kernel<OutT><<<grid, kThreads, SMEM_BYTES, stream>>>(mx, mw, bias, out, M, N, K);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

cudaError_t launch_gate_proj(const void *x, const void *w, const float *bias, float *out, int M,
                             int N, int K, cudaStream_t stream) {
    return launch_gate_proj_t<float>(x, w, bias, out, M, N, K, stream);
}

cudaError_t launch_gate_proj_bf16(const void *x, const void *w, const float *bias, void *out, int M,
                                  int N, int K, cudaStream_t stream) {
    return launch_gate_proj_t<__nv_bfloat16>(x, w, bias, static_cast<__nv_bfloat16 *>(out), M, N, K, stream);
}

cudaError_t read_gemm_flags(unsigned int *flags, bool reset, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(flags, g_gemm_flags, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    if (reset) {
        static const unsigned int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_gemm_flags, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                                    stream);
        if (e != cudaSuccess) return e;
    }
    return cudaStreamSynchronize(stream);
}

}  // namespace kda
