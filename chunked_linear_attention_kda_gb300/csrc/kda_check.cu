// kda_check.cu -- device-side input and output checks: the layout rules of cu_seqlens
// and a count of non-finite values (the NaN/Inf monitoring the bounded gate is meant to
// make unnecessary: "Demystifying Trillion-Parameter MoE Models", Verification). Both
// only read their inputs and write a caller-provided result word; neither traps.
#include <cuda_bf16.h>

#include "kda_internal.h"

namespace kda {
namespace {

// status[0] |= bit 0: cu[0] != 0; bit 1: cu[i + 1] < cu[i] for some i; bit 2:
// cu[n_seq] != n_tok. status[1] = min over the offending i (the pair i, i + 1 for bit 1;
// 0 for bit 0; n_seq for bit 2); status[1] must start at INT32_MAX.
__global__ void validate_cu_kernel(const int32_t *__restrict__ cu, int32_t n_seq, int64_t n_tok,
                                   int32_t *__restrict__ status) {
    unsigned int bits = 0;
    int first = 0x7fffffff;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_seq;
         i += (int64_t)gridDim.x * blockDim.x) {
        if (cu[i + 1] < cu[i]) {
            bits |= 2u;
            first = min(first, (int)i);
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (cu[0] != 0) {
            bits |= 1u;
            first = 0;
        }
        if ((int64_t)cu[n_seq] != n_tok) {
            bits |= 4u;
            first = min(first, n_seq);
        }
    }
    if (bits) {
        atomicOr(reinterpret_cast<unsigned int *>(status), bits);
        atomicMin(status + 1, first);
    }
}

__global__ void init_status_kernel(int32_t *status) {
    status[0] = 0;
    status[1] = 0x7fffffff;
}

template <typename T>
__device__ __forceinline__ float as_f32(T x);
template <>
__device__ __forceinline__ float as_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float as_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__global__ void count_nonfinite_kernel(const T *__restrict__ x, int64_t n,
                                       unsigned long long *__restrict__ count) {
    unsigned int local = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        local += isfinite(as_f32(x[i])) ? 0u : 1u;
    // one atomic per warp
    for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(0xffffffffu, local, o);
    if ((threadIdx.x & 31) == 0 && local) atomicAdd(count, (unsigned long long)local);
}

int grid_for(int64_t n, int threads) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (n + threads - 1) / threads;
    const int64_t cap = (int64_t)sms * 8;
    return (int)(want < 1 ? 1 : (want > cap ? cap : want));
}

}  // namespace

cudaError_t launch_validate_cu(const int32_t *cu, int32_t n_seq, int64_t n_tok, int32_t *status,
                               cudaStream_t stream) {
    init_status_kernel<<<1, 1, 0, stream>>>(status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    validate_cu_kernel<<<grid_for(n_seq > 0 ? n_seq : 1, 256), 256, 0, stream>>>(cu, n_seq, n_tok,
                                                                                status);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(2);
    return e;
}

cudaError_t launch_count_nonfinite(const void *x, int64_t n, bool bf16, unsigned long long *count,
                                   cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const int g = grid_for(n, 256);
    if (bf16)
        count_nonfinite_kernel<<<g, 256, 0, stream>>>(static_cast<const __nv_bfloat16 *>(x), n, count);
    else
        count_nonfinite_kernel<<<g, 256, 0, stream>>>(static_cast<const float *>(x), n, count);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

}  // namespace kda
