// check.cu -- counting the non-finite elements (NaN, +-inf) of a device tensor,
// a device-side check of inputs or results whose answer the caller reads after a
// stream synchronisation: the count is added to a caller-supplied integer in
// device memory, so nothing here waits, traps or asserts.

#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

__device__ __forceinline__ int bad(float x) { return isfinite(x) ? 0 : 1; }
__device__ __forceinline__ int bad_bf16_pair(uint32_t w) {
    return bad(__uint_as_float(w << 16)) + bad(__uint_as_float(w & 0xffff0000u));
}

// 16-byte vectors over the first n - n % per elements, then the tail; one atomic
// per warp whose lanes saw any non-finite element.
template <typename T>
__global__ void __launch_bounds__(256) count_nonfinite_kernel(const T* __restrict__ x, int64_t n,
                                                                unsigned long long* count) {
    constexpr int per = 16 / (int)sizeof(T);
    const int64_t nv = n / per;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int local = 0;
    for (int64_t i = i0; i < nv; i += stride) {
        const uint4 w = ((const uint4*)x)[i];
        if constexpr (sizeof(T) == 4) {
            local += bad(__uint_as_float(w.x)) + bad(__uint_as_float(w.y)) + bad(__uint_as_float(w.z)) +
                     bad(__uint_as_float(w.w));
        } else {
            local += bad_bf16_pair(w.x) + bad_bf16_pair(w.y) + bad_bf16_pair(w.z) + bad_bf16_pair(w.w);
        }
    }
    for (int64_t i = nv * per + i0; i < n; i += stride) {
        if constexpr (sizeof(T) == 4) local += bad(((const float*)x)[i]);
        else local += bad(__bfloat162float(((const __nv_bfloat16*)x)[i]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) local += __shfl_xor_sync(0xffffffffu, local, off);
    if ((threadIdx.x & 31) == 0 && local) atomicAdd(count, (unsigned long long)local);
}

}  // namespace

cudaError_t launch_count_nonfinite(const void* x, int64_t n, InType ty, int64_t* count, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    const int64_t per = ty == InType::BF16 ? 8 : 4;
    const int64_t want = (n / per + 255) / 256 + 1;
    const unsigned grid = (unsigned)(want < (int64_t)sm_count() * 4 ? want : (int64_t)sm_count() * 4);
    unsigned long long* c = (unsigned long long*)count;
    if (ty == InType::BF16)
        count_nonfinite_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>((const __nv_bfloat16*)x, n, c);
    else
        count_nonfinite_kernel<float><<<grid, 256, 0, st>>>((const float*)x, n, c);
    return cudaGetLastError();
}

}  // namespace gdn
