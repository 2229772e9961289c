// varlen.cu -- packed variable-length batches.  Sequence s occupies rows
// cu[s] .. cu[s+1]-1 of the packed tensors [total, H, ...]; gather copies them
// into the padded layout [S, T, H, ...] the chunk kernels run on, filling rows
// t >= len_s with a pad value (zeros for q, k, v, dO; alpha = 1 and beta = 0,
// which leave the state unchanged), and scatter copies the padded results back.
// cu is read on the device: an offset outside [0, total], a decreasing pair, or a
// length above T marks the sequence as empty and sets kVarlenBadOffsets in the
// error word, so no access leaves the buffers.

#include <cuda_runtime.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

// Start and length of sequence s, clamped so that a bad cu never leads out of
// bounds (the sequence then counts as empty and the error bit is set).
__device__ __forceinline__ void seq_span(const int32_t* cu, int s, int64_t total, int T, int64_t& start, int& len,
                                         int* err) {
    const int64_t a = cu[s], e = cu[s + 1];
    if (a < 0 || e < a || e > total || e - a > T) {
        if (err) atomicOr(err, kVarlenBadOffsets);
        start = 0;
        len = 0;
        return;
    }
    start = a;
    len = (int)(e - a);
}

// Rows of `w16` 16-byte words: packed [total, H, w16] <-> padded [S, T, H, w16].
// dir 0: gather (padded rows t >= len get `fill`); dir 1: scatter (rows t < len).
__global__ void rows16_kernel(int S, int T, int H, int w16, int64_t total, const int32_t* __restrict__ cu,
                              const uint4* __restrict__ src, uint4* __restrict__ dst, uint32_t fill, int dir,
                              int* err, const int* merge) {
    const int64_t n = (int64_t)S * T * H * w16;
    if (blockIdx.x == 0 && threadIdx.x == 0 && err) {
        // the sequences must tile the packed rows exactly
        if (cu[0] != 0 || (int64_t)cu[S] != total) atomicOr(err, kVarlenBadOffsets);
        if (merge) atomicOr(err, *merge);  // the chunk kernels' error word, after they ran
    }
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int j = (int)(i % w16);
        const int64_t row = i / w16;  // (s, t, h)
        const int h = (int)(row % H);
        const int t = (int)((row / H) % T);
        const int s = (int)(row / ((int64_t)H * T));
        int64_t start;
        int len;
        seq_span(cu, s, total, T, start, len, (t == 0 && h == 0 && j == 0) ? err : nullptr);
        const int64_t prow = ((start + t) * H + h) * w16 + j;
        if (dir == 0) {
            dst[i] = t < len ? src[prow] : make_uint4(fill, fill, fill, fill);
        } else if (t < len) {
            dst[prow] = src[i];
        }
    }
}

// The same for rows of one 2- or 4-byte element (alpha, beta and their gradients).
template <typename U>
__global__ void elems_kernel(int S, int T, int H, int64_t total, const int32_t* __restrict__ cu,
                             const U* __restrict__ src, U* __restrict__ dst, U fill, int dir, int* err) {
    const int64_t n = (int64_t)S * T * H;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int h = (int)(i % H);
        const int t = (int)((i / H) % T);
        const int s = (int)(i / ((int64_t)H * T));
        int64_t start;
        int len;
        seq_span(cu, s, total, T, start, len, (t == 0 && h == 0) ? err : nullptr);
        const int64_t p = (start + t) * H + h;
        if (dir == 0) {
            dst[i] = t < len ? src[p] : fill;
        } else if (t < len) {
            dst[p] = src[i];
        }
    }
}

unsigned grid_for(int64_t n) {
    const int64_t want = (n + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 16;
    return (unsigned)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_varlen_rows(const Dims& d, int64_t total, const int32_t* cu, int width_bytes, const void* src,
                               void* dst, uint32_t fill, bool scatter, int* err, const int* merge, cudaStream_t st) {
    const int w16 = width_bytes / 16;
    const int64_t n = (int64_t)d.B * d.T * d.H * w16;
    if (n == 0) return cudaSuccess;
    rows16_kernel<<<grid_for(n), 256, 0, st>>>(d.B, d.T, d.H, w16, total, cu, (const uint4*)src, (uint4*)dst, fill,
                                               scatter ? 1 : 0, err, merge);
    return cudaGetLastError();
}

cudaError_t launch_varlen_elems(const Dims& d, int64_t total, const int32_t* cu, int elem_bytes, const void* src,
                                void* dst, uint32_t fill, bool scatter, int* err, cudaStream_t st) {
    const int64_t n = (int64_t)d.B * d.T * d.H;
    if (n == 0) return cudaSuccess;
    if (elem_bytes == 2)
        elems_kernel<uint16_t><<<grid_for(n), 256, 0, st>>>(d.B, d.T, d.H, total, cu, (const uint16_t*)src,
                                                            (uint16_t*)dst, (uint16_t)fill, scatter ? 1 : 0, err);
    else
        elems_kernel<uint32_t><<<grid_for(n), 256, 0, st>>>(d.B, d.T, d.H, total, cu, (const uint32_t*)src,
                                                            (uint32_t*)dst, fill, scatter ? 1 : 0, err);
    return cudaGetLastError();
}

}  // namespace gdn
