// varlen.cu -- packed variable-length batches.  Sequence s occupies rows
// cu[s] .. cu[s+1]-1 of the packed tensors [total, H, ...].  For the tensor-core
// kernels, which read and write the packed tensors in place: the chunk offsets
// of the flat layout and each chunk's first packed row and length.  For the
// other shapes: gather copies the sequences into the padded layout [S, T, H, ...]
// the chunk kernels run on, filling rows t >= len_s with a pad value (zeros for
// q, k, v, dO; alpha = 1 and beta = 0, which leave the state unchanged), and
// scatter copies the padded results back.
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

// ------------------------------------------------ flat chunk layout (SeqMap)
// chunk_off[s] = sum over j < s of ceil(len_j / C), capped at nc_max.  One block;
// thread i sums a contiguous run of sequences, then the block scans the sums.
// order (when not NULL) lists the sequences by chunk count, longest first (ties by
// index), when S <= 1024 (each thread ranks its sequence against all others), and
// 0 .. S-1 otherwise.
__global__ void offsets_kernel(int S, int64_t total, int max_len, int C, int nc_max, const int32_t* __restrict__ cu,
                               int* __restrict__ chunk_off, int* __restrict__ order, int* err) {
    __shared__ int64_t part[1024];
    __shared__ int cnt[1024];
    const int tid = threadIdx.x, nt = blockDim.x;
    const int per = (S + nt - 1) / nt;
    const int s0 = min(S, tid * per), s1 = min(S, s0 + per);
    int64_t sum = 0;
    for (int s = s0; s < s1; ++s) {
        int64_t start;
        int len;
        seq_span(cu, s, total, max_len, start, len, err);
        sum += (len + C - 1) / C;
    }
    part[tid] = sum;
    __syncthreads();
    for (int off = 1; off < nt; off <<= 1) {  // inclusive scan (Hillis-Steele)
        const int64_t x = tid >= off ? part[tid - off] : 0;
        __syncthreads();
        part[tid] += x;
        __syncthreads();
    }
    int64_t run = tid ? part[tid - 1] : 0;
    for (int s = s0; s < s1; ++s) {
        const int a = (int)min(run, (int64_t)nc_max);
        chunk_off[s] = a;
        int64_t start;
        int len;
        seq_span(cu, s, total, max_len, start, len, nullptr);
        run += (len + C - 1) / C;
        if (S <= 1024) cnt[s] = (int)min(run, (int64_t)nc_max) - a;  // chunks of s as laid out
    }
    if (tid == nt - 1) {
        chunk_off[S] = (int)min(part[nt - 1], (int64_t)nc_max);
        if (part[nt - 1] > nc_max || cu[0] != 0 || (int64_t)cu[S] != total) atomicOr(err, kVarlenBadOffsets);
    }
    if (!order) return;
    if (S > 1024) {
        for (int s = tid; s < S; s += nt) order[s] = s;
        return;
    }
    __syncthreads();
    if (tid < S) {  // one sequence per thread (nt >= S)
        const int n = cnt[tid];
        int rank = 0;
        for (int j = 0; j < S; ++j) rank += (cnt[j] > n) || (cnt[j] == n && j < tid);
        order[rank] = tid;
    }
}

// Rows of sequence s that reach the flat layout: its length, cut to its chunks.
__device__ __forceinline__ int flat_len(const int32_t* cu, const int* chunk_off, int s, int64_t total, int C,
                                        int64_t& start) {
    int len;
    seq_span(cu, s, total, 0x7fffffff, start, len, nullptr);
    return (int)min((int64_t)len, (int64_t)(chunk_off[s + 1] - chunk_off[s]) * C);
}

// Largest s in [0, n) with a[s] <= x (a non-decreasing; 0 if none).
__device__ __forceinline__ int last_le(const int* a, int n, int64_t x) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)a[mid] <= x) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// tok[c] / len[c] for flat chunk c: the sequence s owning it (chunk_off[s] <= c <
// chunk_off[s+1]) starts at packed row start_s, so chunk j = c - chunk_off[s] of it
// starts at start_s + j*C with min(C, len_s - j*C) tokens.  Chunks past the last
// sequence get tok 0, len 0.
__global__ void chunk_tokens_kernel(int S, int64_t total, int C, int nc_max, const int32_t* __restrict__ cu,
                                    const int* __restrict__ chunk_off, int* __restrict__ tok, int* __restrict__ len) {
    for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < nc_max; c += gridDim.x * blockDim.x) {
        int t = 0, n = 0;
        if (S > 0 && c < chunk_off[S]) {
            const int s = last_le(chunk_off, S, c);
            int64_t start;
            const int ls = flat_len(cu, chunk_off, s, total, C, start);
            const int j = c - chunk_off[s];
            n = (int)max((int64_t)0, min((int64_t)C, (int64_t)ls - (int64_t)j * C));
            t = n > 0 ? (int)(start + (int64_t)j * C) : 0;
        }
        tok[c] = t;
        len[c] = n;
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

cudaError_t launch_varlen_offsets(int S, int64_t total, int max_len, int C, int nc_max, const int32_t* cu,
                                  int* chunk_off, int* order, int* err, cudaStream_t st) {
    int nt = 32;  // a power of two for the block scan
    while (nt < 1024 && nt < S) nt <<= 1;
    offsets_kernel<<<1, nt, 0, st>>>(S, total, max_len, C, nc_max, cu, chunk_off, order, err);
    return cudaGetLastError();
}

cudaError_t launch_varlen_chunk_tokens(int S, int64_t total, int C, int nc_max, const int32_t* cu,
                                       const int* chunk_off, int* tok, int* len, cudaStream_t st) {
    if (nc_max <= 0) return cudaSuccess;
    const int grid = (nc_max + 255) / 256;
    chunk_tokens_kernel<<<grid < 1024 ? grid : 1024, 256, 0, st>>>(S, total, C, nc_max, cu, chunk_off, tok, len);
    return cudaGetLastError();
}

}  // namespace gdn
