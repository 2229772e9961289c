// reset.cu -- dense batches whose streams restart from the zero state at marked
// positions ("OpenGDN", Scope, lists reset masks among the features it does not
// support; no page gives a formula).  A reset at (b, t) clears the state just
// before token t: the stream continues from the zero state at t, which is the
// recurrence with alpha_t = 0.  Every row of the batch is then a run of segments
// that start at t = 0 or at a reset; laid back to back in the row-major token
// order they are a packed batch over the B*T tokens, whose sequences the varlen
// kernels run independently.  The kernels here build that segmentation from the
// device mask and route the states between rows and segments, so no step needs
// the number of segments on the host: the caller gives an upper bound.

#include <cuda_runtime.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kSegThreads = 1024;

// One block.  Token i = b*T + t starts a segment when t == 0 or reset[i] != 0.
// Writes, for S segments and the bound S_max:
//   cu[s]        start token of segment s (s < min(S, S_max)); B*T for the rest
//                up to cu[S_max], so segments past S are empty;
//   in_map[s]    the row whose initial state segment s starts from, or -1 (a
//                row's first segment, unless the row resets at t = 0);
//   fin_map[s]   the row whose final state segment s ends with, or -1;
//   last[b]      row b's last segment;  first_carry[b]  row b's first segment
//                if its initial state carries into it, else -1;
//   *err         kResetTooManySegments if S > S_max (segments past the bound
//                then merge into the last one: the results are not valid).
__global__ void __launch_bounds__(kSegThreads)
segments_kernel(int B, int T, const uint8_t* __restrict__ reset, int S_max, int32_t* __restrict__ cu,
                int32_t* __restrict__ in_map, int32_t* __restrict__ fin_map, int32_t* __restrict__ last,
                int32_t* __restrict__ first_carry, int* __restrict__ err) {
    __shared__ int wsum[kSegThreads / 32];
    __shared__ int total_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t N = (int64_t)B * T;
    const int64_t per = (N + kSegThreads - 1) / kSegThreads;
    const int64_t lo = (int64_t)tid * per, hi = lo + per < N ? lo + per : N;
    auto starts = [&](int64_t i) { return (i % T) == 0 || reset[i] != 0; };
    for (int s = tid; s < S_max; s += kSegThreads) {
        in_map[s] = -1;
        fin_map[s] = -1;
    }
    int cnt = 0;
    for (int64_t i = lo; i < hi; ++i) cnt += starts(i) ? 1 : 0;
    // exclusive scan of the per-thread counts
    int incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = wsum[lane];
        int wi = w;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += y;
        }
        wsum[lane] = wi - w;  // exclusive over warps
        if (lane == 31) total_s = wi;
    }
    __syncthreads();  // in_map / fin_map cleared, the scan done
    int s = wsum[warp] + incl - cnt;
    for (int64_t i = lo; i < hi; ++i) {
        if (!starts(i)) continue;
        if (s < S_max) {
            cu[s] = (int32_t)i;
            if (i % T == 0) {
                const int b = (int)(i / T);
                const bool carry = reset[i] == 0;
                first_carry[b] = carry ? s : -1;
                if (carry) in_map[s] = b;
            }
        } else if (i % T == 0) {
            first_carry[(int)(i / T)] = -1;
        }
        ++s;
    }
    __syncthreads();
    const int S = total_s;
    const int Sc = S < S_max ? S : S_max;
    for (int j = Sc + tid; j <= S_max; j += kSegThreads) cu[j] = (int32_t)N;
    if (tid == 0 && S > S_max) atomicOr(err, kResetTooManySegments);
    // row b's last segment: the one before row b+1's first (the scan order is row-major)
    for (int b = tid; b < B; b += kSegThreads) {
        int nb;  // first segment of row b + 1 (or S)
        if (b + 1 < B) {
            // count of starts before token (b+1)*T: recompute from cu by binary search
            int l = 0, h = Sc;
            const int64_t key = (int64_t)(b + 1) * T;
            while (l < h) {
                const int m = (l + h) >> 1;
                if ((int64_t)cu[m] < key) l = m + 1;
                else h = m;
            }
            nb = l;
        } else {
            nb = Sc;
        }
        const int lb = nb - 1 < 0 ? 0 : nb - 1;
        last[b] = lb;
        fin_map[lb] = b;
    }
}

// out[r, :] = src[map[r], :] (map[r] < 0 or src NULL: zeros), rows of `row` floats;
// block 0 also ORs *merge_from into *merge_to (after the varlen call).
__global__ void route_kernel(int nrows, int64_t row, const int32_t* __restrict__ map, const float* __restrict__ src,
                             float* __restrict__ out, const int* merge_from, int* merge_to) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && merge_from && merge_to) atomicOr(merge_to, *merge_from);
    const int64_t n4 = (int64_t)nrows * row / 4;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t e = i * 4;
        const int r = (int)(e / row);
        const int m = map[r];
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (m >= 0 && src) v = *(const float4*)(src + (int64_t)m * row + (e - (int64_t)r * row));
        *(float4*)(out + e) = v;
    }
}

}  // namespace

cudaError_t launch_reset_segments(int B, int T, const uint8_t* reset, int S_max, int32_t* cu, int32_t* in_map,
                                  int32_t* fin_map, int32_t* last, int32_t* first_carry, int* err,
                                  cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(err, 0, sizeof(int), st);
    if (e != cudaSuccess) return e;
    segments_kernel<<<1, kSegThreads, 0, st>>>(B, T, reset, S_max, cu, in_map, fin_map, last, first_carry, err);
    return cudaGetLastError();
}

cudaError_t launch_route_states(int nrows, int64_t row, const int32_t* map, const float* src, float* out,
                                const int* merge_from, int* merge_to, cudaStream_t st) {
    const int64_t n4 = (int64_t)nrows * row / 4;
    const int64_t blocks = (n4 + 255) / 256;
    const int grid = (int)(blocks < 1 ? 1 : (blocks > 4 * sm_count() ? 4 * sm_count() : blocks));
    route_kernel<<<grid, 256, 0, st>>>(nrows, row, map, src, out, merge_from, merge_to);
    return cudaGetLastError();
}

}  // namespace gdn
