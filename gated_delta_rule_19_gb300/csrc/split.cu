// split.cu -- the within-call sequence split (two-level scan) of the chunk scans.
//
// Over one chunk the state map is affine ("Sparse Delta Memory: layer and
// kernels", What the layer computes: Phase 2 applies the corrected writes to the
// chunk-start state; "OpenGDN", Core operator reference: the 64-token chunk form):
//     S1^T = A_c S0^T + B_c,   A_c = gamma_C I - K^T diag(e) W,   B_c = K^T diag(e) U~,
// so a run of chunks (a piece) maps S_in to S_out = S_in P^T + R, with P the
// product of its A_c and R its final state from a zero start.  The forward scan
// computes R (zero start) and P^T (start I, U~ read as 0) for every piece in
// parallel; combine_fwd chains the pieces of a sequence,
//     S_in(j+1) = S_in(j) P_j^T + R_j,
// and a second scan runs every piece from its S_in.  The reverse scan's map is
// the transpose: dS_in = dS_out P + D, D the piece's dS_in from a zero dS_out;
// combine_bwd chains those from the last piece back.
//
// States are [V, K] fp32 (V = K = 128 on the tensor-core path), slot
// (s*P + j)*H + h for piece j of sequence s; combine kernels run 16 rows of one
// (sequence, head) per CTA, rows being independent.

#include <cuda_runtime.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kN = 128;    // K = V on the tensor-core path
constexpr int kRows = 16;  // state rows per CTA
constexpr int kTS = kN + 1;  // padded row of the staged transition

// piece_off[s*P + j] = first chunk of piece j of sequence s: its chunks
// [base_s, base_s + n_s) cut into P runs of floor sizes.  base/n from chunk_off
// (packed sequences) or base_s = s*nc, n_s = nc (dense rows of nc chunks).
__global__ void pieces_kernel(int S, int P, int nc, const int* __restrict__ chunk_off, int* __restrict__ piece_off) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i <= S * P; i += gridDim.x * blockDim.x) {
        const int s = i / P, j = i % P;
        if (s == S) {
            piece_off[i] = chunk_off ? chunk_off[S] : S * nc;
            continue;
        }
        const int base = chunk_off ? chunk_off[s] : s * nc;
        const int n = chunk_off ? chunk_off[s + 1] - base : nc;
        piece_off[i] = base + (int)(((int64_t)j * n) / P);
    }
}

// Forward chain: thread (column k = tid & 127, rows 8*(tid >> 7) ..) of the CTA's
// 16 rows; trans is read straight from global memory (coalesced along k).
__global__ void __launch_bounds__(256) combine_fwd_kernel(int P, int H, const float* __restrict__ s0,
                                                          const float* __restrict__ R,
                                                          const float* __restrict__ trans, float* __restrict__ s_in,
                                                          float* __restrict__ sT) {
    __shared__ float cur[kRows][kN];
    const int rb = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
    const int tid = threadIdx.x, k = tid & (kN - 1), r0 = (tid >> 7) * 8;
    const int64_t seq_slot = (int64_t)s * H + h;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int v = rb * kRows + r0 + i;
        cur[r0 + i][k] = s0 ? s0[(seq_slot * kN + v) * kN + k] : 0.f;
    }
    __syncthreads();
    for (int j = 0; j < P; ++j) {
        const int64_t slot = ((int64_t)s * P + j) * H + h;
        const float* tj = trans + slot * kN * kN;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int v = rb * kRows + r0 + i;
            s_in[(slot * kN + v) * kN + k] = cur[r0 + i][k];
            acc[i] = R[(slot * kN + v) * kN + k];
        }
#pragma unroll 4
        for (int m = 0; m < kN; ++m) {
            const float t = tj[m * kN + k];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fmaf(cur[r0 + i][m], t, acc[i]);
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 8; ++i) cur[r0 + i][k] = acc[i];
        __syncthreads();
    }
    if (sT) {
#pragma unroll
        for (int i = 0; i < 8; ++i) sT[(seq_slot * kN + rb * kRows + r0 + i) * kN + k] = cur[r0 + i][k];
    }
}

// Reverse chain: G <- G P_j + D_j from the last piece back, P_j[m][k] =
// trans_j[k][m]; trans_j is staged transposed (padded rows) per piece.
__global__ void __launch_bounds__(256) combine_bwd_kernel(int P, int H, const float* __restrict__ dsT,
                                                          const float* __restrict__ D,
                                                          const float* __restrict__ trans,
                                                          float* __restrict__ ds_out, float* __restrict__ ds0) {
    extern __shared__ float smf[];
    float* tt = smf;               // [kN][kTS]: tt[m][k] = trans_j[k][m]
    float* cur = smf + kN * kTS;   // [kRows][kN]
    const int rb = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
    const int tid = threadIdx.x, k = tid & (kN - 1), r0 = (tid >> 7) * 8;
    const int64_t seq_slot = (int64_t)s * H + h;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int v = rb * kRows + r0 + i;
        cur[(r0 + i) * kN + k] = dsT ? dsT[(seq_slot * kN + v) * kN + k] : 0.f;
    }
    for (int j = P - 1; j >= 0; --j) {
        const int64_t slot = ((int64_t)s * P + j) * H + h;
        const float* tj = trans + slot * kN * kN;
        for (int e = tid; e < kN * kN; e += blockDim.x) {  // read rows of trans_j, write columns of tt
            const int row = e / kN, col = e % kN;
            tt[col * kTS + row] = tj[e];
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int v = rb * kRows + r0 + i;
            ds_out[(slot * kN + v) * kN + k] = cur[(r0 + i) * kN + k];
            acc[i] = D[(slot * kN + v) * kN + k];
        }
#pragma unroll 4
        for (int m = 0; m < kN; ++m) {
            const float p = tt[m * kTS + k];  // P_j[m][k]
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fmaf(cur[(r0 + i) * kN + m], p, acc[i]);
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 8; ++i) cur[(r0 + i) * kN + k] = acc[i];
        __syncthreads();
    }
    if (ds0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) ds0[(seq_slot * kN + rb * kRows + r0 + i) * kN + k] = cur[(r0 + i) * kN + k];
    }
}

}  // namespace

cudaError_t launch_split_pieces(int S, int P, int nc, const int* chunk_off, int* piece_off, cudaStream_t st) {
    const int n = S * P + 1;
    pieces_kernel<<<(n + 255) / 256, 256, 0, st>>>(S, P, nc, chunk_off, piece_off);
    return cudaGetLastError();
}

cudaError_t launch_combine_fwd(int S, int P, int H, const float* s0, const float* R, const float* trans, float* s_in,
                               float* sT, cudaStream_t st) {
    if (S * H == 0) return cudaSuccess;
    combine_fwd_kernel<<<dim3(kN / kRows, H, S), 256, 0, st>>>(P, H, s0, R, trans, s_in, sT);
    return cudaGetLastError();
}

cudaError_t launch_combine_bwd(int S, int P, int H, const float* dsT, const float* D, const float* trans,
                               float* ds_out, float* ds0, cudaStream_t st) {
    if (S * H == 0) return cudaSuccess;
    const int smem = (kN * kTS + kRows * kN) * (int)sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(combine_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    combine_bwd_kernel<<<dim3(kN / kRows, H, S), 256, smem, st>>>(P, H, dsT, D, trans, ds_out, ds0);
    return cudaGetLastError();
}

}  // namespace gdn
