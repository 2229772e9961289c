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
// States are [V, K] fp32 with V = K = 128 (the split runs only for that shape), slot
// (s*P + j)*H + h for piece j of sequence s; combine kernels run 4 rows of one
// (sequence, head) per CTA, rows being independent.

#include <cuda_runtime.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kN = 128;    // K = V
constexpr int kRows = 4;   // state rows per CTA
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

// Forward chain: thread (column k = tid & 127, rows 2*(tid >> 7) ..) of the CTA's
// kRows rows.  trans_j is staged in shared memory per piece; the next piece's is
// read into registers (16 float4 per thread) while this one's products run, so a
// step costs one round trip to L2 instead of one per row of trans_j.  Each output
// sums over m in order, as a plain row-times-matrix product.
__global__ void __launch_bounds__(256) combine_fwd_kernel(int P, int H, const float* __restrict__ s0,
                                                          const float* __restrict__ R,
                                                          const float* __restrict__ trans, float* __restrict__ s_in,
                                                          float* __restrict__ sT) {
    extern __shared__ float smf[];
    float* tt = smf;              // [kN][kN]: trans_j
    float* cur = smf + kN * kN;   // [kRows][kN]
    const int rb = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
    const int tid = threadIdx.x, k = tid & (kN - 1), r0 = (tid >> 7) * 2;
    const int64_t seq_slot = (int64_t)s * H + h;
    float4 pre[16];
    auto load_t = [&](int j) {
        const float4* src = (const float4*)(trans + (((int64_t)s * P + j) * H + h) * kN * kN);
#pragma unroll
        for (int q = 0; q < 16; ++q) pre[q] = src[tid + 256 * q];
    };
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int v = rb * kRows + r0 + i;
        cur[(r0 + i) * kN + k] = s0 ? s0[(seq_slot * kN + v) * kN + k] : 0.f;
    }
    if (P > 0) load_t(0);
    for (int j = 0; j < P; ++j) {
        const int64_t slot = ((int64_t)s * P + j) * H + h;
#pragma unroll
        for (int q = 0; q < 16; ++q) ((float4*)tt)[tid + 256 * q] = pre[q];
        __syncthreads();  // trans_j and the rows of S_in(j) in place
        if (j + 1 < P) load_t(j + 1);
        float acc[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int v = rb * kRows + r0 + i;
            s_in[(slot * kN + v) * kN + k] = cur[(r0 + i) * kN + k];
            acc[i] = R[(slot * kN + v) * kN + k];
        }
#pragma unroll 8
        for (int m = 0; m < kN; ++m) {
            const float t = tt[m * kN + k];
#pragma unroll
            for (int i = 0; i < 2; ++i) acc[i] = fmaf(cur[(r0 + i) * kN + m], t, acc[i]);
        }
        __syncthreads();  // every read of tt and cur done
#pragma unroll
        for (int i = 0; i < 2; ++i) cur[(r0 + i) * kN + k] = acc[i];
    }
    __syncthreads();
    if (sT) {
#pragma unroll
        for (int i = 0; i < 2; ++i) sT[(seq_slot * kN + rb * kRows + r0 + i) * kN + k] = cur[(r0 + i) * kN + k];
    }
}

// Reverse chain: G <- G P_j + D_j from the last piece back, P_j[m][k] =
// trans_j[k][m]; trans_j is staged transposed (padded rows) per piece, the next
// piece's read into registers (coalesced, 64 per thread) during this one's
// products.
__global__ void __launch_bounds__(256) combine_bwd_kernel(int P, int H, const float* __restrict__ dsT,
                                                          const float* __restrict__ D,
                                                          const float* __restrict__ trans,
                                                          float* __restrict__ ds_out, float* __restrict__ ds0) {
    extern __shared__ float smf[];
    float* tt = smf;               // [kN][kTS]: tt[m][k] = trans_j[k][m]
    float* cur = smf + kN * kTS;   // [kRows][kN]
    const int rb = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
    const int tid = threadIdx.x, k = tid & (kN - 1), r0 = (tid >> 7) * 2;
    const int64_t seq_slot = (int64_t)s * H + h;
    float pre[64];
    auto load_t = [&](int j) {
        const float* src = trans + (((int64_t)s * P + j) * H + h) * kN * kN;
#pragma unroll
        for (int q = 0; q < 64; ++q) pre[q] = src[tid + 256 * q];
    };
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int v = rb * kRows + r0 + i;
        cur[(r0 + i) * kN + k] = dsT ? dsT[(seq_slot * kN + v) * kN + k] : 0.f;
    }
    if (P > 0) load_t(P - 1);
    for (int j = P - 1; j >= 0; --j) {
        const int64_t slot = ((int64_t)s * P + j) * H + h;
#pragma unroll
        for (int q = 0; q < 64; ++q) {  // element e = row * kN + col of trans_j -> tt[col][row]
            const int e = tid + 256 * q;
            tt[(e & (kN - 1)) * kTS + (e >> 7)] = pre[q];
        }
        __syncthreads();
        if (j > 0) load_t(j - 1);
        float acc[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int v = rb * kRows + r0 + i;
            ds_out[(slot * kN + v) * kN + k] = cur[(r0 + i) * kN + k];
            acc[i] = D[(slot * kN + v) * kN + k];
        }
#pragma unroll 8
        for (int m = 0; m < kN; ++m) {
            const float p = tt[m * kTS + k];  // P_j[m][k]
#pragma unroll
            for (int i = 0; i < 2; ++i) acc[i] = fmaf(cur[(r0 + i) * kN + m], p, acc[i]);
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 2; ++i) cur[(r0 + i) * kN + k] = acc[i];
    }
    __syncthreads();
    if (ds0) {
#pragma unroll
        for (int i = 0; i < 2; ++i) ds0[(seq_slot * kN + rb * kRows + r0 + i) * kN + k] = cur[(r0 + i) * kN + k];
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
    const int smem = (kN * kN + kRows * kN) * (int)sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(combine_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    combine_fwd_kernel<<<dim3(kN / kRows, H, S), 256, smem, st>>>(P, H, s0, R, trans, s_in, sT);
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
