// decode.cu -- the recurrent step for decoding: a few tokens per call, the state
// read and written once ("OpenGDN", Core operator reference: a stream continued
// exactly through state=; "Sparse Delta Memory: layer and kernels", Execution:
// the single-token call).
//
// Per (b, h) the state S [V, K] advances token by token:
//   S <- alpha S (I - beta k k^T) + beta v k^T = alpha S + beta (v - alpha S k) k^T
//   o  = S q = alpha (S q) + beta (v - alpha S k) (k^T q)
// Row v of S only needs row v, so a warp unit is R rows of one head, kept in
// registers across the call's tokens (lane l holds K/32 consecutive columns), with
// the row dot products S k, S q reduced by butterfly shuffles.  Warps are
// persistent and stream their units' rows in through shared memory ahead of use.
// The kernel is bound by reading and writing the fp32 state once.

#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

__device__ __forceinline__ float ld(const float* p) { return *p; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st(float* p, float x) { *p = x; }
__device__ __forceinline__ void st(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// N consecutive values (N = 1, 2, 4; the address aligned to N elements) as floats.
template <int N>
__device__ __forceinline__ void ldn(const float* p, float* f) {
    if constexpr (N == 4) {
        const float4 x = *(const float4*)p;
        f[0] = x.x, f[1] = x.y, f[2] = x.z, f[3] = x.w;
    } else if constexpr (N == 2) {
        const float2 x = *(const float2*)p;
        f[0] = x.x, f[1] = x.y;
    } else {
        f[0] = *p;
    }
}
template <int N>
__device__ __forceinline__ void ldn(const __nv_bfloat16* p, float* f) {
    if constexpr (N == 4) {
        const uint2 x = *(const uint2*)p;
        f[0] = __uint_as_float(x.x << 16), f[1] = __uint_as_float(x.x & 0xffff0000u);
        f[2] = __uint_as_float(x.y << 16), f[3] = __uint_as_float(x.y & 0xffff0000u);
    } else if constexpr (N == 2) {
        const uint32_t x = *(const uint32_t*)p;
        f[0] = __uint_as_float(x << 16), f[1] = __uint_as_float(x & 0xffff0000u);
    } else {
        f[0] = __bfloat162float(*p);
    }
}
template <int N>
__device__ __forceinline__ void stn(float* p, const float* f) {
    if constexpr (N == 4) {
        *(float4*)p = make_float4(f[0], f[1], f[2], f[3]);
    } else if constexpr (N == 2) {
        *(float2*)p = make_float2(f[0], f[1]);
    } else {
        *p = f[0];
    }
}

constexpr int kRows = 8;    // state rows per warp unit
constexpr int kStages = 3;  // state units in each warp's ring (two in flight while one is used)

// A size-byte (4, 8 or 16) asynchronous copy from global to shared memory.
template <int BYTES>
__device__ __forceinline__ void cp_async(void* dst, const void* src) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
    if constexpr (BYTES == 16)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(d), "l"(src), "n"(BYTES) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Persistent warps: warp w of the grid handles units w, w + W, ... (W warps in the
// grid); unit u is rows v0 .. v0+kRows of head bh = u / (V / kRows).  Lane l holds
// columns [l*KPL, l*KPL + KPL) of each of the unit's rows (K = 32*KPL; for K = 16,
// KPL = 1 and lanes 16-31 hold nothing).  Each warp streams its units' state rows
// through a ring of kStages shared-memory slots with cp.async, two units ahead; a
// lane reads back only the pieces it copied, so its own wait_group orders
// everything and no barrier is needed.
template <typename Tin, int KPL>
__global__ void __launch_bounds__(256, 2)
decode_kernel(Dims d, const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
              const Tin* __restrict__ alpha, const Tin* __restrict__ beta, float* __restrict__ state,
              Tin* __restrict__ o) {
    constexpr int SLOT = kRows * 32 * KPL;  // floats per ring slot
    extern __shared__ __align__(16) float dsm[];
    const int lane = threadIdx.x & 31;
    float* ring = dsm + (threadIdx.x >> 5) * kStages * SLOT;
    const int64_t W = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t w0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int groups = d.V / kRows;
    const int64_t units = (int64_t)d.B * d.H * groups;
    const int K = d.K, V = d.V;
    const int c0 = lane * KPL;
    const bool live = c0 < K;
    auto rows_of = [&](int64_t u) { return state + ((u / groups) * V + (u % groups) * kRows) * K; };
    auto issue = [&](int64_t u, int slot) {
        if (u < units && live) {
            const float* src = rows_of(u);
#pragma unroll
            for (int r = 0; r < kRows; ++r)
                cp_async<4 * KPL>(ring + slot * SLOT + r * 32 * KPL + c0, src + (int64_t)r * K + c0);
        }
        cp_commit();
    };
#pragma unroll
    for (int i = 0; i < kStages - 1; ++i) issue(w0 + i * W, i);

    int j = 0;
#pragma unroll 1
    for (int64_t u = w0; u < units; u += W, ++j) {
        cp_wait<kStages - 2>();  // this unit's rows have landed
        float S[kRows][KPL];
        const float* mine = ring + (j % kStages) * SLOT;
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            if (live) ldn<KPL>(mine + r * 32 * KPL + c0, S[r]);
            else
#pragma unroll
                for (int i = 0; i < KPL; ++i) S[r][i] = 0.f;
        }
        issue(u + (int64_t)(kStages - 1) * W, (j + kStages - 1) % kStages);  // into the slot read last unit

        const int64_t bh = u / groups;
        const int h = (int)(bh % d.H), b = (int)(bh / d.H);
        const int v0 = (int)(u % groups) * kRows;
#pragma unroll 1
        for (int t = 0; t < d.T; ++t) {
            const int64_t tok = ((int64_t)b * d.T + t) * d.H + h;
            float kv[KPL], qv[KPL];
            if (live) {
                ldn<KPL>(k + tok * K + c0, kv);
                ldn<KPL>(q + tok * K + c0, qv);
            } else {
#pragma unroll
                for (int i = 0; i < KPL; ++i) kv[i] = qv[i] = 0.f;
            }
            const float a = ld(alpha + tok), be = ld(beta + tok);
            float vv[kRows];
#pragma unroll
            for (int r4 = 0; r4 < kRows; r4 += 4) ldn<4>(v + tok * V + v0 + r4, vv + r4);
            // red[2r] = (S k)_r, red[2r+1] = (S q)_r, red[2R] = k^T q
            float red[2 * kRows + 1];
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                float sk = 0.f, sq = 0.f;
#pragma unroll
                for (int i = 0; i < KPL; ++i) {
                    sk = fmaf(S[r][i], kv[i], sk);
                    sq = fmaf(S[r][i], qv[i], sq);
                }
                red[2 * r] = sk;
                red[2 * r + 1] = sq;
            }
            float kq = 0.f;
#pragma unroll
            for (int i = 0; i < KPL; ++i) kq = fmaf(kv[i], qv[i], kq);
            red[2 * kRows] = kq;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                for (int jj = 0; jj < 2 * kRows + 1; ++jj) red[jj] += __shfl_xor_sync(0xffffffffu, red[jj], off);
            float ov = 0.f;  // output of row v0 + lane (lanes < kRows)
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                const float uu = be * (vv[r] - a * red[2 * r]);
#pragma unroll
                for (int i = 0; i < KPL; ++i) S[r][i] = fmaf(a, S[r][i], uu * kv[i]);
                const float outr = fmaf(a, red[2 * r + 1], uu * red[2 * kRows]);
                if (lane == r) ov = outr;
            }
            if (lane < kRows) st(o + tok * V + v0 + lane, ov);
        }

        if (live) {
            float* dst = rows_of(u);
#pragma unroll
            for (int r = 0; r < kRows; ++r) stn<KPL>(dst + (int64_t)r * K + c0, S[r]);
        }
    }
    cp_wait<0>();  // no copy outlives the kernel
}

template <typename Tin, int KPL>
cudaError_t launch_kpl(const Dims& d, const void* q, const void* k, const void* v, const void* alpha,
                       const void* beta, float* state, void* o, cudaStream_t st) {
    const int64_t warps = (int64_t)d.B * d.H * (d.V / kRows);  // V is a multiple of kRows (16 .. 128)
    const size_t smem = (size_t)8 * kStages * kRows * 32 * KPL * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<Tin, KPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    int per_sm = 0;
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<Tin, KPL>, 256, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t want = (warps + 7) / 8, cap = (int64_t)per_sm * sm_count();
    const int64_t blocks = want < cap ? want : cap;
    decode_kernel<Tin, KPL><<<(unsigned)blocks, 256, smem, st>>>(d, (const Tin*)q, (const Tin*)k, (const Tin*)v,
                                                                 (const Tin*)alpha, (const Tin*)beta, state,
                                                                 (Tin*)o);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_t(const Dims& d, const void* q, const void* k, const void* v, const void* alpha,
                     const void* beta, float* state, void* o, cudaStream_t st) {
    switch (d.K) {
        case 16:
        case 32: return launch_kpl<Tin, 1>(d, q, k, v, alpha, beta, state, o, st);
        case 64: return launch_kpl<Tin, 2>(d, q, k, v, alpha, beta, state, o, st);
        default: return launch_kpl<Tin, 4>(d, q, k, v, alpha, beta, state, o, st);
    }
}

}  // namespace

cudaError_t launch_decode(const Dims& d, InType ty, const void* q, const void* k, const void* v,
                          const void* alpha, const void* beta, float* state, void* o, cudaStream_t st) {
    if (ty == InType::BF16) return launch_t<__nv_bfloat16>(d, q, k, v, alpha, beta, state, o, st);
    return launch_t<float>(d, q, k, v, alpha, beta, state, o, st);
}

}  // namespace gdn
