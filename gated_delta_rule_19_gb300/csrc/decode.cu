// decode.cu -- the recurrent step for decoding: a few tokens per call, the state
// read and written once ("OpenGDN", Core operator reference: a stream continued
// exactly through state=; "Sparse Delta Memory: layer and kernels", Execution:
// the single-token call).
//
// Per (b, h) the state S [V, K] advances token by token:
//   S <- alpha S (I - beta k k^T) + beta v k^T = alpha S + beta (v - alpha S k) k^T
//   o  = S q = alpha (S q) + beta (v - alpha S k) (k^T q)
// Row v of S only needs row v, so one warp owns R rows of one head, keeps them in
// registers across the call's tokens (lane l holds K/32 consecutive columns, one
// vector load per row), and reduces the row dot products S k, S q with butterfly
// shuffles.  The kernel is bound by reading and writing the fp32 state once.

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

constexpr int kRows = 8;  // state rows per warp (with K = 128: 4 KB of state loads in flight per warp)

// Lane l holds columns [l*KPL, l*KPL + KPL) of each of its rows (K = 32*KPL; for
// K = 16, KPL = 1 and lanes 16-31 hold nothing).
template <typename Tin, int KPL>
__global__ void __launch_bounds__(256)
decode_kernel(Dims d, const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
              const Tin* __restrict__ alpha, const Tin* __restrict__ beta, float* __restrict__ state,
              Tin* __restrict__ o) {
    const int lane = threadIdx.x & 31;
    const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int groups = d.V / kRows;
    if (wid >= (int64_t)d.B * d.H * groups) return;  // whole warps leave together
    const int g = (int)(wid % groups);
    const int64_t bh = wid / groups;  // b * H + h
    const int h = (int)(bh % d.H), b = (int)(bh / d.H);
    const int v0 = g * kRows;
    const int K = d.K, V = d.V;
    const int c0 = lane * KPL;
    const bool live = c0 < K;

    float S[kRows][KPL];
    float* srow = state + (bh * V + v0) * K;
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        if (live) ldn<KPL>(srow + (int64_t)r * K + c0, S[r]);
        else
#pragma unroll
            for (int i = 0; i < KPL; ++i) S[r][i] = 0.f;
    }

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
            for (int j = 0; j < 2 * kRows + 1; ++j) red[j] += __shfl_xor_sync(0xffffffffu, red[j], off);
        float ov = 0.f;  // output of row v0 + lane (lanes < kRows)
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const float u = be * (vv[r] - a * red[2 * r]);
#pragma unroll
            for (int i = 0; i < KPL; ++i) S[r][i] = fmaf(a, S[r][i], u * kv[i]);
            const float outr = fmaf(a, red[2 * r + 1], u * red[2 * kRows]);
            if (lane == r) ov = outr;
        }
        if (lane < kRows) st(o + tok * V + v0 + lane, ov);
    }

    if (live)
#pragma unroll
        for (int r = 0; r < kRows; ++r) stn<KPL>(srow + (int64_t)r * K + c0, S[r]);
}

template <typename Tin, int KPL>
cudaError_t launch_kpl(const Dims& d, const void* q, const void* k, const void* v, const void* alpha,
                       const void* beta, float* state, void* o, cudaStream_t st) {
    const int64_t warps = (int64_t)d.B * d.H * (d.V / kRows);
    const int64_t blocks = (warps + 7) / 8;  // V is a multiple of kRows (16, 32, 64, 128)
    decode_kernel<Tin, KPL><<<(unsigned)blocks, 256, 0, st>>>(d, (const Tin*)q, (const Tin*)k, (const Tin*)v,
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
