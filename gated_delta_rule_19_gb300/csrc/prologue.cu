// prologue.cu -- the step in front of the recurrence in every mixer the pages
// show ("OpenGDN", Mixer: L2-normalized Q/K and per-head alpha/beta gates;
// "Sparse Delta Memory: layer and kernels", What the layer computes: l2-normalised
// weights in the dense limit), fused into one pass each way:
//   q = q_raw (sum_K q_raw^2 + eps)^(-1/2), the same for k (eps = 1e-6);
//   alpha = exp(-softplus(a)) = 1 / (1 + e^a),  beta = sigmoid(b) = 1 / (1 + e^-b);
// and the chain rule back to the raw tensors:
//   dx = r (dy - y (y . dy)) with r = (x . x + eps)^(-1/2), y = x r;
//   da = -dalpha alpha (1 - alpha),  db = dbeta beta (1 - beta).
// Rows (b, t, h) are independent: one warp handles four rows, lane l holds K/32
// consecutive elements of each (one vector load), the row sums are butterfly
// reductions, and the first four lanes compute the four rows' gates.  Both
// kernels are bound by their HBM traffic.

#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr float kEps = 1e-6f;
constexpr int kR = 4;  // rows per warp

template <int N>
__device__ __forceinline__ void ldv(const float* p, float* f) {
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
__device__ __forceinline__ void ldv(const __nv_bfloat16* p, float* f) {
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
__device__ __forceinline__ void stv(float* p, const float* f) {
    if constexpr (N == 4) {
        *(float4*)p = make_float4(f[0], f[1], f[2], f[3]);
    } else if constexpr (N == 2) {
        *(float2*)p = make_float2(f[0], f[1]);
    } else {
        *p = f[0];
    }
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
template <int N>
__device__ __forceinline__ void stv(__nv_bfloat16* p, const float* f) {
    if constexpr (N == 4) {
        *(uint2*)p = make_uint2(pack2(f[0], f[1]), pack2(f[2], f[3]));
    } else if constexpr (N == 2) {
        *(uint32_t*)p = pack2(f[0], f[1]);
    } else {
        *p = __float2bfloat16_rn(f[0]);
    }
}
__device__ __forceinline__ float ld1(const float* p) { return *p; }
__device__ __forceinline__ float ld1(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st1(float* p, float x) { *p = x; }
__device__ __forceinline__ void st1(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// alpha = exp(-softplus(a)) = 1 / (1 + e^a); beta = 1 / (1 + e^-b).  expf saturates
// to inf or 0 for large |x|, giving exactly 0 or 1.
__device__ __forceinline__ float gate_alpha(float a) { return 1.f / (1.f + expf(a)); }
__device__ __forceinline__ float gate_beta(float b) { return 1.f / (1.f + expf(-b)); }

template <int M>
__device__ __forceinline__ void warp_sum(float (&v)[M]) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int j = 0; j < M; ++j) v[j] += __shfl_xor_sync(0xffffffffu, v[j], off);
}

template <typename Tin, int KPL>
__global__ void __launch_bounds__(256)
prologue_fwd_kernel(int64_t N, int K, const Tin* __restrict__ qr, const Tin* __restrict__ kr,
                    const Tin* __restrict__ a, const Tin* __restrict__ b, Tin* __restrict__ q, Tin* __restrict__ k,
                    Tin* __restrict__ alpha, Tin* __restrict__ beta) {
    const int lane = threadIdx.x & 31;
    const int64_t n0 = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * kR;
    if (n0 >= N) return;  // whole warps leave together
    const int c0 = lane * KPL;
    const bool live = c0 < K;
    float xq[kR][KPL], xk[kR][KPL];
#pragma unroll
    for (int r = 0; r < kR; ++r) {
        const int64_t n = n0 + r;
        if (live && n < N) {
            ldv<KPL>(qr + n * K + c0, xq[r]);
            ldv<KPL>(kr + n * K + c0, xk[r]);
        } else {
#pragma unroll
            for (int i = 0; i < KPL; ++i) xq[r][i] = xk[r][i] = 0.f;
        }
    }
    float red[2 * kR];
#pragma unroll
    for (int r = 0; r < kR; ++r) {
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
            sq = fmaf(xq[r][i], xq[r][i], sq);
            sk = fmaf(xk[r][i], xk[r][i], sk);
        }
        red[2 * r] = sq;
        red[2 * r + 1] = sk;
    }
    warp_sum(red);
#pragma unroll
    for (int r = 0; r < kR; ++r) {
        const int64_t n = n0 + r;
        if (!live || n >= N) continue;
        const float rq = rsqrtf(red[2 * r] + kEps), rk = rsqrtf(red[2 * r + 1] + kEps);
        float yq[KPL], yk[KPL];
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
            yq[i] = xq[r][i] * rq;
            yk[i] = xk[r][i] * rk;
        }
        stv<KPL>(q + n * K + c0, yq);
        stv<KPL>(k + n * K + c0, yk);
    }
    if (lane < kR && n0 + lane < N) {
        const int64_t n = n0 + lane;
        st1(alpha + n, gate_alpha(ld1(a + n)));
        st1(beta + n, gate_beta(ld1(b + n)));
    }
}

template <typename Tin, int KPL>
__global__ void __launch_bounds__(256)
prologue_bwd_kernel(int64_t N, int K, const Tin* __restrict__ qr, const Tin* __restrict__ kr,
                    const Tin* __restrict__ a, const Tin* __restrict__ b, const Tin* __restrict__ dq,
                    const Tin* __restrict__ dk, const Tin* __restrict__ dalpha, const Tin* __restrict__ dbeta,
                    Tin* __restrict__ dqr, Tin* __restrict__ dkr, Tin* __restrict__ da, Tin* __restrict__ db) {
    const int lane = threadIdx.x & 31;
    const int64_t n0 = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * kR;
    if (n0 >= N) return;
    const int c0 = lane * KPL;
    const bool live = c0 < K;
    float xq[kR][KPL], xk[kR][KPL], gq[kR][KPL], gk[kR][KPL];
#pragma unroll
    for (int r = 0; r < kR; ++r) {
        const int64_t n = n0 + r;
        if (live && n < N) {
            ldv<KPL>(qr + n * K + c0, xq[r]);
            ldv<KPL>(kr + n * K + c0, xk[r]);
            ldv<KPL>(dq + n * K + c0, gq[r]);
            ldv<KPL>(dk + n * K + c0, gk[r]);
        } else {
#pragma unroll
            for (int i = 0; i < KPL; ++i) xq[r][i] = xk[r][i] = gq[r][i] = gk[r][i] = 0.f;
        }
    }
    // per row: x.x and x.dy for q and k
    float red[4 * kR];
#pragma unroll
    for (int r = 0; r < kR; ++r) {
        float sq = 0.f, sk = 0.f, pq = 0.f, pk = 0.f;
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
            sq = fmaf(xq[r][i], xq[r][i], sq);
            sk = fmaf(xk[r][i], xk[r][i], sk);
            pq = fmaf(xq[r][i], gq[r][i], pq);
            pk = fmaf(xk[r][i], gk[r][i], pk);
        }
        red[4 * r] = sq, red[4 * r + 1] = sk, red[4 * r + 2] = pq, red[4 * r + 3] = pk;
    }
    warp_sum(red);
#pragma unroll
    for (int r = 0; r < kR; ++r) {
        const int64_t n = n0 + r;
        if (!live || n >= N) continue;
        // dx = r dy - x r^3 (x . dy)
        const float rq = rsqrtf(red[4 * r] + kEps), rk = rsqrtf(red[4 * r + 1] + kEps);
        const float cq = rq * rq * rq * red[4 * r + 2], ck = rk * rk * rk * red[4 * r + 3];
        float oq[KPL], ok2[KPL];
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
            oq[i] = rq * gq[r][i] - cq * xq[r][i];
            ok2[i] = rk * gk[r][i] - ck * xk[r][i];
        }
        stv<KPL>(dqr + n * K + c0, oq);
        stv<KPL>(dkr + n * K + c0, ok2);
    }
    if (lane < kR && n0 + lane < N) {
        const int64_t n = n0 + lane;
        const float al = gate_alpha(ld1(a + n)), be = gate_beta(ld1(b + n));
        st1(da + n, -ld1(dalpha + n) * al * (1.f - al));
        st1(db + n, ld1(dbeta + n) * be * (1.f - be));
    }
}

template <typename Tin, int KPL>
cudaError_t launch_fwd_k(int64_t N, int K, const void* qr, const void* kr, const void* a, const void* b, void* q,
                         void* k, void* alpha, void* beta, cudaStream_t st) {
    const int64_t blocks = (N + 8 * kR - 1) / (8 * kR);
    prologue_fwd_kernel<Tin, KPL><<<(unsigned)blocks, 256, 0, st>>>(
        N, K, (const Tin*)qr, (const Tin*)kr, (const Tin*)a, (const Tin*)b, (Tin*)q, (Tin*)k, (Tin*)alpha,
        (Tin*)beta);
    return cudaGetLastError();
}

template <typename Tin, int KPL>
cudaError_t launch_bwd_k(int64_t N, int K, const void* qr, const void* kr, const void* a, const void* b,
                         const void* dq, const void* dk, const void* dalpha, const void* dbeta, void* dqr, void* dkr,
                         void* da, void* db, cudaStream_t st) {
    const int64_t blocks = (N + 8 * kR - 1) / (8 * kR);
    prologue_bwd_kernel<Tin, KPL><<<(unsigned)blocks, 256, 0, st>>>(
        N, K, (const Tin*)qr, (const Tin*)kr, (const Tin*)a, (const Tin*)b, (const Tin*)dq, (const Tin*)dk,
        (const Tin*)dalpha, (const Tin*)dbeta, (Tin*)dqr, (Tin*)dkr, (Tin*)da, (Tin*)db);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t fwd_t(int64_t N, int K, const void* qr, const void* kr, const void* a, const void* b, void* q, void* k,
                  void* alpha, void* beta, cudaStream_t st) {
    switch (K) {
        case 16:
        case 32: return launch_fwd_k<Tin, 1>(N, K, qr, kr, a, b, q, k, alpha, beta, st);
        case 64: return launch_fwd_k<Tin, 2>(N, K, qr, kr, a, b, q, k, alpha, beta, st);
        default: return launch_fwd_k<Tin, 4>(N, K, qr, kr, a, b, q, k, alpha, beta, st);
    }
}

template <typename Tin>
cudaError_t bwd_t(int64_t N, int K, const void* qr, const void* kr, const void* a, const void* b, const void* dq,
                  const void* dk, const void* dalpha, const void* dbeta, void* dqr, void* dkr, void* da, void* db,
                  cudaStream_t st) {
    switch (K) {
        case 16:
        case 32: return launch_bwd_k<Tin, 1>(N, K, qr, kr, a, b, dq, dk, dalpha, dbeta, dqr, dkr, da, db, st);
        case 64: return launch_bwd_k<Tin, 2>(N, K, qr, kr, a, b, dq, dk, dalpha, dbeta, dqr, dkr, da, db, st);
        default: return launch_bwd_k<Tin, 4>(N, K, qr, kr, a, b, dq, dk, dalpha, dbeta, dqr, dkr, da, db, st);
    }
}

}  // namespace

cudaError_t launch_prologue_fwd(const Dims& d, InType ty, const void* qr, const void* kr, const void* a,
                                const void* b, void* q, void* k, void* alpha, void* beta, cudaStream_t st) {
    const int64_t N = (int64_t)d.B * d.T * d.H;
    if (ty == InType::BF16) return fwd_t<__nv_bfloat16>(N, d.K, qr, kr, a, b, q, k, alpha, beta, st);
    return fwd_t<float>(N, d.K, qr, kr, a, b, q, k, alpha, beta, st);
}

cudaError_t launch_prologue_bwd(const Dims& d, InType ty, const void* qr, const void* kr, const void* a,
                                const void* b, const void* dq, const void* dk, const void* dalpha, const void* dbeta,
                                void* dqr, void* dkr, void* da, void* db, cudaStream_t st) {
    const int64_t N = (int64_t)d.B * d.T * d.H;
    if (ty == InType::BF16)
        return bwd_t<__nv_bfloat16>(N, d.K, qr, kr, a, b, dq, dk, dalpha, dbeta, dqr, dkr, da, db, st);
    return bwd_t<float>(N, d.K, qr, kr, a, b, dq, dk, dalpha, dbeta, dqr, dkr, da, db, st);
}

}  // namespace gdn
