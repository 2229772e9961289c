// prologue.cu -- the step in front of the recurrence in every mixer the pages
// show ("OpenGDN", Mixer: L2-normalized Q/K and per-head alpha/beta gates;
// "Sparse Delta Memory: layer and kernels", What the layer computes: l2-normalised
// weights in the dense limit), fused into one pass each way:
//   q = q_raw (sum_K q_raw^2 + eps)^(-1/2), the same for k (eps = 1e-6);
//   alpha = exp(-softplus(a)) = 1 / (1 + e^a),  beta = sigmoid(b) = 1 / (1 + e^-b);
// and the chain rule back to the raw tensors:
//   dx = r (dy - y (y . dy)) with r = (x . x + eps)^(-1/2), y = x r;
//   da = -dalpha alpha (1 - alpha),  db = dbeta beta (1 - beta).
// Rows (b, t, h) are independent.  Each lane owns one 16-byte piece of a row (a
// row spans K * size / 16 neighbouring lanes), the row sums are butterfly
// reductions over those lanes, and the gates of a tile's rows are read and
// written directly, one tile ahead.  Both kernels are bound by their HBM traffic.

#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr float kEps = 1e-6f;

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
    if constexpr (N == 8) {
        const uint4 x = *(const uint4*)p;
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) f[2 * e] = __uint_as_float(w[e] << 16), f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    } else if constexpr (N == 4) {
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
    if constexpr (N == 8) {
        *(uint4*)p = make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
    } else if constexpr (N == 4) {
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

// Sums over aligned groups of L lanes (L a power of two, at most 32).
template <int L, int M>
__device__ __forceinline__ void group_sum(float (&v)[M]) {
#pragma unroll
    for (int off = L / 2; off > 0; off >>= 1)
#pragma unroll
        for (int j = 0; j < M; ++j) v[j] += __shfl_xor_sync(0xffffffffu, v[j], off);
}


// Persistent kernels that stream the rows through shared memory: a tile holds TR
// rows of every input (8 KB per tensor for any K and dtype: two passes of the
// 256 threads, one 16-byte vector per lane, L = K / VPL lanes per row); cp.async
// brings tiles (stages - 1) ahead, so the bytes in flight do not depend on
// registers.  Rows past N are copied from row N - 1 and never stored.  A thread
// reads back exactly the 16-byte pieces it copied (piece tid + 256 p in pass p),
// so its own cp.async.wait_group orders everything: no block barrier.
// Stages of the ring: the forward's tiles hold two tensors, the backward's four.
// More resident CTAs (four per SM forward, three backward) pay more than a deeper
// ring: with two per SM and rings of five and three stages the kernels ran 12%
// and 9% slower.
constexpr int kStagesFwd = 3, kStagesBwd = 2;
static_assert(kStagesFwd >= 2 && kStagesBwd >= 2, "a ring holds the current tile and the next");

__device__ __forceinline__ void cp16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Waits until at most N of this thread's copy groups are still pending.
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <typename Tin, int K>
struct Pipe {
    static constexpr int ROWB = K * (int)sizeof(Tin);  // bytes per row
    static constexpr int VPL = 16 / (int)sizeof(Tin);  // elements per lane
    static constexpr int L = ROWB / 16;                // lanes per row
    static constexpr int RPP = 256 / L;                // rows per pass
    static constexpr int TR = 2 * RPP;                 // rows per tile
    static constexpr int TILEB = TR * ROWB;            // bytes per tensor and tile (8192)
    static_assert(L >= 1 && L <= 32 && TR <= 256, "a row within one warp; a tile's gates one per thread");
};

// Tile `tile` of the NIN tensors `src` into stage `stg` (2 x NIN 16-byte copies per thread).
template <typename Tin, int K, int NIN>
__device__ __forceinline__ void issue_tile(unsigned char* sm, int stg, int64_t tile, int64_t N,
                                           const Tin* const (&src)[NIN]) {
    using G = Pipe<Tin, K>;
    const int tid = threadIdx.x;
#pragma unroll
    for (int t = 0; t < NIN; ++t) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c = tid + 256 * h;  // 16-byte chunk of the tile
            const int r = c / G::L;
            int64_t n = tile * G::TR + r;
            if (n > N - 1) n = N - 1;
            cp16(sm + (stg * NIN + t) * G::TILEB + c * 16,
                 (const unsigned char*)src[t] + n * G::ROWB + (c % G::L) * 16);
        }
    }
}

template <typename Tin, int K>
__global__ void __launch_bounds__(256, 4)
prologue_fwd_kernel(int64_t N, const Tin* __restrict__ qr, const Tin* __restrict__ kr, const Tin* __restrict__ a,
                  const Tin* __restrict__ b, Tin* __restrict__ q, Tin* __restrict__ k, Tin* __restrict__ alpha,
                  Tin* __restrict__ beta) {
    using G = Pipe<Tin, K>;
    extern __shared__ __align__(16) unsigned char psm[];
    const int tid = threadIdx.x, sub = tid / G::L, c0 = (tid % G::L) * G::VPL;
    const int64_t ntiles = (N + G::TR - 1) / G::TR;
    const Tin* const src[2] = {qr, kr};
    constexpr int kStages = kStagesFwd;
    // gate logits of the next tile are read one tile ahead (thread tid: row tid)
    const bool grow = tid < G::TR;
    auto gates_in = [&](int64_t t, float& x, float& y) {
        const int64_t n = t * G::TR + tid;
        if (grow && t < ntiles && n < N) x = ld1(a + n), y = ld1(b + n);
    };
    float ga = 0.f, gb = 0.f;
    gates_in(blockIdx.x, ga, gb);
    for (int i = 0; i < kStages - 1; ++i) {
        const int64_t t = blockIdx.x + (int64_t)i * gridDim.x;
        if (t < ntiles) issue_tile<Tin, K, 2>(psm, i, t, N, src);
        cp_commit();
    }
    int j = 0;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++j) {
        cp_wait<kStages - 2>();  // groups 0 .. j done: this tile's pieces have landed
        const int64_t nt = tile + (int64_t)(kStages - 1) * gridDim.x;
        if (nt < ntiles) issue_tile<Tin, K, 2>(psm, (j + kStages - 1) % kStages, nt, N, src);
        cp_commit();
        float ga_n = 0.f, gb_n = 0.f;
        gates_in(tile + gridDim.x, ga_n, gb_n);
        const unsigned char* st = psm + (j % kStages) * 2 * G::TILEB;
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            const int r = pass * G::RPP + sub;
            const int64_t n = tile * G::TR + r;
            float xq[G::VPL], xk[G::VPL];
            ldv<G::VPL>((const Tin*)(st + r * G::ROWB) + c0, xq);
            ldv<G::VPL>((const Tin*)(st + G::TILEB + r * G::ROWB) + c0, xk);
            float red[2] = {0.f, 0.f};
#pragma unroll
            for (int i = 0; i < G::VPL; ++i) {
                red[0] = fmaf(xq[i], xq[i], red[0]);
                red[1] = fmaf(xk[i], xk[i], red[1]);
            }
            group_sum<G::L>(red);
            if (n < N) {
                const float rq = rsqrtf(red[0] + kEps), rk = rsqrtf(red[1] + kEps);
#pragma unroll
                for (int i = 0; i < G::VPL; ++i) {
                    xq[i] *= rq;
                    xk[i] *= rk;
                }
                stv<G::VPL>(q + n * K + c0, xq);
                stv<G::VPL>(k + n * K + c0, xk);
            }
        }
        if (grow && tile * G::TR + tid < N) {
            const int64_t n = tile * G::TR + tid;
            st1(alpha + n, gate_alpha(ga));
            st1(beta + n, gate_beta(gb));
        }
        ga = ga_n, gb = gb_n;
    }
}

template <typename Tin, int K>
__global__ void __launch_bounds__(256, 3)
prologue_bwd_kernel(int64_t N, const Tin* __restrict__ qr, const Tin* __restrict__ kr, const Tin* __restrict__ a,
                  const Tin* __restrict__ b, const Tin* __restrict__ dq, const Tin* __restrict__ dk,
                  const Tin* __restrict__ dalpha, const Tin* __restrict__ dbeta, Tin* __restrict__ dqr,
                  Tin* __restrict__ dkr, Tin* __restrict__ da, Tin* __restrict__ db) {
    using G = Pipe<Tin, K>;
    extern __shared__ __align__(16) unsigned char psm[];
    const int tid = threadIdx.x, sub = tid / G::L, c0 = (tid % G::L) * G::VPL;
    const int64_t ntiles = (N + G::TR - 1) / G::TR;
    const Tin* const src[4] = {qr, kr, dq, dk};
    constexpr int kStages = kStagesBwd;
    const bool grow = tid < G::TR;
    auto gates_in = [&](int64_t t, float (&x)[4]) {
        const int64_t n = t * G::TR + tid;
        if (grow && t < ntiles && n < N) x[0] = ld1(a + n), x[1] = ld1(b + n), x[2] = ld1(dalpha + n), x[3] = ld1(dbeta + n);
    };
    float gv[4] = {0.f, 0.f, 0.f, 0.f};
    gates_in(blockIdx.x, gv);
    for (int i = 0; i < kStages - 1; ++i) {
        const int64_t t = blockIdx.x + (int64_t)i * gridDim.x;
        if (t < ntiles) issue_tile<Tin, K, 4>(psm, i, t, N, src);
        cp_commit();
    }
    int j = 0;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++j) {
        cp_wait<kStages - 2>();
        const int64_t nt = tile + (int64_t)(kStages - 1) * gridDim.x;
        if (nt < ntiles) issue_tile<Tin, K, 4>(psm, (j + kStages - 1) % kStages, nt, N, src);
        cp_commit();
        float gv_n[4] = {0.f, 0.f, 0.f, 0.f};
        gates_in(tile + gridDim.x, gv_n);
        const unsigned char* st = psm + (j % kStages) * 4 * G::TILEB;
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            const int r = pass * G::RPP + sub;
            const int64_t n = tile * G::TR + r;
            float xq[G::VPL], xk[G::VPL], gq[G::VPL], gk[G::VPL];
            ldv<G::VPL>((const Tin*)(st + r * G::ROWB) + c0, xq);
            ldv<G::VPL>((const Tin*)(st + G::TILEB + r * G::ROWB) + c0, xk);
            ldv<G::VPL>((const Tin*)(st + 2 * G::TILEB + r * G::ROWB) + c0, gq);
            ldv<G::VPL>((const Tin*)(st + 3 * G::TILEB + r * G::ROWB) + c0, gk);
            // x.x and x.dy for q and k
            float red[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < G::VPL; ++i) {
                red[0] = fmaf(xq[i], xq[i], red[0]);
                red[1] = fmaf(xk[i], xk[i], red[1]);
                red[2] = fmaf(xq[i], gq[i], red[2]);
                red[3] = fmaf(xk[i], gk[i], red[3]);
            }
            group_sum<G::L>(red);
            if (n < N) {
                // dx = r dy - x r^3 (x . dy)
                const float rq = rsqrtf(red[0] + kEps), rk = rsqrtf(red[1] + kEps);
                const float cq = rq * rq * rq * red[2], ck = rk * rk * rk * red[3];
#pragma unroll
                for (int i = 0; i < G::VPL; ++i) {
                    gq[i] = rq * gq[i] - cq * xq[i];
                    gk[i] = rk * gk[i] - ck * xk[i];
                }
                stv<G::VPL>(dqr + n * K + c0, gq);
                stv<G::VPL>(dkr + n * K + c0, gk);
            }
        }
        if (grow && tile * G::TR + tid < N) {
            const int64_t n = tile * G::TR + tid;
            const float al = gate_alpha(gv[0]), be = gate_beta(gv[1]);
            st1(da + n, -gv[2] * al * (1.f - al));
            st1(db + n, gv[3] * be * (1.f - be));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) gv[i] = gv_n[i];
    }
}

// Grid: the resident CTAs of every SM (at most the number of tiles).
template <typename KernelT>
int64_t pipe_grid(KernelT kern, size_t smem, int64_t ntiles, cudaError_t& e) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    int per_sm = 0;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, smem);
    if (per_sm < 1) per_sm = 1;
    const int64_t g = (int64_t)per_sm * sm_count();
    return g < ntiles ? g : ntiles;
}

template <typename Tin, int K>
cudaError_t launch_fwd_k(int64_t N, const void* qr, const void* kr, const void* a, const void* b, void* q, void* k,
                         void* alpha, void* beta, cudaStream_t st) {
    using G = Pipe<Tin, K>;
    const size_t smem = (size_t)kStagesFwd * 2 * G::TILEB;
    cudaError_t e;
    const int64_t grid = pipe_grid(prologue_fwd_kernel<Tin, K>, smem, (N + G::TR - 1) / G::TR, e);
    if (e != cudaSuccess) return e;
    prologue_fwd_kernel<Tin, K><<<(unsigned)grid, 256, smem, st>>>(N, (const Tin*)qr, (const Tin*)kr, (const Tin*)a,
                                                                 (const Tin*)b, (Tin*)q, (Tin*)k, (Tin*)alpha,
                                                                 (Tin*)beta);
    return cudaGetLastError();
}

template <typename Tin, int K>
cudaError_t launch_bwd_k(int64_t N, const void* qr, const void* kr, const void* a, const void* b, const void* dq,
                         const void* dk, const void* dalpha, const void* dbeta, void* dqr, void* dkr, void* da,
                         void* db, cudaStream_t st) {
    using G = Pipe<Tin, K>;
    const size_t smem = (size_t)kStagesBwd * 4 * G::TILEB;
    cudaError_t e;
    const int64_t grid = pipe_grid(prologue_bwd_kernel<Tin, K>, smem, (N + G::TR - 1) / G::TR, e);
    if (e != cudaSuccess) return e;
    prologue_bwd_kernel<Tin, K><<<(unsigned)grid, 256, smem, st>>>(
        N, (const Tin*)qr, (const Tin*)kr, (const Tin*)a, (const Tin*)b, (const Tin*)dq, (const Tin*)dk,
        (const Tin*)dalpha, (const Tin*)dbeta, (Tin*)dqr, (Tin*)dkr, (Tin*)da, (Tin*)db);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t fwd_t(int64_t N, int K, const void* qr, const void* kr, const void* a, const void* b, void* q, void* k,
                  void* alpha, void* beta, cudaStream_t st) {
    switch (K) {
        case 16: return launch_fwd_k<Tin, 16>(N, qr, kr, a, b, q, k, alpha, beta, st);
        case 32: return launch_fwd_k<Tin, 32>(N, qr, kr, a, b, q, k, alpha, beta, st);
        case 64: return launch_fwd_k<Tin, 64>(N, qr, kr, a, b, q, k, alpha, beta, st);
        default: return launch_fwd_k<Tin, 128>(N, qr, kr, a, b, q, k, alpha, beta, st);
    }
}

template <typename Tin>
cudaError_t bwd_t(int64_t N, int K, const void* qr, const void* kr, const void* a, const void* b, const void* dq,
                  const void* dk, const void* dalpha, const void* dbeta, void* dqr, void* dkr, void* da, void* db,
                  cudaStream_t st) {
    switch (K) {
        case 16: return launch_bwd_k<Tin, 16>(N, qr, kr, a, b, dq, dk, dalpha, dbeta, dqr, dkr, da, db, st);
        case 32: return launch_bwd_k<Tin, 32>(N, qr, kr, a, b, dq, dk, dalpha, dbeta, dqr, dkr, da, db, st);
        case 64: return launch_bwd_k<Tin, 64>(N, qr, kr, a, b, dq, dk, dalpha, dbeta, dqr, dkr, da, db, st);
        default: return launch_bwd_k<Tin, 128>(N, qr, kr, a, b, dq, dk, dalpha, dbeta, dqr, dkr, da, db, st);
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
