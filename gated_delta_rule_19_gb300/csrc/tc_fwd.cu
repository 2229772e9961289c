// tc_fwd.cu -- tensor-core (tcgen05 + TMA) forward for bf16 inputs, K = V = 128,
// chunk 64.
//
// prep_fwd_tc (one CTA per chunk, chunk-parallel; "Sparse Delta Memory: layer and
// kernels", "What the layer computes", Phase 1 and Solve):
//   TMA loads of the chunk's K, Q, V tiles (128B-swizzled, K-major);
//   one M=128 MMA gives [K;Q] K^T = [K K^T ; Q K^T] in TMEM;
//   A = strict_lower(beta_r Gam_ri (K K^T)_ri) -> fp32 solve T = (I + A)^-1
//   (16x16 diagonal blocks in registers, off-diagonal blocks in shared memory);
//   Mqk = lower(Gam .* Q K^T) -> bf16;
//   W^T = K^T (T diag(beta gamma))^T and Ut^T = V^T (T diag(beta))^T as M=128
//   MMAs with K and V read MN-major from the same tiles;
//   W, Ut, Mqk leave through TMA stores as bf16 [rows = chunk*64 + r][...].
//
// scan_fwd_tc (one CTA per (V-slice of Vt rows, head, batch); Phase 2):
//   the state slice S^T [K=128, Vt] lives in registers (fp32, thread k = row k) and
//   as a bf16 MMA operand in shared memory; per chunk
//     Y = Q S0^T, X = W S0^T          (M=64 MMAs)
//     U = Ut - X,  Uh = diag(exp(G_C - G)) U
//     O = diag(gamma) Y + Mqk U       (M=64 MMA)
//     S1^T = gamma_C S0^T + K^T Uh    (M=128 MMA)
//   with the next chunk's Q, W, K, Mqk tiles prefetched by TMA (two stages).
//
// Every wait is bounded (2 s); a wait that gives up raises the error flag, and
// the block leaves its loop together (block-wide vote) after draining its copies.

#include <cudaTypedefs.h>

#include "gdn_internal.h"
#include "tc.cuh"

namespace gdn {
namespace {

using namespace tc;
using bf16 = __nv_bfloat16;

constexpr int kC = 64;
constexpr int kD = 128;  // K = V = 128

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// In-place inclusive prefix sum of x[0..64) by one warp.
__device__ __forceinline__ void warp_cumsum64(float* x) {
    const int lane = threadIdx.x & 31;
    float a = x[2 * lane], b = x[2 * lane + 1];
    b += a;
    float incl = b;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    const float excl = incl - b;
    x[2 * lane] = a + excl;
    x[2 * lane + 1] = b + excl;
}

// T = (I + A)^-1 for strictly lower A (64 x 64, row stride 65), fp32.  128 threads.
// Diagonal 16x16 blocks: warp w solves block w, lane j < 16 carries column j in
// registers (no synchronisation inside a block).  Then block rows I = 1..3:
// T_IJ = -T_II * sum_{J<=L<I} A_IL T_LJ.  Only the lower blocks of Tf are written.
__device__ void solve_unit_lower_64(const float* A, float* Tf, float* X) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (lane < 16) {
        const int base = warp * 16, j = lane;
        float t[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < r; ++i) acc += A[(base + r) * 65 + base + i] * t[i];
            t[r] = (r < j) ? 0.f : (r == j ? 1.f : -acc);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) Tf[(base + r) * 65 + base + j] = t[r];
    }
    __syncthreads();
#pragma unroll 1
    for (int I = 1; I < 4; ++I) {
        const int n = I * 256;
        for (int idx = tid; idx < n; idx += 128) {
            const int J = idx >> 8, r = (idx >> 4) & 15, c = idx & 15;
            float acc = 0.f;
            for (int L = J; L < I; ++L) {
                const float* ar = A + (I * 16 + r) * 65 + L * 16;
                const float* tc_ = Tf + (L * 16) * 65 + J * 16 + c;
#pragma unroll
                for (int m = 0; m < 16; ++m) acc += ar[m] * tc_[m * 65];
            }
            X[idx] = acc;
        }
        __syncthreads();
        for (int idx = tid; idx < n; idx += 128) {
            const int J = idx >> 8, r = (idx >> 4) & 15, c = idx & 15;
            const float* tr = Tf + (I * 16 + r) * 65 + I * 16;
            float acc = 0.f;
            for (int m = 0; m <= r; ++m) acc += tr[m] * X[(J << 8) + (m << 4) + c];
            Tf[(I * 16 + r) * 65 + J * 16 + c] = -acc;
        }
        __syncthreads();
    }
}

// Shared-memory plan of prep_fwd_tc (offsets from a 1024-aligned base).
constexpr int P_QK = 0;           // [K_0 | Q_0 | K_1 | Q_1], 8 KB each (64 rows x 64 bf16)
constexpr int P_V = 32768;        // V_0 | V_1
constexpr int P_T1 = 49152;       // T diag(beta gamma), bf16 K-major
constexpr int P_T2 = 57344;       // T diag(beta)
constexpr int P_AF = 65536;       // fp32 A [64][65]
constexpr int P_TF = P_AF + 64 * 65 * 4;
constexpr int P_XF = P_TF + 64 * 65 * 4;
constexpr int P_G = P_XF + 768 * 4;  // G, gamma, beta: 3 x 64 floats
constexpr int P_BAR = P_G + 3 * 64 * 4;
constexpr int P_END = P_BAR + 64;
constexpr size_t kPrepSmem = P_END + 1024;

__global__ void __launch_bounds__(128, 2)
prep_fwd_tc(Dims d, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_W,
            const __grid_constant__ CUtensorMap tm_U, const __grid_constant__ CUtensorMap tm_M,
            const bf16* __restrict__ alpha, const bf16* __restrict__ beta, float* __restrict__ Gout,
            bf16* __restrict__ Tout, int* err) {
    extern __shared__ unsigned char smraw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    float* Af = (float*)(sm + P_AF);
    float* Tf = (float*)(sm + P_TF);
    float* Xf = (float*)(sm + P_XF);
    float* Gs = (float*)(sm + P_G);
    float* gs = Gs + 64;
    float* bs = gs + 64;
    uint64_t* bars = (uint64_t*)(sm + P_BAR);  // [0] TMA, [1] MMA
    uint32_t* tslot = (uint32_t*)(sm + P_BAR + 16);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int t0 = c * kC;
    const int64_t chunk = ((int64_t)b * d.H + h) * d.NC + c;
    const int row0 = (int)(chunk * kC);

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&bars[0], 6 * 8192);
        for (int j = 0; j < 2; ++j) {
            tma_load_4d(sm + P_QK + j * 16384, &tm_k, &bars[0], 64 * j, h, t0, b);
            tma_load_4d(sm + P_QK + j * 16384 + 8192, &tm_q, &bars[0], 64 * j, h, t0, b);
            tma_load_4d(sm + P_V + j * 8192, &tm_v, &bars[0], 64 * j, h, t0, b);
        }
    }
    if (warp == 0) {
        tmem_alloc(tslot, 128);
        tmem_relinquish();
    }
    if (tid < 64) {
        const int t = t0 + tid;
        float a = 1.f, be = 0.f;  // padding: alpha = 1, beta = 0 leaves the state unchanged
        if (t < d.T) {
            const int64_t gi = ((int64_t)b * d.T + t) * d.H + h;
            a = __bfloat162float(alpha[gi]);
            be = __bfloat162float(beta[gi]);
        }
        Gs[tid] = logf(a);
        bs[tid] = be;
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    if (warp == 0) {
        warp_cumsum64(Gs);
        __syncwarp();
        gs[2 * lane] = expf(Gs[2 * lane]);
        gs[2 * lane + 1] = expf(Gs[2 * lane + 1]);
    }
    bool ok = true;
    if (tid == 0) {
        ok = mbar_wait(&bars[0], 0, err, 1);
        if (ok) {
            const uint32_t id = idesc_bf16(128, 64, false, false);
            const uint32_t base = smem_u32(sm + P_QK);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t a = base + (s >> 2) * 16384 + (s & 3) * 32;
                mma_bf16_ss(tmem, sdesc(a, 16, 1024, SW_128B), sdesc(a, 16, 1024, SW_128B), id, s > 0);
            }
            mma_commit(&bars[1]);
        }
    }
    __syncthreads();  // G, gamma, beta visible
    ok = mbar_wait(&bars[1], 0, err, 2) && ok;
    __syncwarp();
    fence_after_sync();
    // Gram epilogue.  Warps 0-1: rows of K K^T -> A (fp32).  Warps 2-3: rows of
    // Q K^T -> Mqk (bf16, into the dead Q_0 slot as a 128B-swizzled tile).
    {
        const int r = tid & 63;
        const float Gr = Gs[r];
        const float br = bs[r];
        unsigned char* mt = sm + P_QK + 8192;
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
            tmem_wait_ld(v);
            if (warp < 2) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int i = c0 + j;
                    Af[r * 65 + i] = (i < r) ? br * expf(Gr - Gs[i]) * __uint_as_float(v[j]) : 0.f;
                }
            } else {
                uint32_t pk[8];
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    const int i = c0 + j;
                    const float m0 = (i <= r) ? expf(Gr - Gs[i]) * __uint_as_float(v[j]) : 0.f;
                    const float m1 = (i + 1 <= r) ? expf(Gr - Gs[i + 1]) * __uint_as_float(v[j + 1]) : 0.f;
                    pk[j >> 1] = pack_bf16(m0, m1);
                }
                *(uint4*)(mt + sw128_off(r, c0)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                *(uint4*)(mt + sw128_off(r, c0 + 8)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
        }
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    if (tid == 0) {
        tma_store_2d(&tm_M, sm + P_QK + 8192, 0, row0);
        bulk_commit();
    }
    solve_unit_lower_64(Af, Tf, Xf);  // ends with __syncthreads
    // B operands of the recompute: T1 = T diag(beta gamma), T2 = T diag(beta), bf16
    // K-major [r][i], zero above the diagonal.
    {
        const int r = tid >> 1, i0 = (tid & 1) * 32;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t p0[4], p1[4], p2[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = i0 + q * 8 + 2 * e;
                const float ta = (i <= r) ? Tf[r * 65 + i] : 0.f;
                const float tb = (i + 1 <= r) ? Tf[r * 65 + i + 1] : 0.f;
                p0[e] = pack_bf16(ta, tb);
                p1[e] = pack_bf16(ta * bs[i] * gs[i], tb * bs[i + 1] * gs[i + 1]);
                p2[e] = pack_bf16(ta * bs[i], tb * bs[i + 1]);
            }
            if (Tout)
                *(uint4*)(Tout + ((int64_t)row0 + r) * kC + i0 + q * 8) = make_uint4(p0[0], p0[1], p0[2], p0[3]);
            *(uint4*)(sm + P_T1 + sw128_off(r, i0 + q * 8)) = make_uint4(p1[0], p1[1], p1[2], p1[3]);
            *(uint4*)(sm + P_T2 + sw128_off(r, i0 + q * 8)) = make_uint4(p2[0], p2[1], p2[2], p2[3]);
        }
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid == 0 && ok) {
        // W^T [k, r] = K^T T1^T and Ut^T [v, r] = V^T T2^T: A read MN-major from the
        // K / V tiles (64-wide column blocks 16 KB / 8 KB apart), B = T1 / T2.
        const uint32_t id = idesc_bf16(128, 64, true, false);
        const uint32_t kb = smem_u32(sm + P_QK), vb = smem_u32(sm + P_V);
        const uint32_t t1 = smem_u32(sm + P_T1), t2 = smem_u32(sm + P_T2);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            mma_bf16_ss(tmem + 64, sdesc(kb + s * 2048, 16384, 1024, SW_128B),
                        sdesc(t1 + s * 32, 16, 1024, SW_128B), id, s > 0);
            mma_bf16_ss(tmem + 0, sdesc(vb + s * 2048, 8192, 1024, SW_128B),
                        sdesc(t2 + s * 32, 16, 1024, SW_128B), id, s > 0);
        }
        mma_commit(&bars[1]);
    }
    ok = __syncthreads_and(ok);
    if (ok) ok = mbar_wait(&bars[1], 1, err, 4);
    __syncwarp();
    fence_after_sync();
    // Epilogue: thread k holds row k of W^T / Ut^T -> write W[r][k], Ut[r][v] into
    // the K / V tile slots (dead now) as 128B-swizzled K-major tiles.
    {
        const int k = tid;
        unsigned char* wt = sm + P_QK + (k >> 6) * 16384;
        unsigned char* ut = sm + P_V + (k >> 6) * 8192;
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 16) {
            uint32_t w[16], u[16];
            tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + 64 + c0, w);
            tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c0, u);
            tmem_wait_ld(w);
            tmem_wait_ld(u);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                *(bf16*)(wt + sw128_off(c0 + j, k & 63)) = __float2bfloat16_rn(__uint_as_float(w[j]));
                *(bf16*)(ut + sw128_off(c0 + j, k & 63)) = __float2bfloat16_rn(__uint_as_float(u[j]));
            }
        }
    }
    if (tid < 64) Gout[(int64_t)row0 + tid] = Gs[tid];
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    if (tid == 0) {
        for (int j = 0; j < 2; ++j) {
            tma_store_2d(&tm_W, sm + P_QK + j * 16384, 64 * j, row0);
            tma_store_2d(&tm_U, sm + P_V + j * 8192, 64 * j, row0);
        }
        bulk_commit();
        bulk_wait0();
    }
    __syncwarp();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// ---------------------------------------------------------------------------
template <int Vt>
struct ScanPlan {
    static constexpr int STAGE = 57344;         // Q 16K | W 16K | K 16K | Mqk 8K
    static constexpr int S_OP = 2 * STAGE;      // S0^T operand [128 k][Vt] bf16, MN-major, no swizzle
    static constexpr int U_OP = S_OP + kD * Vt * 2;  // U  [64 tok][Vt]
    static constexpr int UH_OP = U_OP + kC * Vt * 2; // Uh [64 tok][Vt]
    static constexpr int BAR = UH_OP + kC * Vt * 2;  // tma[2], mma1, mma2
    static constexpr int END = BAR + 64;
    static constexpr size_t SMEM = END + 1024;
    static constexpr uint32_t TMEM_COLS = (4 * Vt <= 32) ? 32 : (4 * Vt <= 64 ? 64 : (4 * Vt <= 128 ? 128 : 256));
};

template <int Vt>
__global__ void __launch_bounds__(128, 1)
scan_fwd_tc(Dims d, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_W, const __grid_constant__ CUtensorMap tm_M,
            const bf16* __restrict__ Ut, const float* __restrict__ G, const float* s0,
            bf16* __restrict__ o, float* sT, bf16* __restrict__ states, int* err) {
    using P = ScanPlan<Vt>;
    extern __shared__ unsigned char smraw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    uint64_t* tbar = (uint64_t*)(sm + P::BAR);
    uint64_t* bar1 = tbar + 2;
    uint64_t* bar2 = tbar + 3;
    uint32_t* tslot = (uint32_t*)(sm + P::BAR + 32);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int v0 = blockIdx.x * Vt, h = blockIdx.y, b = blockIdx.z;
    const int64_t strm = (int64_t)b * d.H + h;
    const int NC = d.NC;

    auto issue_loads = [&](int c) {
        unsigned char* st = sm + (c & 1) * P::STAGE;
        const int row = (int)((strm * NC + c) * kC);
        mbar_arrive_expect_tx(&tbar[c & 1], 7 * 8192);
        for (int j = 0; j < 2; ++j) {
            tma_load_4d(st + j * 8192, &tm_q, &tbar[c & 1], 64 * j, h, c * kC, b);
            tma_load_2d(st + 16384 + j * 8192, &tm_W, &tbar[c & 1], 64 * j, row);
            tma_load_4d(st + 32768 + j * 8192, &tm_k, &tbar[c & 1], 64 * j, h, c * kC, b);
        }
        tma_load_2d(st + 49152, &tm_M, &tbar[c & 1], 0, row);
    };

    if (tid == 0) {
        mbar_init(&tbar[0], 1);
        mbar_init(&tbar[1], 1);
        mbar_init(bar1, 1);
        mbar_init(bar2, 1);
        fence_mbar_init();
        issue_loads(0);
        if (NC > 1) issue_loads(1);
    }
    if (warp == 0) {
        tmem_alloc(tslot, P::TMEM_COLS);
        tmem_relinquish();
    }
    // State slice: thread k holds S[v0 + v][k], v < Vt.
    const int k = tid;
    float s[Vt];
#pragma unroll
    for (int v = 0; v < Vt; ++v) s[v] = s0 ? s0[(strm * d.V + v0 + v) * kD + k] : 0.f;
    auto write_state_operand = [&]() {
        // MN-major, no swizzle: element (v, k) at (v/8)*2048 + k*16 + (v%8)*2
#pragma unroll
        for (int g = 0; g < Vt / 8; ++g) {
            uint4 pk = make_uint4(pack_bf16(s[8 * g + 0], s[8 * g + 1]), pack_bf16(s[8 * g + 2], s[8 * g + 3]),
                                  pack_bf16(s[8 * g + 4], s[8 * g + 5]), pack_bf16(s[8 * g + 6], s[8 * g + 7]));
            *(uint4*)(sm + P::S_OP + g * 2048 + k * 16) = pk;
        }
    };
    write_state_operand();
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t tY = tmem, tX = tmem + Vt, tO = tmem + 2 * Vt, tS = tmem + 3 * Vt;
    const uint32_t lanebase = (uint32_t)(warp * 32) << 16;
    const int r = warp * 16 + (lane & 15);  // token row of this thread in the M=64 results
    const bool rowthr = lane < 16;

    bool ok = true;
    int c = 0;
#pragma unroll 1
    for (; c < NC; ++c) {
        const int stg = c & 1;
        unsigned char* st = sm + stg * P::STAGE;
        const int64_t chunk = strm * NC + c;
        const int t0 = c * kC;
        // chunk-start state -> saved boundary states
        if (states) {  // bf16, [chunk][k][v]: this thread's row k, columns v0 .. v0+Vt
            uint4* St = (uint4*)(states + (chunk * kD + k) * d.V + v0);
#pragma unroll
            for (int g = 0; g < Vt / 8; ++g)
                St[g] = make_uint4(pack_bf16(s[8 * g + 0], s[8 * g + 1]), pack_bf16(s[8 * g + 2], s[8 * g + 3]),
                                   pack_bf16(s[8 * g + 4], s[8 * g + 5]), pack_bf16(s[8 * g + 6], s[8 * g + 7]));
        }
        if (tid == 0) {
            bool okt = mbar_wait(&tbar[stg], (c >> 1) & 1, err, 8);
            if (okt) {
                const uint32_t id = idesc_bf16(64, Vt, false, true);
                const uint32_t qb = smem_u32(st), wb = smem_u32(st + 16384), sb = smem_u32(sm + P::S_OP);
#pragma unroll
                for (int s2 = 0; s2 < 8; ++s2) {
                    const uint64_t bd = sdesc(sb + s2 * 256, 128, 2048, SW_NONE);
                    const uint32_t ao = (s2 >> 2) * 8192 + (s2 & 3) * 32;
                    mma_bf16_ss(tY, sdesc(qb + ao, 16, 1024, SW_128B), bd, id, s2 > 0);
                    mma_bf16_ss(tX, sdesc(wb + ao, 16, 1024, SW_128B), bd, id, s2 > 0);
                }
                mma_commit(bar1);
            }
        }
        // per-row inputs of this chunk (overlap with the MMA)
        const float* Gc = G + chunk * kC;
        const float GC = Gc[kC - 1];
        const float gC = expf(GC);
        const float Gr = Gc[r];
        const float gr = expf(Gr), er = expf(GC - Gr);
        uint32_t utr[Vt / 2];
        {
            const uint4* up = (const uint4*)(Ut + (chunk * kC + r) * (int64_t)d.V + v0);
#pragma unroll
            for (int q = 0; q < Vt / 8; ++q) {
                uint4 x = up[q];
                utr[4 * q + 0] = x.x; utr[4 * q + 1] = x.y; utr[4 * q + 2] = x.z; utr[4 * q + 3] = x.w;
            }
        }
        ok = mbar_wait(bar1, c & 1, err, 16) && ok;
        __syncwarp();
        fence_after_sync();
        // U = Ut - X, Uh = e_r U  (row r, threads with lane < 16); Y kept as gamma_r Y.
        float y[Vt];
#pragma unroll
        for (int c0 = 0; c0 < Vt; c0 += 16) {
            uint32_t xv[16], yv[16];
            tmem_ld16(tX + lanebase + c0, xv);
            tmem_ld16(tY + lanebase + c0, yv);
            tmem_wait_ld(xv);
            tmem_wait_ld(yv);
            uint32_t pu[8], ph[8];
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
                const uint32_t uw = utr[(c0 + j) >> 1];
                const float u0 = bf_lo(uw) - __uint_as_float(xv[j]);
                const float u1 = bf_hi(uw) - __uint_as_float(xv[j + 1]);
                pu[j >> 1] = pack_bf16(u0, u1);
                ph[j >> 1] = pack_bf16(er * u0, er * u1);
                y[c0 + j] = gr * __uint_as_float(yv[j]);
                y[c0 + j + 1] = gr * __uint_as_float(yv[j + 1]);
            }
            if (rowthr) {
                // MN-major, no swizzle: element (v, r) at (v/8)*1024 + r*16 + (v%8)*2
                *(uint4*)(sm + P::U_OP + ((c0 >> 3) + 0) * 1024 + r * 16) = make_uint4(pu[0], pu[1], pu[2], pu[3]);
                *(uint4*)(sm + P::U_OP + ((c0 >> 3) + 1) * 1024 + r * 16) = make_uint4(pu[4], pu[5], pu[6], pu[7]);
                *(uint4*)(sm + P::UH_OP + ((c0 >> 3) + 0) * 1024 + r * 16) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
                *(uint4*)(sm + P::UH_OP + ((c0 >> 3) + 1) * 1024 + r * 16) = make_uint4(ph[4], ph[5], ph[6], ph[7]);
            }
        }
        fence_proxy_async();
        fence_before_sync();
        ok = __syncthreads_and(ok);
        if (!ok) break;
        fence_after_sync();
        if (tid == 0) {
            const uint32_t ub = smem_u32(sm + P::U_OP), uhb = smem_u32(sm + P::UH_OP);
            const uint32_t mb = smem_u32(st + 49152), kb = smem_u32(st + 32768);
            const uint32_t id2 = idesc_bf16(64, Vt, false, true);
            const uint32_t id3 = idesc_bf16(128, Vt, true, true);
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2) {
                mma_bf16_ss(tO, sdesc(mb + s2 * 32, 16, 1024, SW_128B), sdesc(ub + s2 * 256, 128, 1024, SW_NONE),
                            id2, s2 > 0);
                mma_bf16_ss(tS, sdesc(kb + s2 * 2048, 8192, 1024, SW_128B),
                            sdesc(uhb + s2 * 256, 128, 1024, SW_NONE), id3, s2 > 0);
            }
            mma_commit(bar2);
        }
        ok = mbar_wait(bar2, c & 1, err, 32) && ok;
        fence_after_sync();
        if (tid == 0 && ok && c + 2 < NC) issue_loads(c + 2);
        __syncwarp();
        // O = gamma Y + Mqk U
#pragma unroll
        for (int c0 = 0; c0 < Vt; c0 += 16) {
            uint32_t ov[16];
            tmem_ld16(tO + lanebase + c0, ov);
            tmem_wait_ld(ov);
            if (o && rowthr && t0 + r < d.T) {
                uint32_t po[8];
#pragma unroll
                for (int j = 0; j < 16; j += 2)
                    po[j >> 1] = pack_bf16(y[c0 + j] + __uint_as_float(ov[j]), y[c0 + j + 1] + __uint_as_float(ov[j + 1]));
                uint4* op = (uint4*)(o + (((int64_t)b * d.T + t0 + r) * d.H + h) * d.V + v0 + c0);
                op[0] = make_uint4(po[0], po[1], po[2], po[3]);
                op[1] = make_uint4(po[4], po[5], po[6], po[7]);
            }
        }
        // S1^T = gamma_C S0^T + K^T Uh  (thread k = lane of the M=128 result)
#pragma unroll
        for (int c0 = 0; c0 < Vt; c0 += 16) {
            uint32_t sv[16];
            tmem_ld16(tS + lanebase + c0, sv);
            tmem_wait_ld(sv);
#pragma unroll
            for (int j = 0; j < 16; ++j) s[c0 + j] = gC * s[c0 + j] + __uint_as_float(sv[j]);
        }
        write_state_operand();
        fence_proxy_async();
        fence_before_sync();
        ok = __syncthreads_and(ok);
        if (!ok) break;
        fence_after_sync();
    }
    if (ok && sT) {
#pragma unroll
        for (int v = 0; v < Vt; ++v) sT[(strm * d.V + v0 + v) * kD + k] = s[v];
    }
    if (!ok && tid == 0) {
        // drain the loads still in flight (bounded) before leaving
        for (int cc = c; cc < NC && cc < c + 2; ++cc) mbar_wait(&tbar[cc & 1], (cc >> 1) & 1, nullptr, 0);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, P::TMEM_COLS);
}

template <int Vt>
cudaError_t launch_scan_vt(const Dims& d, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mW,
                           const CUtensorMap& mM, const TcBufs& tb, const float* s0, void* o, float* sT,
                           bf16* states, cudaStream_t st) {
    using P = ScanPlan<Vt>;
    auto kern = scan_fwd_tc<Vt>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(kD / Vt, d.H, d.B);
    kern<<<grid, 128, P::SMEM, st>>>(d, mq, mk, mW, mM, tb.Ut, tb.G, s0, (bf16*)o, sT, states, tb.err);
    return cudaGetLastError();
}

}  // namespace

bool tc_fwd_supported(const Dims& d, InType ty) {
    return ty == InType::BF16 && d.K == kD && d.V == kD && d.C == kC;
}

int tc_scan_vt(const Dims& d) {
    const int64_t sms = sm_count();
    for (int vt : {16, 32, 64})
        if (d.NS() * (kD / vt) <= sms) return vt;
    return 64;
}

cudaError_t launch_prep_tc(const Dims& d, const void* q, const void* k, const void* v, const void* alpha,
                           const void* beta, const TcBufs& tb, cudaStream_t st) {
    CUtensorMap mq, mk, mv, mW, mU, mM;
    const int64_t rows = d.NS() * d.NC * kC;
    if (!tmap_bthd(&mq, q, d.B, d.T, d.H, kD) || !tmap_bthd(&mk, k, d.B, d.T, d.H, kD) ||
        !tmap_bthd(&mv, v, d.B, d.T, d.H, kD) || !tmap_rows(&mW, tb.W, rows, kD) ||
        !tmap_rows(&mU, tb.Ut, rows, kD) || !tmap_rows(&mM, tb.Mqk, rows, kC))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(prep_fwd_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrepSmem);
    if (e != cudaSuccess) return e;
    dim3 grid(d.NC, d.H, d.B);
    prep_fwd_tc<<<grid, 128, kPrepSmem, st>>>(d, mq, mk, mv, mW, mU, mM, (const bf16*)alpha, (const bf16*)beta,
                                              tb.G, tb.T, tb.err);
    return cudaGetLastError();
}

cudaError_t launch_scan_fwd_tc(const Dims& d, const void* q, const void* k, const TcBufs& tb, const float* s0,
                               void* o, float* sT, __nv_bfloat16* states, cudaStream_t st) {
    CUtensorMap mq, mk, mW, mM;
    const int64_t rows = d.NS() * d.NC * kC;
    if (!tmap_bthd(&mq, q, d.B, d.T, d.H, kD) || !tmap_bthd(&mk, k, d.B, d.T, d.H, kD) ||
        !tmap_rows(&mW, tb.W, rows, kD) || !tmap_rows(&mM, tb.Mqk, rows, kC))
        return cudaErrorInvalidValue;
    switch (tc_scan_vt(d)) {
        case 16: return launch_scan_vt<16>(d, mq, mk, mW, mM, tb, s0, o, sT, states, st);
        case 32: return launch_scan_vt<32>(d, mq, mk, mW, mM, tb, s0, o, sT, states, st);
        default: return launch_scan_vt<64>(d, mq, mk, mW, mM, tb, s0, o, sT, states, st);
    }
}

}  // namespace gdn
