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

#include <cstring>

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
    // stage: [W_0 | Q_0 | W_1 | Q_1] (stacked A of one M=128 MMA) | K_0 | K_1 | Mqk | Ut slice
    static constexpr int OFF_WQ = 0, OFF_K = 32768, OFF_M = 49152, OFF_UT = 57344;
    static constexpr int STAGE = 57344 + kC * Vt * 2;
    static constexpr int S_OP = 2 * STAGE;           // S0^T [Vt/8][128 k][8] (MN-major, no swizzle)
    static constexpr int U_OP = S_OP + kD * Vt * 2;  // U  [Vt/8][64 tok][8]
    static constexpr int UH_OP = U_OP + kC * Vt * 2; // Uh
    static constexpr int O_OP = UH_OP + kC * Vt * 2; // output tile, same layout
    static constexpr int BAR = O_OP + kC * Vt * 2;   // tma[2], XY, S, O
    static constexpr int END = BAR + 64;
    static constexpr size_t SMEM = END + 1024;
    // TMEM: [X;Y] (two buffers), O2, DS, each Vt columns
    static constexpr uint32_t TMEM_COLS = (4 * Vt <= 32) ? 32 : (4 * Vt <= 64 ? 64 : (4 * Vt <= 128 ? 128 : 256));
};

// Loads W consecutive fp32 TMEM columns (W = 16 or 32) of this thread's lane.
template <int W>
__device__ __forceinline__ void tmem_cols(uint32_t taddr, float* f) {
    if constexpr (W == 16) {
        uint32_t r[16];
        tmem_ld16(taddr, r);
        tmem_wait_ld(r);
#pragma unroll
        for (int j = 0; j < 16; ++j) f[j] = __uint_as_float(r[j]);
    } else {
        uint32_t r[32];
        tmem_ld32(taddr, r);
        tmem_wait_ld(r);
#pragma unroll
        for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(r[j]);
    }
}
// Two W-column groups, one wait.
template <int W>
__device__ __forceinline__ void tmem_cols2(uint32_t ta, uint32_t tb, float* fa, float* fb) {
    if constexpr (W == 16) {
        uint32_t a[16], b2[16];
        tmem_ld16(ta, a);
        tmem_ld16(tb, b2);
        tmem_wait_ld(a);
        tmem_wait_ld(b2);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            fa[j] = __uint_as_float(a[j]);
            fb[j] = __uint_as_float(b2[j]);
        }
    } else {
        uint32_t a[32], b2[32];
        tmem_ld32x2(ta, tb, a, b2);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            fa[j] = __uint_as_float(a[j]);
            fb[j] = __uint_as_float(b2[j]);
        }
    }
}

// 256 threads.  Warp w reaches TMEM lanes 32*(w%4) ..; warps w and w+4 split the
// columns.  Lanes 0-63 hold X = W S0^T (rows of U), lanes 64-127 hold Y = Q S0^T
// and the output term; the state update uses all 128 lanes (rows k).
template <int Vt>
__global__ void __launch_bounds__(256, 1)
scan_fwd_tc(Dims d, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_W, const __grid_constant__ CUtensorMap tm_M,
            const __grid_constant__ CUtensorMap tm_Ut, const __grid_constant__ CUtensorMap tm_o,
            const __grid_constant__ CUtensorMap tm_st, const float* __restrict__ G, const float* s0,
            float* sT, int write_o, int write_states, int* err) {
    using P = ScanPlan<Vt>;
    constexpr int HV = Vt / 2;  // columns per thread
    extern __shared__ unsigned char smraw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    uint64_t* tbar = (uint64_t*)(sm + P::BAR);
    uint64_t* barXY = tbar + 2;
    uint64_t* barS = tbar + 3;
    uint64_t* barO = tbar + 4;
    uint32_t* tslot = (uint32_t*)(sm + P::BAR + 48);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sub = warp & 3, half = warp >> 2;
    const int lanerow = 32 * sub + lane;  // TMEM lane of this thread
    const int cb = half * HV;             // first column of this thread
    const bool issuer = tid == 96;        // warp 3 (output side) issues MMAs and copies
    const int v0 = blockIdx.x * Vt, h = blockIdx.y, b = blockIdx.z;
    const int64_t strm = (int64_t)b * d.H + h;
    const int NC = d.NC;

    auto issue_loads = [&](int c) {
        unsigned char* st = sm + (c & 1) * P::STAGE;
        const int row = (int)((strm * NC + c) * kC);
        uint64_t* bar = &tbar[c & 1];
        mbar_arrive_expect_tx(bar, 7 * 8192 + kC * Vt * 2);
        for (int j = 0; j < 2; ++j) {
            tma_load_2d(st + P::OFF_WQ + j * 16384, &tm_W, bar, 64 * j, row);
            tma_load_4d(st + P::OFF_WQ + j * 16384 + 8192, &tm_q, bar, 64 * j, h, c * kC, b);
            tma_load_4d(st + P::OFF_K + j * 8192, &tm_k, bar, 64 * j, h, c * kC, b);
        }
        tma_load_2d(st + P::OFF_M, &tm_M, bar, 0, row);
        tma_load_3d(st + P::OFF_UT, &tm_Ut, bar, 0, row, v0 / 8);
    };

    if (issuer) {
        for (int i = 0; i < 5; ++i) mbar_init(&tbar[i], 1);
        fence_mbar_init();
        issue_loads(0);
        if (NC > 1) issue_loads(1);
    }
    if (warp == 0) {
        tmem_alloc(tslot, P::TMEM_COLS);
        tmem_relinquish();
    }
    // State: thread holds S[v0 + cb + j][k = lanerow], j < HV.
    const int k = lanerow;
    float s[HV];
#pragma unroll
    for (int j = 0; j < HV; ++j) s[j] = s0 ? s0[(strm * d.V + v0 + cb + j) * kD + k] : 0.f;
    auto write_state_operand = [&]() {
        // MN-major, no swizzle: element (v, k) at (v/8)*2048 + k*16 + (v%8)*2
#pragma unroll
        for (int g = 0; g < HV / 8; ++g)
            *(uint4*)(sm + P::S_OP + (cb / 8 + g) * 2048 + k * 16) =
                make_uint4(pack_bf16(s[8 * g + 0], s[8 * g + 1]), pack_bf16(s[8 * g + 2], s[8 * g + 3]),
                           pack_bf16(s[8 * g + 4], s[8 * g + 5]), pack_bf16(s[8 * g + 6], s[8 * g + 7]));
    };
    write_state_operand();
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t tXY0 = tmem, tO = tmem + 2 * Vt, tS = tmem + 3 * Vt;
    const uint32_t lanebase = (uint32_t)(sub * 32) << 16;
    const bool urow = sub < 2;            // lanes 0-63: rows of U (r = lanerow)
    const int r = urow ? lanerow : lanerow - 64;  // token row (both sides)

    const uint64_t dS = sdesc(smem_u32(sm + P::S_OP), 128, 2048, SW_NONE);
    const uint64_t dU = sdesc(smem_u32(sm + P::U_OP), 128, 1024, SW_NONE);
    const uint64_t dUh = sdesc(smem_u32(sm + P::UH_OP), 128, 1024, SW_NONE);
    const uint32_t id = idesc_bf16(128, Vt, false, true);
    const uint32_t idmn = idesc_bf16(128, Vt, true, true);

    float GC_n = G[strm * NC * kC + kC - 1], Gr_n = G[strm * NC * kC + r];
    float gr_prev = 0.f;

    // Output of chunk cc (threads on lanes 64-127): O = gamma Y + Mqk U.
    auto output_epilogue = [&](int cc, bool& okk) {
        okk = mbar_wait(barO, cc & 1, err, 64) && okk;
        __syncwarp();
        fence_after_sync();
        if (issuer && okk && cc + 2 < NC) issue_loads(cc + 2);
        __syncwarp();
        float y[HV], ov[HV];
        if constexpr (HV == 8) {
            uint32_t a[8], b2[8];
            // two 8-column halves through the x16 loader would over-read; use the
            // x16 load on a 16-column window and keep our half
            uint32_t wa[16], wb[16];
            tmem_ld16(tXY0 + (uint32_t)((cc & 1) * Vt) + lanebase, wa);
            tmem_ld16(tO + lanebase, wb);
            tmem_wait_ld(wa);
            tmem_wait_ld(wb);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                a[j] = half ? wa[8 + j] : wa[j];
                b2[j] = half ? wb[8 + j] : wb[j];
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                y[j] = __uint_as_float(a[j]);
                ov[j] = __uint_as_float(b2[j]);
            }
        } else {
            tmem_cols2<HV>(tXY0 + (uint32_t)((cc & 1) * Vt) + lanebase + cb, tO + lanebase + cb, y, ov);
        }
#pragma unroll
        for (int g = 0; g < HV / 8; ++g) {
            float f[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = gr_prev * y[8 * g + j] + ov[8 * g + j];
            *(uint4*)(sm + P::O_OP + (cb / 8 + g) * 1024 + r * 16) =
                make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]),
                           pack_bf16(f[6], f[7]));
        }
    };

    bool ok = true;
    int c = 0;
#pragma unroll 1
    for (; c < NC; ++c) {
        const int stg = c & 1;
        unsigned char* st = sm + stg * P::STAGE;
        const int64_t chunk = strm * NC + c;
        if (issuer) {
            if (write_states) {  // chunk-start state -> saved boundary states, by TMA
                tma_store_3d(&tm_st, sm + P::S_OP, 0, (int)(chunk * kD), v0 / 8);
                bulk_commit();
            }
            const bool okt = mbar_wait(&tbar[stg], (c >> 1) & 1, err, 8);
            if (okt) {
                // [X; Y] = [W; Q] S0^T in one M=128 MMA chain
                const uint64_t dWQ = sdesc(smem_u32(st + P::OFF_WQ), 16, 1024, SW_128B);
#pragma unroll
                for (int s2 = 0; s2 < 8; ++s2)
                    mma_bf16_ss(tXY0 + (uint32_t)(stg * Vt), desc_add(dWQ, (s2 >> 2) * 16384 + (s2 & 3) * 32),
                                desc_add(dS, s2 * 256), id, s2 > 0);
                mma_commit(barXY);
            }
        }
        const float GC = GC_n;
        const float gC = expf(GC);
        const float Gr = Gr_n;
        const float gr = expf(Gr), er = expf(GC - Gr);
        if (c + 1 < NC) {
            GC_n = G[(chunk + 1) * kC + kC - 1];
            Gr_n = G[(chunk + 1) * kC + r];
        }
        if (!urow && c > 0) output_epilogue(c - 1, ok);  // overlaps this chunk's first MMAs
        gr_prev = gr;
        if (urow) {
            ok = mbar_wait(&tbar[stg], (c >> 1) & 1, err, 8) && ok;  // Ut slice is read below
            ok = mbar_wait(barXY, c & 1, err, 16) && ok;
            __syncwarp();
            fence_after_sync();
            // U = Ut - X, Uh = e_r U  (row r, columns cb .. cb+HV)
            float xg[HV];
            if constexpr (HV == 8) {
                uint32_t w16[16];
                tmem_ld16(tXY0 + (uint32_t)(stg * Vt) + lanebase, w16);
                tmem_wait_ld(w16);
#pragma unroll
                for (int j = 0; j < 8; ++j) xg[j] = __uint_as_float(half ? w16[8 + j] : w16[j]);
            } else {
                tmem_cols<HV>(tXY0 + (uint32_t)(stg * Vt) + lanebase + cb, xg);
            }
#pragma unroll
            for (int g = 0; g < HV / 8; ++g) {
                const int gg = cb / 8 + g;
                const uint4 uq = *(const uint4*)(st + P::OFF_UT + gg * 1024 + r * 16);
                const uint32_t uw4[4] = {uq.x, uq.y, uq.z, uq.w};
                float u[8], uh[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    u[2 * e] = bf_lo(uw4[e]) - xg[8 * g + 2 * e];
                    u[2 * e + 1] = bf_hi(uw4[e]) - xg[8 * g + 2 * e + 1];
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) uh[j] = er * u[j];
                // MN-major, no swizzle: element (v, r) at (v/8)*1024 + r*16 + (v%8)*2
                *(uint4*)(sm + P::U_OP + gg * 1024 + r * 16) =
                    make_uint4(pack_bf16(u[0], u[1]), pack_bf16(u[2], u[3]), pack_bf16(u[4], u[5]), pack_bf16(u[6], u[7]));
                *(uint4*)(sm + P::UH_OP + gg * 1024 + r * 16) =
                    make_uint4(pack_bf16(uh[0], uh[1]), pack_bf16(uh[2], uh[3]), pack_bf16(uh[4], uh[5]), pack_bf16(uh[6], uh[7]));
            }
        }
        fence_proxy_async();
        fence_before_sync();
        if (issuer) bulk_wait_read0();  // the states store no longer reads S0^T
        ok = __syncthreads_and(ok);
        if (!ok) break;
        fence_after_sync();
        if (issuer) {
            if (c > 0 && write_o) {  // output tile of the previous chunk
                tma_store_5d(&tm_o, sm + P::O_OP, 0, (c - 1) * kC, v0 / 8, h, b);
                bulk_commit();
            }
            const uint64_t dK = sdesc(smem_u32(st + P::OFF_K), 8192, 1024, SW_128B);
            // rows 0-63 of this A are the K_1 block (unused rows), rows 64-127 are Mqk
            const uint64_t dM = sdesc(smem_u32(st + P::OFF_K + 8192), 16, 1024, SW_128B);
            // S1^T update first (critical), then the output term
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2)
                mma_bf16_ss(tS, desc_add(dK, s2 * 2048), desc_add(dUh, s2 * 256), idmn, s2 > 0);
            mma_commit(barS);
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2)
                mma_bf16_ss(tO, desc_add(dM, s2 * 32), desc_add(dU, s2 * 256), id, s2 > 0);
            mma_commit(barO);
        }
        ok = mbar_wait(barS, c & 1, err, 32) && ok;
        __syncwarp();
        fence_after_sync();
        // S1^T = gamma_C S0^T + K^T Uh
        {
            float sv[HV];
            if constexpr (HV == 8) {
                uint32_t w16[16];
                tmem_ld16(tS + lanebase, w16);
                tmem_wait_ld(w16);
#pragma unroll
                for (int j = 0; j < 8; ++j) sv[j] = __uint_as_float(half ? w16[8 + j] : w16[j]);
            } else {
                tmem_cols<HV>(tS + lanebase + cb, sv);
            }
#pragma unroll
            for (int j = 0; j < HV; ++j) s[j] = gC * s[j] + sv[j];
        }
        write_state_operand();
        fence_proxy_async();
        fence_before_sync();
        if (issuer) bulk_wait_read0();  // the output store no longer reads the O tile
        ok = __syncthreads_and(ok);
        if (!ok) break;
        fence_after_sync();
    }
    if (ok && NC > 0) {
        if (!urow) output_epilogue(NC - 1, ok);
        fence_proxy_async();
        fence_before_sync();
        ok = __syncthreads_and(ok);
        if (issuer && ok && write_o) {
            tma_store_5d(&tm_o, sm + P::O_OP, 0, (NC - 1) * kC, v0 / 8, h, b);
            bulk_commit();
        }
    }
    if (ok && sT) {
#pragma unroll
        for (int j = 0; j < HV; ++j) sT[(strm * d.V + v0 + cb + j) * kD + k] = s[j];
    }
    if (issuer) {
        if (!ok) {
            // drain what may still be in flight (bounded) before leaving
            for (int cc = c; cc < NC && cc < c + 2; ++cc) mbar_wait(&tbar[cc & 1], (cc >> 1) & 1, nullptr, 0);
            mbar_wait(barO, (c > 0 ? c - 1 : 0) & 1, nullptr, 0);
        }
        bulk_wait0();
    }
    __syncwarp();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, P::TMEM_COLS);
}

template <int Vt>
cudaError_t launch_scan_vt(const Dims& d, const void* q, const void* k, const TcBufs& tb, const float* s0,
                           void* o, float* sT, bf16* states, cudaStream_t st) {
    using P = ScanPlan<Vt>;
    CUtensorMap mq, mk, mW, mM, mUt, mo, mst;
    const int64_t rows = d.NS() * d.NC * kC;
    if (!tmap_bthd(&mq, q, d.B, d.T, d.H, kD) || !tmap_bthd(&mk, k, d.B, d.T, d.H, kD) ||
        !tmap_rows(&mW, tb.W, rows, kD) || !tmap_rows(&mM, tb.Mqk, rows, kC) ||
        !tmap_core8_rows(&mUt, tb.Ut, rows, kD, kC, Vt / 8))
        return cudaErrorInvalidValue;
    memset(&mo, 0, sizeof(mo));
    memset(&mst, 0, sizeof(mst));
    if (o && !tmap_core8_bthd(&mo, o, d.B, d.T, d.H, kD, Vt / 8)) return cudaErrorInvalidValue;
    if (states && !tmap_core8_rows(&mst, states, d.NS() * d.NC * kD, kD, kD, Vt / 8))
        return cudaErrorInvalidValue;
    auto kern = scan_fwd_tc<Vt>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(kD / Vt, d.H, d.B);
    kern<<<grid, 256, P::SMEM, st>>>(d, mq, mk, mW, mM, mUt, mo, mst, tb.G, s0, sT, o != nullptr,
                                     states != nullptr, tb.err);
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
    switch (tc_scan_vt(d)) {
        case 16: return launch_scan_vt<16>(d, q, k, tb, s0, o, sT, states, st);
        case 32: return launch_scan_vt<32>(d, q, k, tb, s0, o, sT, states, st);
        default: return launch_scan_vt<64>(d, q, k, tb, s0, o, sT, states, st);
    }
}

}  // namespace gdn
