// tc_bwd.cu -- tensor-core (tcgen05 + TMA) backward for bf16 inputs, K = V = 128,
// chunk 64 ("Sparse Delta Memory: layer and kernels", "What the layer computes":
// the backward walks the chunks in reverse; "OpenGDN", "Core operator
// reference": the reverse keeps chunk-boundary states and recomputes the 64x64
// systems).  Three kernels after the chunk recompute (prep_fwd_tc with T):
//
// scan_bwd_tc (one CTA per (V-slice, head, batch), chunks in reverse order; the
// gradient of the chunk's end state dS1^T [K, Vt] lives in registers):
//     dU   = Mqk^T dO + diag(exp(G_C - G)) K dS1^T
//     dS0^T = gamma_C dS1^T + Q^T diag(gamma) dO - W^T dU
//   writes dU and dS1 (bf16) per chunk and d(initial state).
//
// grad_qk_tc (one CTA per chunk): U = Ut - W S0^T, then
//     dMqk = dO U^T,   dQK = Gam .* lower(dMqk)
//     dQ^T = S0^T (diag(gamma) dO)^T + K^T dQK^T                 -> dq
//     dK^T (part) = dS1^T (diag(e) U)^T + Q^T dQK                -> scratch
//     dW^T = -S0^T dU^T                                          -> scratch
//     dG (part): gamma in O, Gam in Mqk, exp(G_C - G) in Khat, gamma_C in S1.
//
// grad_wy_tc (one CTA per chunk), through T = (I + A)^-1:
//     Qm = dW K^T,  P = dU V^T,  dT = strict_lower(diag(beta)(P + Qm diag(gamma)))^T-wise
//     dA = strict_lower(-T^T (dT T^T)),  E = diag(beta)(Gam .* dA)
//     dV^T = dU^T T diag(beta)                                   -> dv
//     dK^T = dK^T (part) + dW^T T diag(beta gamma) + K^T (E + E^T) -> dk
//     dbeta, dG (rest), dlog alpha = reverse cumsum of dG, dalpha = dlog alpha / alpha.
//
// Every wait is bounded (2 s) and raises the error flag when it gives up.

#include "gdn_internal.h"
#include "tc.cuh"

namespace gdn {
namespace {

using namespace tc;
using bf16 = __nv_bfloat16;

constexpr int kC = 64;
constexpr int kD = 128;

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

__device__ __forceinline__ uint4 pack8(const float* f) {
    return make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]),
                      pack_bf16(f[6], f[7]));
}

// ============================================================ reverse scan
template <int Vt>
struct BScan {
    static constexpr int STAGE = 57344;              // Mqk 8K | K 16K | Q 16K | W 16K
    static constexpr int OFF_M = 0, OFF_K = 8192, OFF_Q = 24576, OFF_W = 40960;
    static constexpr int DS_OP = 2 * STAGE;          // dS1^T [128 k][Vt], MN-major, no swizzle
    static constexpr int DO_OP = DS_OP + kD * Vt * 2;  // dO [64 s][Vt]
    static constexpr int GDO_OP = DO_OP + kC * Vt * 2; // gamma dO
    static constexpr int DU_OP = GDO_OP + kC * Vt * 2; // dU
    static constexpr int BAR = DU_OP + kC * Vt * 2;
    static constexpr size_t SMEM = BAR + 64 + 1024;
    static constexpr uint32_t TMEM_COLS = (3 * Vt <= 64) ? 64 : (3 * Vt <= 128 ? 128 : 256);
};

template <int Vt>
__global__ void __launch_bounds__(128, 1)
scan_bwd_tc(Dims d, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_W, const __grid_constant__ CUtensorMap tm_M,
            const bf16* __restrict__ d_o, const float* __restrict__ G, const float* dsT,
            bf16* __restrict__ dU_out, bf16* __restrict__ dS1_out, float* ds0, int* err) {
    using P = BScan<Vt>;
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

    auto issue_loads = [&](int it) {
        const int c = NC - 1 - it;
        unsigned char* st = sm + (it & 1) * P::STAGE;
        uint64_t* bar = &tbar[it & 1];
        const int row = (int)((strm * NC + c) * kC);
        mbar_arrive_expect_tx(bar, 7 * 8192);
        tma_load_2d(st + P::OFF_M, &tm_M, bar, 0, row);
        for (int j = 0; j < 2; ++j) {
            tma_load_4d(st + P::OFF_K + j * 8192, &tm_k, bar, 64 * j, h, c * kC, b);
            tma_load_4d(st + P::OFF_Q + j * 8192, &tm_q, bar, 64 * j, h, c * kC, b);
            tma_load_2d(st + P::OFF_W + j * 8192, &tm_W, bar, 64 * j, row);
        }
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
    const int k = tid;
    float ds[Vt];
#pragma unroll
    for (int v = 0; v < Vt; ++v) ds[v] = dsT ? dsT[(strm * d.V + v0 + v) * kD + k] : 0.f;
    auto write_ds_operand = [&]() {
#pragma unroll
        for (int g = 0; g < Vt / 8; ++g) *(uint4*)(sm + P::DS_OP + g * 2048 + k * 16) = pack8(&ds[8 * g]);
    };
    write_ds_operand();
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t tA = tmem, tB = tmem + Vt, tCc = tmem + 2 * Vt;
    const uint32_t lanebase = (uint32_t)(warp * 32) << 16;
    const int r = warp * 16 + (lane & 15);
    const bool rowthr = lane < 16;

    bool ok = true;
    int it = 0;
#pragma unroll 1
    for (; it < NC; ++it) {
        const int c = NC - 1 - it;
        const int stg = it & 1;
        unsigned char* st = sm + stg * P::STAGE;
        const int64_t chunk = strm * NC + c;
        const int t0 = c * kC;
        const float* Gc = G + chunk * kC;
        const float GC = Gc[kC - 1];
        const float gC = expf(GC);
        const float Gr = Gc[r];
        const float gr = expf(Gr), er = expf(GC - Gr);
        // dO row r of this slice -> operands dO and gamma dO (MN-major, no swizzle)
        {
            uint32_t dor[Vt / 2];
            if (t0 + r < d.T) {
                const uint4* p = (const uint4*)(d_o + (((int64_t)b * d.T + t0 + r) * d.H + h) * d.V + v0);
#pragma unroll
                for (int q = 0; q < Vt / 8; ++q) {
                    uint4 x = p[q];
                    dor[4 * q] = x.x; dor[4 * q + 1] = x.y; dor[4 * q + 2] = x.z; dor[4 * q + 3] = x.w;
                }
            } else {
#pragma unroll
                for (int q = 0; q < Vt / 2; ++q) dor[q] = 0u;
            }
            if (rowthr) {
#pragma unroll
                for (int g = 0; g < Vt / 8; ++g) {
                    *(uint4*)(sm + P::DO_OP + g * 1024 + r * 16) =
                        make_uint4(dor[4 * g], dor[4 * g + 1], dor[4 * g + 2], dor[4 * g + 3]);
                    float f[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        f[2 * e] = gr * bf_lo(dor[4 * g + e]);
                        f[2 * e + 1] = gr * bf_hi(dor[4 * g + e]);
                    }
                    *(uint4*)(sm + P::GDO_OP + g * 1024 + r * 16) = pack8(f);
                }
            }
        }
        // the gradient of this chunk's end state, for the chunk-local gradients
        {
            uint4* dst = (uint4*)(dS1_out + (chunk * kD + k) * d.V + v0);
#pragma unroll
            for (int g = 0; g < Vt / 8; ++g) dst[g] = pack8(&ds[8 * g]);
        }
        fence_proxy_async();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        if (tid == 0) {
            const bool okt = mbar_wait(&tbar[stg], (it >> 1) & 1, err, 8);
            if (okt) {
                const uint32_t mb = smem_u32(st + P::OFF_M), kb = smem_u32(st + P::OFF_K);
                const uint32_t qb = smem_u32(st + P::OFF_Q);
                const uint32_t dob = smem_u32(sm + P::DO_OP), gdob = smem_u32(sm + P::GDO_OP);
                const uint32_t dsb = smem_u32(sm + P::DS_OP);
                const uint32_t ida = idesc_bf16(64, Vt, true, true);
                const uint32_t idb = idesc_bf16(64, Vt, false, true);
                const uint32_t idc = idesc_bf16(128, Vt, true, true);
#pragma unroll
                for (int s2 = 0; s2 < 8; ++s2)
                    mma_bf16_ss(tB, desc_kmaj(kb, 64, s2), sdesc(dsb + s2 * 256, 128, 2048, SW_NONE), idb, s2 > 0);
#pragma unroll
                for (int s2 = 0; s2 < 4; ++s2) {
                    mma_bf16_ss(tA, desc_mnmaj(mb, 64, s2), sdesc(dob + s2 * 256, 128, 1024, SW_NONE), ida, s2 > 0);
                    mma_bf16_ss(tCc, desc_mnmaj(qb, 64, s2), sdesc(gdob + s2 * 256, 128, 1024, SW_NONE), idc,
                                s2 > 0);
                }
                mma_commit(bar1);
            }
        }
        ok = mbar_wait(bar1, it & 1, err, 16) && ok;
        __syncwarp();
        fence_after_sync();
        // dU = Mqk^T dO + e_r (K dS1^T)
#pragma unroll
        for (int c0 = 0; c0 < Vt; c0 += 16) {
            float a[16], bb[16], u[16];
            tmem_load16f(tA + lanebase + c0, a);
            tmem_load16f(tB + lanebase + c0, bb);
#pragma unroll
            for (int j = 0; j < 16; ++j) u[j] = a[j] + er * bb[j];
            if (rowthr) {
                const uint4 lo = pack8(u), hi = pack8(u + 8);
                *(uint4*)(sm + P::DU_OP + (c0 >> 3) * 1024 + r * 16) = lo;
                *(uint4*)(sm + P::DU_OP + ((c0 >> 3) + 1) * 1024 + r * 16) = hi;
                uint4* gp = (uint4*)(dU_out + (chunk * kC + r) * d.V + v0 + c0);
                gp[0] = lo;
                gp[1] = hi;
            }
        }
        fence_proxy_async();
        fence_before_sync();
        ok = __syncthreads_and(ok);
        if (!ok) break;
        fence_after_sync();
        if (tid == 0) {
            const uint32_t wb = smem_u32(st + P::OFF_W), dub = smem_u32(sm + P::DU_OP);
            const uint32_t idd = idesc_bf16(128, Vt, true, true, true);  // -W^T dU
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2)
                mma_bf16_ss(tCc, desc_mnmaj(wb, 64, s2), sdesc(dub + s2 * 256, 128, 1024, SW_NONE), idd, 1u);
            mma_commit(bar2);
        }
        ok = mbar_wait(bar2, it & 1, err, 32) && ok;
        __syncwarp();
        fence_after_sync();
        if (tid == 0 && ok && it + 2 < NC) issue_loads(it + 2);
        __syncwarp();
#pragma unroll
        for (int c0 = 0; c0 < Vt; c0 += 16) {
            float x[16];
            tmem_load16f(tCc + lanebase + c0, x);
#pragma unroll
            for (int j = 0; j < 16; ++j) ds[c0 + j] = gC * ds[c0 + j] + x[j];
        }
        write_ds_operand();
        fence_proxy_async();
        fence_before_sync();
        ok = __syncthreads_and(ok);
        if (!ok) break;
        fence_after_sync();
    }
    if (ok && ds0) {
#pragma unroll
        for (int v = 0; v < Vt; ++v) ds0[(strm * d.V + v0 + v) * kD + k] = ds[v];
    }
    if (!ok && tid == 0) {
        for (int i2 = it; i2 < NC && i2 < it + 2; ++i2) mbar_wait(&tbar[i2 & 1], (i2 >> 1) & 1, nullptr, 0);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, P::TMEM_COLS);
}

// ====================================================== chunk gradients (1)
namespace qk {
constexpr int Q = 0, K = 16384, DO = 32768, W = 49152, DU = 65536;  // [64 x 128] tiles
constexpr int S0 = 81920, DS1 = 114688;                              // [128 x 128] tiles
constexpr int U = 147456, EU = 163840;                               // [64 x 128]
constexpr int DQK = 180224;                                          // [64 x 64]
constexpr int E1 = 188416;                                           // fp32 [64][65]
constexpr int VEC = E1 + 64 * 65 * 4;                                // 8 x 64 floats + 128
constexpr int BAR = VEC + (8 * 64 + 128) * 4;
constexpr size_t SMEM = BAR + 64 + 1024;
}  // namespace qk

__global__ void __launch_bounds__(128, 1)
grad_qk_tc(Dims d, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
           const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_W,
           const __grid_constant__ CUtensorMap tm_dU, const __grid_constant__ CUtensorMap tm_S0,
           const __grid_constant__ CUtensorMap tm_dS1, const __grid_constant__ CUtensorMap tm_dq,
           const bf16* __restrict__ Ut, const bf16* __restrict__ Mqk, const float* __restrict__ G,
           float* __restrict__ dKp, bf16* __restrict__ dWt, float* __restrict__ dGp, int* err) {
    extern __shared__ unsigned char smraw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    float* E1f = (float*)(sm + qk::E1);
    float* Gs = (float*)(sm + qk::VEC);
    float* gs = Gs + 64;
    float* eR = gs + 64;
    float* dG1 = eR + 64;
    float* rE1 = dG1 + 64;
    float* cE1 = rE1 + 64;
    float* red = cE1 + 128;  // 128
    uint64_t* bars = (uint64_t*)(sm + qk::BAR);  // [0] TMA, [1] MMA
    uint32_t* tslot = (uint32_t*)(sm + qk::BAR + 16);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int t0 = c * kC;
    const int64_t chunk = ((int64_t)b * d.H + h) * d.NC + c;
    const int row0 = (int)(chunk * kC);
    const int krow0 = (int)(chunk * kD);

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&bars[0], 18 * 8192);
        for (int j = 0; j < 2; ++j) {
            tma_load_4d(sm + qk::Q + j * 8192, &tm_q, &bars[0], 64 * j, h, t0, b);
            tma_load_4d(sm + qk::K + j * 8192, &tm_k, &bars[0], 64 * j, h, t0, b);
            tma_load_4d(sm + qk::DO + j * 8192, &tm_do, &bars[0], 64 * j, h, t0, b);
            tma_load_2d(sm + qk::W + j * 8192, &tm_W, &bars[0], 64 * j, row0);
            tma_load_2d(sm + qk::DU + j * 8192, &tm_dU, &bars[0], 64 * j, row0);
            for (int i = 0; i < 2; ++i) {
                tma_load_2d(sm + qk::S0 + j * 16384 + i * 8192, &tm_S0, &bars[0], 64 * j, krow0 + 64 * i);
                tma_load_2d(sm + qk::DS1 + j * 16384 + i * 8192, &tm_dS1, &bars[0], 64 * j, krow0 + 64 * i);
            }
        }
    }
    if (warp == 0) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    if (tid < 64) {
        Gs[tid] = G[(int64_t)row0 + tid];
        gs[tid] = expf(Gs[tid]);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t lanebase = (uint32_t)(warp * 32) << 16;
    const int r = warp * 16 + (lane & 15);
    const bool rowthr = lane < 16;
    const float GC = Gs[63], gC = gs[63];
    const float Gr = Gs[r], gr = gs[r], er = expf(GC - Gr);
    const uint32_t sQ = smem_u32(sm + qk::Q), sK = smem_u32(sm + qk::K), sDO = smem_u32(sm + qk::DO);
    const uint32_t sW = smem_u32(sm + qk::W), sDU = smem_u32(sm + qk::DU);
    const uint32_t sS0 = smem_u32(sm + qk::S0), sDS1 = smem_u32(sm + qk::DS1);
    const uint32_t sU = smem_u32(sm + qk::U), sEU = smem_u32(sm + qk::EU), sDQK = smem_u32(sm + qk::DQK);

    bool ok = true;
    // ---- phase 1: X = W S0^T, Y = Q S0^T, Z = K dS1^T   (M=64, N=128, K over k)
    if (tid == 0) {
        ok = mbar_wait(&bars[0], 0, err, 1);
        if (ok) {
            const uint32_t id = idesc_bf16(64, 128, false, true);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                mma_bf16_ss(tmem + 0, desc_kmaj(sW, 64, s), desc_mnmaj(sS0, 128, s), id, s > 0);
                mma_bf16_ss(tmem + 128, desc_kmaj(sQ, 64, s), desc_mnmaj(sS0, 128, s), id, s > 0);
                mma_bf16_ss(tmem + 256, desc_kmaj(sK, 64, s), desc_mnmaj(sDS1, 128, s), id, s > 0);
            }
            mma_commit(&bars[1]);
        }
    }
    ok = mbar_wait(&bars[0], 0, err, 1) && ok;  // every thread reads the dO tile below
    ok = mbar_wait(&bars[1], 0, err, 2) && ok;
    __syncwarp();
    fence_after_sync();
    {
        float eacc = 0.f, gacc = 0.f;
        const uint4* up = (const uint4*)(Ut + ((int64_t)row0 + r) * kD);
#pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 16) {
            float x[16], y[16], z[16], u[16], eu[16], dd[8], de[8];
            tmem_load16f(tmem + 0 + lanebase + c0, x);
            tmem_load16f(tmem + 128 + lanebase + c0, y);
            tmem_load16f(tmem + 256 + lanebase + c0, z);
            const uint4 ua = up[c0 / 8], ub = up[c0 / 8 + 1];
            const uint32_t uw[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                u[2 * j] = bf_lo(uw[j]) - x[2 * j];
                u[2 * j + 1] = bf_hi(uw[j]) - x[2 * j + 1];
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                eu[j] = er * u[j];
                eacc += u[j] * z[j];
            }
            tile_get8(sm + qk::DO, 64, r, c0, dd);
            tile_get8(sm + qk::DO, 64, r, c0 + 8, de);
#pragma unroll
            for (int j = 0; j < 8; ++j) gacc += dd[j] * y[j] + de[j] * y[8 + j];
            if (rowthr) {
                tile_put16(sm + qk::U, 64, r, c0, u);
                tile_put16(sm + qk::EU, 64, r, c0, eu);
            }
        }
        if (rowthr) {
            eR[r] = er * eacc;
            dG1[r] = gr * gacc;
        }
    }
    fence_proxy_async();
    fence_before_sync();
    ok = __syncthreads_and(ok);
    fence_after_sync();
    // ---- phase 2 (K over v): dMqk = dO U^T (M=64); dQ1^T = S0^T dO^T, dW^T = -S0^T dU^T,
    //      dK^T = dS1^T (eU)^T (M=128)
    if (tid == 0 && ok) {
        const uint32_t id64 = idesc_bf16(64, 64, false, false);
        const uint32_t id128 = idesc_bf16(128, 64, false, false);
        const uint32_t id128n = idesc_bf16(128, 64, false, false, true);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            mma_bf16_ss(tmem + 0, desc_kmaj(sDO, 64, s), desc_kmaj(sU, 64, s), id64, s > 0);
            mma_bf16_ss(tmem + 64, desc_kmaj(sS0, 128, s), desc_kmaj(sDO, 64, s), id128, s > 0);
            mma_bf16_ss(tmem + 128, desc_kmaj(sS0, 128, s), desc_kmaj(sDU, 64, s), id128n, s > 0);
            mma_bf16_ss(tmem + 192, desc_kmaj(sDS1, 128, s), desc_kmaj(sEU, 64, s), id128, s > 0);
        }
        mma_commit(&bars[1]);
    }
    {   // <dS1, S0> over the chunk (both tiles share one layout)
        const uint4* a = (const uint4*)(sm + qk::S0) + tid * 16;
        const uint4* bq = (const uint4*)(sm + qk::DS1) + tid * 16;
        float acc = 0.f;
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {
            const uint4 x = a[i], y = bq[i];
            const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) acc += bf_lo(xw[e]) * bf_lo(yw[e]) + bf_hi(xw[e]) * bf_hi(yw[e]);
        }
        red[tid] = acc;
    }
    if (ok) ok = mbar_wait(&bars[1], 1, err, 4);
    __syncwarp();
    fence_after_sync();
    {
        const uint4* mp = (const uint4*)(Mqk + ((int64_t)row0 + r) * kC);
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 16) {
            float dm[16], dq[16];
            tmem_load16f(tmem + 0 + lanebase + c0, dm);
            const uint4 ma = mp[c0 / 8], mb = mp[c0 / 8 + 1];
            const uint32_t mw[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int i = c0 + j;
                const float mq = (j & 1) ? bf_hi(mw[j >> 1]) : bf_lo(mw[j >> 1]);
                if (rowthr) E1f[r * 65 + i] = dm[j] * mq;
                dq[j] = (i <= r) ? expf(Gr - Gs[i]) * dm[j] : 0.f;
            }
            if (rowthr) tile_put16(sm + qk::DQK, 64, r, c0, dq);
        }
        // dW^T row k -> scratch
        uint4* wp = (uint4*)(dWt + ((int64_t)krow0 + tid) * kC);
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 16) {
            float w[16];
            tmem_load16f(tmem + 128 + lanebase + c0, w);
            wp[c0 / 8] = pack8(w);
            wp[c0 / 8 + 1] = pack8(w + 8);
        }
    }
    fence_proxy_async();
    fence_before_sync();
    ok = __syncthreads_and(ok);
    fence_after_sync();
    // ---- phase 3 (K over tokens): dQ2^T = K^T dQK^T;  dK^T += Q^T dQK
    if (tid == 0 && ok) {
        const uint32_t idq = idesc_bf16(128, 64, true, false);
        const uint32_t idk = idesc_bf16(128, 64, true, true);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            mma_bf16_ss(tmem + 256, desc_mnmaj(sK, 64, s), desc_kmaj(sDQK, 64, s), idq, s > 0);
            mma_bf16_ss(tmem + 192, desc_mnmaj(sQ, 64, s), desc_mnmaj(sDQK, 64, s), idk, 1u);
        }
        mma_commit(&bars[1]);
    }
    if (tid < 64) {
        float re = 0.f, ce = 0.f;
        for (int i = 0; i < 64; ++i) {
            re += E1f[tid * 65 + i];
            ce += E1f[i * 65 + tid];
        }
        rE1[tid] = re;
        cE1[tid] = ce;
    }
    if (ok) ok = mbar_wait(&bars[1], 0, err, 4);
    __syncwarp();
    fence_after_sync();
    {
        unsigned char* dqt = sm + qk::S0;  // the S0 tile is dead: dq tile [64 r x 128 k]
        float* kp = dKp + ((int64_t)krow0 + tid) * kC;
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 16) {
            float q1[16], q2[16], kk[16];
            tmem_load16f(tmem + 64 + lanebase + c0, q1);
            tmem_load16f(tmem + 256 + lanebase + c0, q2);
            tmem_load16f(tmem + 192 + lanebase + c0, kk);
#pragma unroll
            for (int j = 0; j < 16; ++j)
                *(bf16*)(dqt + tile_off(64, c0 + j, tid)) = __float2bfloat16_rn(gs[c0 + j] * q1[j] + q2[j]);
#pragma unroll
            for (int j = 0; j < 16; j += 4) *(float4*)(kp + c0 + j) = make_float4(kk[j], kk[j + 1], kk[j + 2], kk[j + 3]);
        }
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    if (tid == 0) {
        float ip = 0.f, es = 0.f;
        for (int i = 0; i < 128; ++i) ip += red[i];
        for (int i = 0; i < 64; ++i) es += eR[i];
        red[0] = ip;
        red[1] = es;
    }
    __syncthreads();
    if (tid < 64) {
        float g = dG1[tid] + rE1[tid] - cE1[tid] - eR[tid];
        if (tid == 63) g += gC * red[0] + red[1];
        dGp[(int64_t)row0 + tid] = g;
    }
    if (tid == 0) {
        for (int j = 0; j < 2; ++j) tma_store_4d(&tm_dq, sm + qk::S0 + j * 8192, 64 * j, h, t0, b);
        bulk_commit();
        bulk_wait0();
    }
    __syncwarp();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, 512);
}


// ====================================================== chunk gradients (2)
namespace wy {
constexpr int K = 0, V = 16384, DWT = 32768, DU = 49152;   // K, V, dU [64 x 128]; dW^T [128 x 64]
constexpr int T = 65536, T1 = 73728, T2 = 81920, DT = 90112, Y = 98304, E = 106496;  // [64 x 64]
constexpr int OUT = 114688;                                // dk tile [64 x 128]
constexpr int C1 = 131072, C2 = C1 + 64 * 65 * 4, KK = C2 + 64 * 65 * 4;  // fp32 [64][65]
constexpr int VEC = KK + 64 * 65 * 4;                      // 10 x 64 floats
constexpr int BAR = VEC + 10 * 64 * 4;
constexpr size_t SMEM = BAR + 64 + 1024;
}  // namespace wy

__global__ void __launch_bounds__(128, 1)
grad_wy_tc(Dims d, const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
           const __grid_constant__ CUtensorMap tm_dWt, const __grid_constant__ CUtensorMap tm_dU,
           const __grid_constant__ CUtensorMap tm_T, const __grid_constant__ CUtensorMap tm_dk,
           const __grid_constant__ CUtensorMap tm_dv, const bf16* __restrict__ alpha,
           const bf16* __restrict__ beta, const float* __restrict__ G, const float* __restrict__ dKp,
           const float* __restrict__ dGp, bf16* __restrict__ dalpha, bf16* __restrict__ dbeta, int* err) {
    extern __shared__ unsigned char smraw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    float* C1f = (float*)(sm + wy::C1);
    float* C2f = (float*)(sm + wy::C2);
    float* KKf = (float*)(sm + wy::KK);
    float* Gs = (float*)(sm + wy::VEC);
    float* gs = Gs + 64;
    float* bs = gs + 64;
    float* as_ = bs + 64;
    float* dB12 = as_ + 64;
    float* dGw = dB12 + 64;
    float* dB3 = dGw + 64;
    float* rE2 = dB3 + 64;
    float* cE2 = rE2 + 64;
    float* dGq = cE2 + 64;
    uint64_t* bars = (uint64_t*)(sm + wy::BAR);
    uint32_t* tslot = (uint32_t*)(sm + wy::BAR + 16);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int t0 = c * kC;
    const int64_t chunk = ((int64_t)b * d.H + h) * d.NC + c;
    const int row0 = (int)(chunk * kC);
    const int krow0 = (int)(chunk * kD);

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&bars[0], 9 * 8192);
        for (int j = 0; j < 2; ++j) {
            tma_load_4d(sm + wy::K + j * 8192, &tm_k, &bars[0], 64 * j, h, t0, b);
            tma_load_4d(sm + wy::V + j * 8192, &tm_v, &bars[0], 64 * j, h, t0, b);
            tma_load_2d(sm + wy::DWT + j * 8192, &tm_dWt, &bars[0], 0, krow0 + 64 * j);
            tma_load_2d(sm + wy::DU + j * 8192, &tm_dU, &bars[0], 64 * j, row0);
        }
        tma_load_2d(sm + wy::T, &tm_T, &bars[0], 0, row0);
    }
    if (warp == 0) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    if (tid < 64) {
        const int t = t0 + tid;
        float a = 1.f, be = 0.f;
        if (t < d.T) {
            const int64_t gi = ((int64_t)b * d.T + t) * d.H + h;
            a = __bfloat162float(alpha[gi]);
            be = __bfloat162float(beta[gi]);
        }
        Gs[tid] = G[(int64_t)row0 + tid];
        gs[tid] = expf(Gs[tid]);
        bs[tid] = be;
        as_[tid] = a;
        dGq[tid] = dGp[(int64_t)row0 + tid];
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t lanebase = (uint32_t)(warp * 32) << 16;
    const int r = warp * 16 + (lane & 15);  // row of the M=64 results held by this thread
    const bool rowthr = lane < 16;
    const uint32_t sK = smem_u32(sm + wy::K), sV = smem_u32(sm + wy::V), sDWT = smem_u32(sm + wy::DWT);
    const uint32_t sDU = smem_u32(sm + wy::DU), sT = smem_u32(sm + wy::T), sT1 = smem_u32(sm + wy::T1);
    const uint32_t sT2 = smem_u32(sm + wy::T2), sDT = smem_u32(sm + wy::DT), sY = smem_u32(sm + wy::Y);
    const uint32_t sE = smem_u32(sm + wy::E);

    bool ok = mbar_wait(&bars[0], 0, err, 1);
    // ---- phase 1: Qm = dW K^T (K over k), P = dU V^T (K over v), KK = K K^T   (M=64)
    if (tid == 0 && ok) {
        const uint32_t idq = idesc_bf16(64, 64, true, false);
        const uint32_t id = idesc_bf16(64, 64, false, false);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            mma_bf16_ss(tmem + 0, desc_mnmaj(sDWT, 128, s), desc_kmaj(sK, 64, s), idq, s > 0);
            mma_bf16_ss(tmem + 64, desc_kmaj(sDU, 64, s), desc_kmaj(sV, 64, s), id, s > 0);
            mma_bf16_ss(tmem + 128, desc_kmaj(sK, 64, s), desc_kmaj(sK, 64, s), id, s > 0);
        }
        mma_commit(&bars[1]);
    }
    {   // T1 = T diag(beta gamma), T2 = T diag(beta): scale the columns of the T tile
        const int rr = tid >> 1, c00 = (tid & 1) * 32;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float f[8], f1[8], f2[8];
            tile_get8(sm + wy::T, 64, rr, c00 + 8 * q, f);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int cc = c00 + 8 * q + j;
                f2[j] = f[j] * bs[cc];
                f1[j] = f2[j] * gs[cc];
            }
            *(uint4*)(sm + wy::T1 + tile_off(64, rr, c00 + 8 * q)) = pack8(f1);
            *(uint4*)(sm + wy::T2 + tile_off(64, rr, c00 + 8 * q)) = pack8(f2);
        }
    }
    if (ok) ok = mbar_wait(&bars[1], 0, err, 2);
    __syncwarp();
    fence_after_sync();
    // rows s: C1 = T (P + Qm diag(gamma)), C2 = T Qm, dT (strictly lower), KK
#pragma unroll 1
    for (int c0 = 0; c0 < 64; c0 += 16) {
        float qm[16], p[16], kk[16], t8a[8], t8b[8], dt[16];
        tmem_load16f(tmem + 0 + lanebase + c0, qm);
        tmem_load16f(tmem + 64 + lanebase + c0, p);
        tmem_load16f(tmem + 128 + lanebase + c0, kk);
        tile_get8(sm + wy::T, 64, r, c0, t8a);
        tile_get8(sm + wy::T, 64, r, c0 + 8, t8b);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int rc = c0 + j;
            const float tsr = j < 8 ? t8a[j] : t8b[j - 8];
            const float pv = p[j] + gs[rc] * qm[j];
            dt[j] = (rc < r) ? bs[rc] * pv : 0.f;
            if (rowthr) {
                C1f[r * 65 + rc] = tsr * pv;
                C2f[r * 65 + rc] = tsr * qm[j];
                KKf[r * 65 + rc] = kk[j];
            }
        }
        if (rowthr) tile_put16(sm + wy::DT, 64, r, c0, dt);
    }
    fence_proxy_async();
    fence_before_sync();
    ok = __syncthreads_and(ok);
    fence_after_sync();
    // ---- phase 2: Y = dT T^T   (M=64, K over tokens)
    if (tid == 0 && ok) {
        const uint32_t id = idesc_bf16(64, 64, false, false);
#pragma unroll
        for (int s = 0; s < 4; ++s) mma_bf16_ss(tmem + 0, desc_kmaj(sDT, 64, s), desc_kmaj(sT, 64, s), id, s > 0);
        mma_commit(&bars[1]);
    }
    if (tid < 64) {
        float a1 = 0.f, a2 = 0.f;
        for (int s2 = 0; s2 < 64; ++s2) {
            a1 += C1f[s2 * 65 + tid];
            a2 += C2f[s2 * 65 + tid];
        }
        dB12[tid] = a1;
        dGw[tid] = bs[tid] * gs[tid] * a2;
    }
    if (ok) ok = mbar_wait(&bars[1], 1, err, 4);
    __syncwarp();
    fence_after_sync();
#pragma unroll 1
    for (int c0 = 0; c0 < 64; c0 += 16) {
        float y[16];
        tmem_load16f(tmem + 0 + lanebase + c0, y);
        if (rowthr) tile_put16(sm + wy::Y, 64, r, c0, y);
    }
    fence_proxy_async();
    fence_before_sync();
    ok = __syncthreads_and(ok);
    fence_after_sync();
    // ---- phase 3: dA = -T^T Y (M=64), dV^T = dU^T T2 (M=128); K over tokens
    if (tid == 0 && ok) {
        const uint32_t ida = idesc_bf16(64, 64, true, true, true);
        const uint32_t idv = idesc_bf16(128, 64, true, true);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            mma_bf16_ss(tmem + 64, desc_mnmaj(sT, 64, s), desc_mnmaj(sY, 64, s), ida, s > 0);
            mma_bf16_ss(tmem + 192, desc_mnmaj(sDU, 64, s), desc_mnmaj(sT2, 64, s), idv, s > 0);
        }
        mma_commit(&bars[1]);
    }
    if (ok) ok = mbar_wait(&bars[1], 0, err, 8);
    __syncwarp();
    fence_after_sync();
    {   // rows a: dbeta3, E = beta_a Gam .* dA (strictly lower), E2 = E .* KK
        const float Ga = Gs[r], ba = bs[r];
        float b3 = 0.f, re2 = 0.f;
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 16) {
            float da[16];
            tmem_load16f(tmem + 64 + lanebase + c0, da);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int bc = c0 + j;
                const float m = (bc < r) ? da[j] : 0.f;
                const float gam = (bc < r) ? expf(Ga - Gs[bc]) : 0.f;
                const float kk = KKf[r * 65 + bc];
                b3 += gam * m * kk;
                const float e = ba * gam * m;
                re2 += e * kk;
                if (rowthr) {
                    C1f[r * 65 + bc] = e * kk;
                    C2f[r * 65 + bc] = e;
                }
            }
        }
        if (rowthr) {
            dB3[r] = b3;
            rE2[r] = re2;
        }
        // dV^T row v -> dv[r][v] into the dU tile (dead now)
        unsigned char* dvt = sm + wy::DU;
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 16) {
            float x[16];
            tmem_load16f(tmem + 192 + lanebase + c0, x);
#pragma unroll
            for (int j = 0; j < 16; ++j) *(bf16*)(dvt + tile_off(64, c0 + j, tid)) = __float2bfloat16_rn(x[j]);
        }
    }
    fence_proxy_async();
    fence_before_sync();
    ok = __syncthreads_and(ok);
    fence_after_sync();
    if (tid == 0) {
        for (int j = 0; j < 2; ++j) tma_store_4d(&tm_dv, sm + wy::DU + j * 8192, 64 * j, h, t0, b);
        bulk_commit();
    }
    {   // S = E + E^T (bf16 tile), column sums of E2
        const int rr = tid >> 1, c00 = (tid & 1) * 32;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float f[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int cc = c00 + 8 * q + j;
                f[j] = C2f[rr * 65 + cc] + C2f[cc * 65 + rr];
            }
            *(uint4*)(sm + wy::E + tile_off(64, rr, c00 + 8 * q)) = pack8(f);
        }
        if (tid < 64) {
            float ce = 0.f;
            for (int a = 0; a < 64; ++a) ce += C1f[a * 65 + tid];
            cE2[tid] = ce;
        }
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    // ---- phase 4: dK^T = dW^T T1 + K^T (E + E^T)   (M=128, K over tokens)
    if (tid == 0 && ok) {
        const uint32_t id1 = idesc_bf16(128, 64, false, true);
        const uint32_t id2 = idesc_bf16(128, 64, true, false);
#pragma unroll
        for (int s = 0; s < 4; ++s) mma_bf16_ss(tmem + 256, desc_kmaj(sDWT, 128, s), desc_mnmaj(sT1, 64, s), id1, s > 0);
#pragma unroll
        for (int s = 0; s < 4; ++s) mma_bf16_ss(tmem + 256, desc_mnmaj(sK, 64, s), desc_kmaj(sE, 64, s), id2, 1u);
        mma_commit(&bars[1]);
    }
    if (tid == 0) {
        // dG, then dlog alpha = reverse within-chunk cumsum, dalpha = dlog alpha / alpha
        float run = 0.f;
        for (int rr = 63; rr >= 0; --rr) {
            run += dGq[rr] + dGw[rr] + rE2[rr] - cE2[rr];
            const int t = t0 + rr;
            if (t < d.T) {
                const int64_t gi = ((int64_t)b * d.T + t) * d.H + h;
                dalpha[gi] = __float2bfloat16_rn(run / as_[rr]);
                dbeta[gi] = __float2bfloat16_rn(dB12[rr] + dB3[rr]);
            }
        }
    }
    if (ok) ok = mbar_wait(&bars[1], 1, err, 16);
    __syncwarp();
    fence_after_sync();
    {
        const float* kp = dKp + ((int64_t)krow0 + tid) * kC;
        unsigned char* out = sm + wy::OUT;
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 16) {
            float x[16];
            tmem_load16f(tmem + 256 + lanebase + c0, x);
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
                const float4 pk = *(const float4*)(kp + c0 + j);
                x[j] += pk.x;
                x[j + 1] += pk.y;
                x[j + 2] += pk.z;
                x[j + 3] += pk.w;
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) *(bf16*)(out + tile_off(64, c0 + j, tid)) = __float2bfloat16_rn(x[j]);
        }
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    if (tid == 0) {
        for (int j = 0; j < 2; ++j) tma_store_4d(&tm_dk, sm + wy::OUT + j * 8192, 64 * j, h, t0, b);
        bulk_commit();
        bulk_wait0();
    }
    __syncwarp();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

template <int Vt>
cudaError_t launch_scan_bwd_vt(const Dims& d, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mW,
                               const CUtensorMap& mM, const void* d_o, const TcBufs& tb, const float* dsT,
                               const TcBwdBufs& bb, float* ds0, cudaStream_t st) {
    using P = BScan<Vt>;
    auto kern = scan_bwd_tc<Vt>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(kD / Vt, d.H, d.B);
    kern<<<grid, 128, P::SMEM, st>>>(d, mq, mk, mW, mM, (const bf16*)d_o, tb.G, dsT, bb.dU, bb.dS1, ds0, tb.err);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scan_bwd_tc(const Dims& d, const void* q, const void* k, const void* d_o, const TcBufs& tb,
                               const float* dsT, const TcBwdBufs& bb, float* ds0, cudaStream_t st) {
    CUtensorMap mq, mk, mW, mM;
    const int64_t rows = d.NS() * d.NC * kC;
    if (!tmap_bthd(&mq, q, d.B, d.T, d.H, kD) || !tmap_bthd(&mk, k, d.B, d.T, d.H, kD) ||
        !tmap_rows(&mW, tb.W, rows, kD) || !tmap_rows(&mM, tb.Mqk, rows, kC))
        return cudaErrorInvalidValue;
    switch (tc_scan_vt(d)) {
        case 16: return launch_scan_bwd_vt<16>(d, mq, mk, mW, mM, d_o, tb, dsT, bb, ds0, st);
        case 32: return launch_scan_bwd_vt<32>(d, mq, mk, mW, mM, d_o, tb, dsT, bb, ds0, st);
        default: return launch_scan_bwd_vt<64>(d, mq, mk, mW, mM, d_o, tb, dsT, bb, ds0, st);
    }
}

cudaError_t launch_grad_qk_tc(const Dims& d, const void* q, const void* k, const void* d_o, const TcBufs& tb,
                              const __nv_bfloat16* states, const TcBwdBufs& bb, void* dq, cudaStream_t st) {
    CUtensorMap mq, mk, mdo, mW, mdU, mS0, mdS1, mdq;
    const int64_t rows = d.NS() * d.NC * kC;
    const int64_t krows = d.NS() * d.NC * kD;
    if (!tmap_bthd(&mq, q, d.B, d.T, d.H, kD) || !tmap_bthd(&mk, k, d.B, d.T, d.H, kD) ||
        !tmap_bthd(&mdo, d_o, d.B, d.T, d.H, kD) || !tmap_rows(&mW, tb.W, rows, kD) ||
        !tmap_rows(&mdU, bb.dU, rows, kD) || !tmap_rows(&mS0, states, krows, kD) ||
        !tmap_rows(&mdS1, bb.dS1, krows, kD) || !tmap_bthd(&mdq, dq, d.B, d.T, d.H, kD))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(grad_qk_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)qk::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(d.NC, d.H, d.B);
    grad_qk_tc<<<grid, 128, qk::SMEM, st>>>(d, mq, mk, mdo, mW, mdU, mS0, mdS1, mdq, tb.Ut, tb.Mqk, tb.G, bb.dKp,
                                            bb.dWt, bb.dGp, tb.err);
    return cudaGetLastError();
}

cudaError_t launch_grad_wy_tc(const Dims& d, const void* k, const void* v, const void* alpha, const void* beta,
                              const TcBufs& tb, const TcBwdBufs& bb, void* dk, void* dv, void* dalpha, void* dbeta,
                              cudaStream_t st) {
    CUtensorMap mk, mv, mdWt, mdU, mT, mdk, mdv;
    const int64_t rows = d.NS() * d.NC * kC;
    const int64_t krows = d.NS() * d.NC * kD;
    if (!tmap_bthd(&mk, k, d.B, d.T, d.H, kD) || !tmap_bthd(&mv, v, d.B, d.T, d.H, kD) ||
        !tmap_rows(&mdWt, bb.dWt, krows, kC) || !tmap_rows(&mdU, bb.dU, rows, kD) ||
        !tmap_rows(&mT, tb.T, rows, kC) || !tmap_bthd(&mdk, dk, d.B, d.T, d.H, kD) ||
        !tmap_bthd(&mdv, dv, d.B, d.T, d.H, kD))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(grad_wy_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wy::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(d.NC, d.H, d.B);
    grad_wy_tc<<<grid, 128, wy::SMEM, st>>>(d, mk, mv, mdWt, mdU, mT, mdk, mdv, (const bf16*)alpha,
                                            (const bf16*)beta, tb.G, bb.dKp, bb.dGp, (bf16*)dalpha, (bf16*)dbeta,
                                            tb.err);
    return cudaGetLastError();
}

}  // namespace gdn
