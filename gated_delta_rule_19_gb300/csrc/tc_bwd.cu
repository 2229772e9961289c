// tc_bwd.cu -- tensor-core (tcgen05 + TMA) backward for bf16 inputs, chunk 64, K and
// V of 16 to 128 ("Sparse Delta Memory: layer and kernels", "What the layer computes":
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
// grad_qk_tc (chunk-parallel; persistent, one CTA per SM), from U = Ut - W S0^T as
// the forward scan wrote it:
//     dMqk = dO U^T,   dQK = Gam .* lower(dMqk)
//     dQ^T = S0^T (diag(gamma) dO)^T + K^T dQK^T                 -> dq
//     dK^T (part) = dS1^T (diag(e) U)^T + Q^T dQK                -> scratch
//     dW^T = -S0^T dU^T                                          -> scratch
//     dG (part): gamma in O, Gam in Mqk, exp(G_C - G) in Khat, gamma_C in S1.
//
// grad_wy_tc (chunk-parallel; persistent, two CTAs per SM), through T = (I + A)^-1:
//     Qm = dW K^T,  P = dU V^T,  dT = strict_lower(diag(beta)(P + Qm diag(gamma)))^T-wise
//     dA = strict_lower(-T^T (dT T^T)),  E = diag(beta)(Gam .* dA)
//     dV^T = dU^T T diag(beta)                                   -> dv
//     dK^T = dK^T (part) + dW^T T diag(beta gamma) + K^T (E + E^T) -> dk
//     dbeta, dG (rest), dlog alpha = reverse cumsum of dG, dalpha = dlog alpha / alpha.
//
// Every wait is bounded (2 s unless a test sets a shorter limit) and raises the error
// flag when it gives up.

#include <algorithm>

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

template <int W>
__device__ __forceinline__ void tmem_cols(uint32_t taddr, float* f) {
    if constexpr (W == 24) {
        uint32_t a[8], b[8], c[8];
        tmem_ld8(taddr, a);
        tmem_ld8(taddr + 8, b);
        tmem_ld8(taddr + 16, c);
        tmem_wait_ld(a);
        tmem_wait_ld(b);
        tmem_wait_ld(c);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            f[j] = __uint_as_float(a[j]);
            f[8 + j] = __uint_as_float(b[j]);
            f[16 + j] = __uint_as_float(c[j]);
        }
    } else if constexpr (W == 16) {
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
template <int W>
__device__ __forceinline__ void tmem_cols2(uint32_t ta, uint32_t tb, float* fa, float* fb) {
    if constexpr (W == 24) {
        uint32_t a0[8], a1[8], a2[8], b0[8], b1[8], b2[8];
        tmem_ld8(ta, a0);
        tmem_ld8(ta + 8, a1);
        tmem_ld8(ta + 16, a2);
        tmem_ld8(tb, b0);
        tmem_ld8(tb + 8, b1);
        tmem_ld8(tb + 16, b2);
        tmem_wait_ld(a0);
        tmem_wait_ld(a1);
        tmem_wait_ld(a2);
        tmem_wait_ld(b0);
        tmem_wait_ld(b1);
        tmem_wait_ld(b2);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            fa[j] = __uint_as_float(a0[j]);
            fa[8 + j] = __uint_as_float(a1[j]);
            fa[16 + j] = __uint_as_float(a2[j]);
            fb[j] = __uint_as_float(b0[j]);
            fb[8 + j] = __uint_as_float(b1[j]);
            fb[16 + j] = __uint_as_float(b2[j]);
        }
    } else if constexpr (W == 16) {
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

// Column sums of a 32 x 16 block held one row per lane: on return lanes l and l+16
// hold the sum over the 32 rows of column l % 16.  15 + 1 shuffles.
__device__ __forceinline__ float warp_colsum16(float (&v)[16]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1) {
        const bool upper = lane & w;
#pragma unroll
        for (int j = 0; j < w; ++j) {
            const float send = upper ? v[j] : v[j + w];
            const float keep = upper ? v[j + w] : v[j];
            v[j] = keep + __shfl_xor_sync(0xffffffffu, send, w);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
}

// ============================================================ reverse scan
template <int Vt>
struct BScan {
    // TMA stages: three (more lead) where they fit, up to 48-column slices
    static constexpr int NS = Vt <= 48 ? 3 : 2;
    // stage: Mqk 8K | K_0 | K_1 | Q_0 | Q_1 | W_0 | W_1 (8K each) | dO slice [Vt/8][64][8]
    static constexpr int OFF_M = 0, OFF_K = 8192, OFF_Q = 24576, OFF_W = 40960, OFF_DO = 57344;
    static constexpr int STAGE = 57344 + kC * Vt * 2;   // a multiple of 1024 (swizzled operands)
    static constexpr int DS_OP = NS * STAGE;            // dS1^T [Vt/8][128 k][8], MN-major, no swizzle
    static constexpr int GDO_OP = DS_OP + kD * Vt * 2;  // gamma dO, two buffers [Vt/8][64][8]
    static constexpr int DU_OP = GDO_OP + 2 * kC * Vt * 2;  // dU of iteration it in buffer it & 1
    static constexpr int BAR = DU_OP + 2 * kC * Vt * 2;  // tma[NS], bar1, bar2, then the TMEM slot at +48
    static constexpr size_t SMEM = BAR + 64 + 1024;
    // tA (two buffers), tB, tCc
    static constexpr uint32_t TMEM_COLS = (4 * Vt <= 64) ? 64 : (4 * Vt <= 128 ? 128 : 256);
};

// 320 threads: warps 0-7 run the epilogues, warp 8 issues the MMAs and warp 9 the
// TMA copies (lane 0 of each).  Warps w and w+4 (w < 4) split the columns of TMEM
// lanes 32*w ..  Lanes 0-63: rows of dU (critical); lanes 64-127 prepare the next
// chunk's gamma dO operand; all lanes update dS^T (rows k).  The three roles run
// separate loops with the same two block-wide barriers per chunk.
template <int Vt, bool kPacked>
__global__ void __launch_bounds__(320, 1)
scan_bwd_tc(Dims d, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_W, const __grid_constant__ CUtensorMap tm_M,
            const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_dU,
            const __grid_constant__ CUtensorMap tm_dS1, const float* __restrict__ G, const float* dsT,
            float* ds0, const int* __restrict__ chunk_off, const int* __restrict__ order, int* err) {
    using P = BScan<Vt>;
    constexpr int HV = Vt / 2;
    constexpr int NS = P::NS;
    extern __shared__ unsigned char smraw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    uint64_t* tbar = (uint64_t*)(sm + P::BAR);
    uint64_t* bar1 = tbar + NS;
    uint64_t* bar2 = tbar + NS + 1;
    uint32_t* tslot = (uint32_t*)(sm + P::BAR + 48);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool mma_warp = warp == 8, tma_warp = warp == 9, epi = warp < 8;
    const bool mma_issuer = tid == 256, tma_issuer = tid == 288;
    const int sub = warp & 3, half = (warp >> 2) & 1;
    const int lanerow = 32 * sub + lane;
    const int cb = half * HV;
    const bool urow = sub < 2;
    const int r = urow ? lanerow : lanerow - 64;
    const int v0 = blockIdx.x * Vt, h = blockIdx.y;
    // Stream (b = blockIdx.z, h) runs chunks d.NC-1 .. 0 of its row of chunks.  With
    // packed sequences (chunk_off) the data is one row of chunks per head (B = 1):
    // sequence s = blockIdx.z runs chunks chunk_off[s+1]-1 .. chunk_off[s] of it,
    // with the state gradients in slot s*H + h.  c below counts this CTA's chunks.
    // `order` (or NULL) maps grid row z to the sequence it runs.
    const int zs = order ? order[blockIdx.z] : (int)blockIdx.z;
    int b = zs, c0 = 0, NC = d.NC;
    const int64_t sidx = (int64_t)zs * d.H + h;  // state slot
    if (chunk_off) {
        c0 = chunk_off[zs];
        NC = chunk_off[zs + 1] - c0;
        b = 0;
    }
    const int64_t cbase = ((int64_t)b * d.H + h) * d.NC + c0;  // global index of chunk c = 0

    // Iteration it (chunk NC-1-it) into stage it % NS (the n-th use of a stage
    // completes phase n & 1).
    auto issue_loads = [&](int it) {
        const int c = NC - 1 - it;
        unsigned char* st = sm + (it % NS) * P::STAGE;
        uint64_t* bar = &tbar[it % NS];
        const int row = (int)((cbase + c) * kC);
        const int t0 = chunk_tok<kPacked>(d, c0 + c);
        mbar_arrive_expect_tx(bar, 7 * 8192 + kC * Vt * 2);
        tma_load_2d(st + P::OFF_M, &tm_M, bar, 0, row);
        for (int j = 0; j < 2; ++j) {
            tma_load_4d(st + P::OFF_K + j * 8192, &tm_k, bar, 64 * j, h, t0, b);
            tma_load_4d(st + P::OFF_Q + j * 8192, &tm_q, bar, 64 * j, h, t0, b);
            tma_load_2d(st + P::OFF_W + j * 8192, &tm_W, bar, 64 * j, row);
        }
        tma_load_5d(st + P::OFF_DO, &tm_do, bar, 0, t0, v0 / 8, h, b);
    };

    int issued = 0;  // iterations whose loads were issued (TMA issuer)
    if (tma_issuer) {
        for (int i = 0; i < NS + 2; ++i) mbar_init(&tbar[i], 1);
        fence_mbar_init();
        for (; issued < NS && issued < NC; ++issued) issue_loads(issued);
    }
    if (warp == 0) {
        tmem_alloc(tslot, P::TMEM_COLS);
        tmem_relinquish();
    }
    const int k = lanerow;
    float ds[HV];
#pragma unroll
    for (int j = 0; j < HV; ++j) {
        const int v = v0 + cb + j;  // a 48-wide slice runs past V = 128 (zero columns)
        // the caller's [V, K] gradient (K, V <= 128); rows and columns past them are zero
        ds[j] = (epi && dsT && v < d.V && k < d.K) ? dsT[(sidx * d.V + v) * d.K + k] : 0.f;
    }
    auto write_ds_operand = [&]() {
#pragma unroll
        for (int g = 0; g < HV / 8; ++g)
            *(uint4*)(sm + P::DS_OP + (cb / 8 + g) * 2048 + k * 16) = pack8(&ds[8 * g]);
    };
    if (epi) write_ds_operand();
    // G of a chunk is fetched one chunk ahead.
    float GC_n = (NC > 0 && epi) ? G[(cbase + NC - 1) * kC + kC - 1] : 0.f;
    float Gr_n = (NC > 0 && epi) ? G[(cbase + NC - 1) * kC + r] : 0.f;
    // gamma dO operand (buffer it2 & 1) of iteration it2's chunk, from its stage;
    // rows of lanes 64-127; uses gamma_r = exp(Gr_n) of that chunk.  Rows past the
    // chunk's tokens (a packed batch's ragged chunk reads the next sequence's dO)
    // are zero.
    auto write_gdo_operand = [&](int it2, bool& okk) {
        okk = mbar_wait(&tbar[it2 % NS], (it2 / NS) & 1, err, 8, d.wait_ns) && okk;
        const bool live = !kPacked || r < chunk_valid<true>(d, c0 + NC - 1 - it2);
        const float gr = expf(Gr_n);
        const unsigned char* dsrc = sm + (it2 % NS) * P::STAGE + P::OFF_DO;
        unsigned char* ddst = sm + P::GDO_OP + (it2 & 1) * (kC * Vt * 2);
#pragma unroll
        for (int g = 0; g < HV / 8; ++g) {
            const int gg = cb / 8 + g;
            const uint4 x = *(const uint4*)(dsrc + gg * 1024 + r * 16);
            const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
            float f[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                f[2 * e] = live ? gr * bf_lo(w4[e]) : 0.f;
                f[2 * e + 1] = live ? gr * bf_hi(w4[e]) : 0.f;
            }
            *(uint4*)(ddst + gg * 1024 + r * 16) = pack8(f);
        }
    };
    bool ok = true;
    if (epi && !urow && NC > 0) write_gdo_operand(0, ok);
    fence_proxy_async();
    fence_before_sync();
    ok = __syncthreads_and(ok);
    fence_after_sync();
    const uint32_t tmem = *tslot;
    // Mqk^T dO of iteration it in buffer it & 1 (the second at column 3 Vt)
    const uint32_t tB = tmem + Vt, tCc = tmem + 2 * Vt;
    auto tA_of = [&](int it2) { return tmem + (uint32_t)((it2 & 1) * 3 * Vt); };
    const uint32_t lanebase = (uint32_t)(sub * 32) << 16;
    const uint64_t dDS = sdesc(smem_u32(sm + P::DS_OP), 128, 2048, SW_NONE);
    const uint32_t idn = idesc_bf16(128, Vt, false, true);
    const uint32_t idm = idesc_bf16(128, Vt, true, true);
    const uint32_t idneg = idesc_bf16(128, Vt, true, true, true);  // -W^T dU

    int it = 0;
    int b1_last = -1, b2_last = -1;  // last iterations committed to bar1 / bar2 (MMA issuer)
    bool a_ahead = false;            // Mqk^T dO of iteration it issued during the previous one
    // Mqk^T dO (off the chunk-to-chunk chain) of iteration it2 from its stage
    auto issue_tA = [&](int it2) {
        unsigned char* st2 = sm + (it2 % NS) * P::STAGE;
        const uint64_t dM = sdesc(smem_u32(st2 + P::OFF_M), 8192, 1024, SW_128B);
        const uint64_t dDO = sdesc(smem_u32(st2 + P::OFF_DO), 128, 1024, SW_NONE);
#pragma unroll
        for (int s2 = 0; s2 < 4; ++s2)
            mma_bf16_ss(tA_of(it2), desc_add(dM, s2 * 2048), desc_add(dDO, s2 * 256), idm, s2 > 0);
    };
    if (mma_warp) {
#pragma unroll 1
        for (; ok && it < NC; ++it) {
            const int stg = it % NS;
            unsigned char* st = sm + stg * P::STAGE;
            if (mma_issuer) {
                ok = mbar_wait(&tbar[stg], (it / NS) & 1, err, 8, d.wait_ns) && ok;
                if (ok) {
                    // rows 64-127 of the first two A operands are neighbouring tiles (unused)
                    const uint64_t dK = sdesc(smem_u32(st + P::OFF_K), 16, 1024, SW_128B);
                    const uint64_t dQ = sdesc(smem_u32(st + P::OFF_Q), 8192, 1024, SW_128B);
                    const uint64_t dG =
                        sdesc(smem_u32(sm + P::GDO_OP + (it & 1) * (kC * Vt * 2)), 128, 1024, SW_NONE);
                    if (!a_ahead) issue_tA(it);
#pragma unroll
                    for (int s2 = 0; s2 < 8; ++s2)
                        mma_bf16_ss(tB, desc_add(dK, (s2 >> 2) * 8192 + (s2 & 3) * 32), desc_add(dDS, s2 * 256),
                                    idn, s2 > 0);
                    mma_commit(bar1);
                    b1_last = it;
#pragma unroll
                    for (int s2 = 0; s2 < 4; ++s2)
                        mma_bf16_ss(tCc, desc_add(dQ, s2 * 2048), desc_add(dG, s2 * 256), idm, s2 > 0);
                }
            }
            __syncwarp();
            fence_before_sync();
            ok = __syncthreads_and(ok);  // 1: dU and the next gamma dO written
            if (!ok) break;
            fence_after_sync();
            if (mma_issuer) {
                const uint64_t dW = sdesc(smem_u32(st + P::OFF_W), 8192, 1024, SW_128B);
                const uint64_t dDU = sdesc(smem_u32(sm + P::DU_OP + (it & 1) * (kC * Vt * 2)), 128, 1024, SW_NONE);
#pragma unroll
                for (int s2 = 0; s2 < 4; ++s2)
                    mma_bf16_ss(tCc, desc_add(dW, s2 * 2048), desc_add(dDU, s2 * 256), idneg, 1u);
                mma_commit(bar2);
                b2_last = it;
                // the next iteration's Mqk^T dO now if its tiles are in (never waits: with
                // two stages they are requested only after bar2), covered by its bar1
                a_ahead = it + 1 < NC && mbar_test_wait(&tbar[(it + 1) % NS], ((it + 1) / NS) & 1);
                if (a_ahead) issue_tA(it + 1);
            }
            __syncwarp();
            fence_before_sync();
            ok = __syncthreads_and(ok);  // 2: dS^T written
            if (!ok) break;
            fence_after_sync();
        }
    } else if (tma_warp) {
#pragma unroll 1
        for (; ok && it < NC; ++it) {
            const int64_t chunk = cbase + (NC - 1 - it);
            if (tma_issuer) {
                // the gradient of this chunk's end state, for the chunk-local gradients
                tma_store_3d(&tm_dS1, sm + P::DS_OP, 0, (int)(chunk * kD), v0 / 8);
                bulk_commit();
                // With three stages, iteration it - 1 + NS goes into the stage of
                // iteration it - 1 here, where this warp idles (its MMAs are done:
                // bar2 of it - 1 was waited before the previous barrier 2); it is
                // first read by the gamma dO operand during iteration it + 1.
                if (NS >= 3 && ok && it > 0 && issued < NC) {
                    ok = mbar_wait(bar2, (it - 1) & 1, err, 32, d.wait_ns) && ok;
                    if (ok) issue_loads(issued++);
                }
                bulk_wait_read0();  // it has read dS1^T (rewritten after barrier 1)
            }
            __syncwarp();
            fence_before_sync();
            ok = __syncthreads_and(ok);  // 1
            if (!ok) break;
            fence_after_sync();
            if (tma_issuer) {
                tma_store_3d(&tm_dU, sm + P::DU_OP + (it & 1) * (kC * Vt * 2), 0, (int)(chunk * kC), v0 / 8);
                bulk_commit();
                // with two stages, iteration it + NS into this iteration's stage as
                // soon as its MMAs are done (its gamma dO operand is read next iteration)
                if (NS < 3 && ok && issued < NC) {
                    ok = mbar_wait(bar2, it & 1, err, 32, d.wait_ns) && ok;
                    if (ok) issue_loads(issued++);
                }
                bulk_wait_read1();  // the dU store of the previous iteration has read its buffer
            }
            __syncwarp();
            fence_before_sync();
            ok = __syncthreads_and(ok);  // 2
            if (!ok) break;
            fence_after_sync();
        }
    } else {
#pragma unroll 1
        for (; ok && it < NC; ++it) {
            const int c = NC - 1 - it;
            const int64_t chunk = cbase + c;
            const float GC = GC_n;
            const float gC = expf(GC);
            const float er = expf(GC - Gr_n);
            if (c > 0) {
                GC_n = G[(chunk - 1) * kC + kC - 1];
                Gr_n = G[(chunk - 1) * kC + r];
            }
            if (urow) {
                ok = mbar_wait(bar1, it & 1, err, 16, d.wait_ns) && ok;
                __syncwarp();
                fence_after_sync();
                // dU = Mqk^T dO + e_r (K dS1^T)  (row r, columns cb .. cb+HV)
                float a[HV], bb[HV];
                if constexpr (HV == 8) {
                    uint32_t wa[16], wb[16];
                    tmem_ld16(tA_of(it) + lanebase, wa);
                    tmem_ld16(tB + lanebase, wb);
                    tmem_wait_ld(wa);
                    tmem_wait_ld(wb);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        a[j] = __uint_as_float(half ? wa[8 + j] : wa[j]);
                        bb[j] = __uint_as_float(half ? wb[8 + j] : wb[j]);
                    }
                } else {
                    tmem_cols2<HV>(tA_of(it) + lanebase + cb, tB + lanebase + cb, a, bb);
                }
                unsigned char* du = sm + P::DU_OP + (it & 1) * (kC * Vt * 2);
#pragma unroll
                for (int g = 0; g < HV / 8; ++g) {
                    float u[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) u[j] = a[8 * g + j] + er * bb[8 * g + j];
                    *(uint4*)(du + (cb / 8 + g) * 1024 + r * 16) = pack8(u);
                }
            } else if (c > 0) {
                write_gdo_operand(it + 1, ok);  // operand of the next chunk (c - 1)
            }
            fence_proxy_async();
            fence_before_sync();
            ok = __syncthreads_and(ok);  // 1
            if (!ok) break;
            fence_after_sync();
            ok = mbar_wait(bar2, it & 1, err, 32, d.wait_ns) && ok;
            __syncwarp();
            fence_after_sync();
            {
                float x[HV];
                if constexpr (HV == 8) {
                    uint32_t w16[16];
                    tmem_ld16(tCc + lanebase, w16);
                    tmem_wait_ld(w16);
#pragma unroll
                    for (int j = 0; j < 8; ++j) x[j] = __uint_as_float(half ? w16[8 + j] : w16[j]);
                } else {
                    tmem_cols<HV>(tCc + lanebase + cb, x);
                }
#pragma unroll
                for (int j = 0; j < HV; ++j) ds[j] = gC * ds[j] + x[j];
            }
            write_ds_operand();
            fence_proxy_async();
            fence_before_sync();
            ok = __syncthreads_and(ok);  // 2
            if (!ok) break;
            fence_after_sync();
        }
    }
    if (ok && ds0 && epi) {
#pragma unroll
        for (int j = 0; j < HV; ++j)
            if (v0 + cb + j < d.V && k < d.K) ds0[(sidx * d.V + v0 + cb + j) * d.K + k] = ds[j];
    }
    if (tma_issuer) {
        // on an error, the loads still in flight (bounded waits) before leaving
        if (!ok)
            for (int i2 = it; i2 < issued; ++i2) mbar_wait(&tbar[i2 % NS], (i2 / NS) & 1, nullptr, 0);
        bulk_wait_read0();  // stores have read their tiles; their writes complete on their own
    }
    if (mma_issuer && !ok) {  // the MMAs still in flight, before the TMEM is freed
        if (b1_last >= 0) mbar_wait(bar1, b1_last & 1, nullptr, 0);
        if (a_ahead) {  // uncommitted MMAs of the next iteration
            mma_commit(bar1);
            mbar_wait(bar1, (b1_last + 1) & 1, nullptr, 0);
        }
        if (b2_last >= 0) mbar_wait(bar2, b2_last & 1, nullptr, 0);
    }
    __syncwarp();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, P::TMEM_COLS);
}

// ====================================================== chunk gradients (1)
namespace qk {
// group A (free once phase 1's MMAs are done): U | [dO_0 | dU_0 | dO_1 | dU_1] | S0^T | dS1^T
constexpr int U = 0;                   // [64 x 128]: U_0 | U_1
constexpr int DO = 16384;              // stacked [dO; dU] (M / N = 128), column blocks 16 KB apart
constexpr int S0 = 49152, DS1 = 81920; // [128 x 128], column blocks 16 KB apart
// group B (free once phase 2's MMAs are done)
constexpr int Q = 114688, K = 131072;  // [64 x 128]: two column blocks 8 KB apart
// results
constexpr int DQK = 147456;            // [64 x 64]
constexpr int DWT = 155648;            // dW^T [128 x 64] (two 64-row halves)
constexpr int DQ = 172032;             // dq [64 x 128]
constexpr int DKP = 188416;            // dK^T part [128 x 64]
constexpr int VEC = 204800;            // Gs gs | dG1p[4] eRp[4] rE1[4] | cE1[8][16] | red[512] | 8 | rqs
constexpr int NVEC = 2 * 64 + 3 * 256 + 128 + 512 + 8 + 64;
constexpr int DD = 212992;             // raw prologue: diag(-q . dq) [64 x 64], zero off the diagonal
static_assert(VEC + NVEC * 4 <= DD, "vectors before the diagonal tile");
constexpr int BAR = DD + 8192;
constexpr size_t SMEM = BAR + 64 + 1024;
static_assert(SMEM <= 232448, "one CTA per SM");
}  // namespace qk

// Chunk gradients on the q side, from the forward's U (= U~ - W S0^T, saved by the
// forward scan), the chunk-start state S0, and the reverse scan's dU and dS1:
//   phase 1 (operands all loaded):
//     S0^T [dO; dU]^T          -> dQ1^T = S0^T dO^T  and  -dW^T = S0^T dU^T  (N = 128)
//     [dO; dU] U^T (rows 0-63) -> dMqk = dO U^T                               (N = 64)
//     dS1^T U^T                -> dK'^T = (U dS1)^T                           (N = 64)
//   epilogue 1: dQK = Gam .* lower(dMqk); dW^T out; the dG sums
//     dG1_r = sum_k Q_rk dQ1_rk  (= sum_v dO_rv (Q S0^T)_rv, gamma in O),
//     eR_r  = sum_k K_rk dK'_rk  (= sum_v U_rv (K dS1^T)_rv, exp(G_C - G) in Khat),
//     E1 = dMqk .* Mqk row and column sums (Gam in Mqk), <dS1, S0> (gamma_C in S1)
//   phase 2: dQ2^T = K^T dQK^T,  QK^T = Q^T dQK                               (N = 64)
//   epilogue 2: dq = gamma dQ1 + dQ2; dK^T part = exp(G_C - G) dK'^T + Q^T dQK; dG part.
// Persistent, 512 threads, one CTA per SM: CTA i starts with chunk i and takes
// further chunks from a work counter.  Warps w, w+4, w+8, w+12 reach TMEM lanes
// 32*(w%4) .. and split the columns of every epilogue.  Group A tiles of the next
// chunk are requested as soon as phase 1's MMAs are done, group B after phase 2.
template <bool kRaw, bool kPacked>
__global__ void __launch_bounds__(512, 1)
grad_qk_tc(Dims d, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
           const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_U,
           const __grid_constant__ CUtensorMap tm_dU, const __grid_constant__ CUtensorMap tm_S0,
           const __grid_constant__ CUtensorMap tm_dS1, const __grid_constant__ CUtensorMap tm_dq,
           const __grid_constant__ CUtensorMap tm_dKp, const __grid_constant__ CUtensorMap tm_dWt,
           const bf16* __restrict__ Mqk, const float* __restrict__ G, float* __restrict__ dGp, RawPrologue raw,
           bf16* __restrict__ dq_rows, int* err) {
    extern __shared__ unsigned char smraw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    float* Gs = (float*)(sm + qk::VEC);
    float* gs = Gs + 64;
    float* dG1p = gs + 64;   // [4 lane quarters][64 tokens]
    float* eRp = dG1p + 256; // [4][64]
    float* rE1 = eRp + 256;  // [4 column quarters][64 rows]
    float* cE1 = rE1 + 256;  // [2 row halves][4 column quarters][16]
    float* red = cE1 + 128;  // 512
    float* fin = red + 512;  // <dS1, S0>, sum_i e_i eR_i
    float* rqs = fin + 8;    // raw prologue: 1 / |q_raw| of the chunk's tokens
    // [0] loads A, [1] loads B, [2] phase 1 MMAs, [3] phase 2 MMAs
    uint64_t* bars = (uint64_t*)(sm + qk::BAR);
    uint32_t* tslot = (uint32_t*)(sm + qk::BAR + 40);
    int* s_next = (int*)(sm + qk::BAR + 44);  // the chunk after this one

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sub = warp & 3, qtr = warp >> 2;
    const int lanerow = 32 * sub + lane;  // TMEM lane: a row k of the [128 x .] products
    const bool urow = sub < 2;            // lanes 0-63: rows of the [64 x 64] product
    const int r = urow ? lanerow : lanerow - 64;
    const int cb = qtr * 16;              // this thread's 16 columns of a 64-column product
    const int64_t nchunks = d.NS() * d.NC;
    constexpr int kIssuer = 64;  // MMAs, loads and stores: lane 0 of warp 2

    auto decode = [&](int64_t ch, int& b, int& h, int& c) {
        c = (int)(ch % d.NC);
        const int64_t bh = ch / d.NC;
        h = (int)(bh % d.H);
        b = (int)(bh / d.H);
    };
    auto load_A = [&](int64_t ch) {
        int b, h, c;
        decode(ch, b, h, c);
        const int row0 = (int)(ch * kC), krow0 = (int)(ch * kD);
        mbar_arrive_expect_tx(&bars[0], 14 * 8192);
        for (int j = 0; j < 2; ++j) {
            tma_load_2d(sm + qk::U + j * 8192, &tm_U, &bars[0], 64 * j, row0);
            tma_load_4d(sm + qk::DO + j * 16384, &tm_do, &bars[0], 64 * j, h, chunk_tok<kPacked>(d, c), b);
            tma_load_2d(sm + qk::DO + j * 16384 + 8192, &tm_dU, &bars[0], 64 * j, row0);
            for (int i = 0; i < 2; ++i) {
                tma_load_2d(sm + qk::S0 + j * 16384 + i * 8192, &tm_S0, &bars[0], 64 * j, krow0 + 64 * i);
                tma_load_2d(sm + qk::DS1 + j * 16384 + i * 8192, &tm_dS1, &bars[0], 64 * j, krow0 + 64 * i);
            }
        }
    };
    auto load_B = [&](int64_t ch) {
        int b, h, c;
        decode(ch, b, h, c);
        mbar_arrive_expect_tx(&bars[1], 4 * 8192);
        for (int j = 0; j < 2; ++j) {
            tma_load_4d(sm + qk::Q + j * 8192, &tm_q, &bars[1], 64 * j, h, chunk_tok<kPacked>(d, c), b);
            tma_load_4d(sm + qk::K + j * 8192, &tm_k, &bars[1], 64 * j, h, chunk_tok<kPacked>(d, c), b);
        }
    };

    const int64_t first = blockIdx.x;
    // warp 3 keeps the next chunk's G (2 tokens per lane) in registers
    float2 gnext = make_float2(0.f, 0.f), rnext = gnext;
    auto load_rq = [&](int64_t c2) {  // 1 / |q_raw| of tokens 2 lane, 2 lane + 1 (raw prologue)
        int b2, h2, cc;
        decode(c2, b2, h2, cc);
        const int t = cc * kC + 2 * lane;
        const int64_t gi = ((int64_t)b2 * d.T + t) * d.H + h2;
        rnext.x = t < d.T ? raw.rq[gi] : 0.f;
        rnext.y = t + 1 < d.T ? raw.rq[gi + d.H] : 0.f;
    };
    int claimed = 0;  // lane 0 of warp 3: the next chunk, claimed from the work counter a chunk ahead
    if (warp == 3 && first < nchunks) {
        gnext = *(const float2*)(G + first * kC + 2 * lane);
        if (kRaw) load_rq(first);
        if (lane == 0) claimed = (int)gridDim.x + atomicAdd(err + kSchedQk, 1);
    }
    // issued counts (thread kIssuer): load groups A and B, phase 1 and 2 commits;
    // on an error the last of each is waited for (bounded) before the CTA leaves
    int na = 0, nb = 0, n1 = 0, n2 = 0;
    if (tid == kIssuer) {
        for (int i = 0; i < 4; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        if (first < nchunks) {
            load_A(first);
            load_B(first);
            na = nb = 1;
        }
    }
    if (warp == 0) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    if (kRaw) {  // the diagonal tile's zeros, written once
        for (int i = tid; i < 512; i += 512) *(uint4*)(sm + qk::DD + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t lanebase = (uint32_t)(sub * 32) << 16;
    // TMEM columns: dQ1^T 0-63 and -dW^T 64-127 (tQW), dMqk 128-191 (then dQ2^T),
    // dK'^T 192-255, Q^T dQK 256-319
    const uint32_t tQW = tmem, tQ1 = tmem, tDW = tmem + 64, tDM = tmem + 128, tQ2 = tmem + 128,
                   tDK = tmem + 192, tQK = tmem + 256;
    const uint32_t sU = smem_u32(sm + qk::U), sDO = smem_u32(sm + qk::DO), sS0 = smem_u32(sm + qk::S0);
    const uint32_t sDS1 = smem_u32(sm + qk::DS1), sQ = smem_u32(sm + qk::Q), sK = smem_u32(sm + qk::K);
    const uint32_t sDQK = smem_u32(sm + qk::DQK);

    // rows of Mqk (this quarter's 16 columns) of row r, read a chunk ahead
    uint4 mqv[2];
    auto load_mq = [&](int64_t c2) {
        const uint4* mp = (const uint4*)(Mqk + (c2 * kC + r) * kC + cb);
        mqv[0] = mp[0];
        mqv[1] = mp[1];
    };
    if (urow && first < nchunks) load_mq(first);
    bool ok = true;
    int n = 0;
    int64_t nxt = first;
#pragma unroll 1
    for (int64_t ch = first; ch < nchunks; ch = nxt, ++n) {
        int b, h, c;
        decode(ch, b, h, c);
        const int t0 = chunk_tok<kPacked>(d, c);  // first token of the chunk
        const int nv = kPacked ? chunk_valid<true>(d, c) : kC;  // its tokens (packed)
        const int row0 = (int)(ch * kC), krow0 = (int)(ch * kD);
        const int ph = n & 1;
        if (warp == 3) {
            const int nx = __shfl_sync(0xffffffffu, claimed, 0);
            if (lane == 0) {
                *s_next = nx;
                if (nx < nchunks) claimed = (int)gridDim.x + atomicAdd(err + kSchedQk, 1);
            }
            Gs[2 * lane] = gnext.x;
            Gs[2 * lane + 1] = gnext.y;
            gs[2 * lane] = expf(gnext.x);
            gs[2 * lane + 1] = expf(gnext.y);
            rqs[2 * lane] = rnext.x;
            rqs[2 * lane + 1] = rnext.y;
            if (nx < nchunks) {
                gnext = *(const float2*)(G + (int64_t)nx * kC + 2 * lane);
                if (kRaw) load_rq(nx);
            }
        }
        // ---- phase 1 (K over v): S0^T [dO; dU]^T (N=128), [dO; dU] U^T and dS1^T U^T (N=64)
        if (tid == kIssuer) {
            ok = mbar_wait(&bars[0], ph, err, 1, d.wait_ns) && ok;
            if (ok) {
                const uint32_t id128 = idesc_bf16(128, 128, false, false);
                const uint32_t id64 = idesc_bf16(128, 64, false, false);
                const uint64_t ds0 = sdesc(sS0, 16, 1024, SW_128B), ddo = sdesc(sDO, 16, 1024, SW_128B);
                const uint64_t dds1 = sdesc(sDS1, 16, 1024, SW_128B), du = sdesc(sU, 16, 1024, SW_128B);
#pragma unroll
                for (int s2 = 0; s2 < 8; ++s2) {
                    const uint32_t o128 = (s2 >> 2) * 16384 + (s2 & 3) * 32, o64 = (s2 >> 2) * 8192 + (s2 & 3) * 32;
                    mma_bf16_ss(tQW, desc_add(ds0, o128), desc_add(ddo, o128), id128, s2 > 0);
                    mma_bf16_ss(tDM, desc_add(ddo, o128), desc_add(du, o64), id64, s2 > 0);
                    mma_bf16_ss(tDK, desc_add(dds1, o128), desc_add(du, o64), id64, s2 > 0);
                }
                mma_commit(&bars[2]);
                ++n1;
            }
        }
        ok = mbar_wait(&bars[0], ph, err, 1, d.wait_ns) && ok;  // S0 and dS1 (read below)
        {   // <dS1, S0> over the chunk (both tiles share one layout), coalesced, while
            // phase 1's MMAs run
            const uint4* a = (const uint4*)(sm + qk::S0) + tid;
            const uint4* bq = (const uint4*)(sm + qk::DS1) + tid;
            float acc = 0.f;
#pragma unroll 4
            for (int i = 0; i < 4; ++i) {
                const uint4 x = a[i * 512], y = bq[i * 512];
                const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) acc += bf_lo(xw[e]) * bf_lo(yw[e]) + bf_hi(xw[e]) * bf_hi(yw[e]);
            }
            red[tid] = acc;
        }
        if (ok) ok = mbar_wait(&bars[2], ph, err, 2);
        __syncwarp();
        fence_after_sync();
        // the previous chunk's stores no longer read the result tiles (rewritten below)
        if (tid == kIssuer) bulk_wait_read0();
        fence_before_sync();
        ok = __syncthreads_and(ok);  // Gs / gs, the next chunk's index; S0^T, dS1^T read
        fence_after_sync();
        if (!ok) break;
        nxt = *s_next;
        const bool has_next = nxt < nchunks;
        // every group A tile is dead (phase 1's MMAs are done): the next chunk's
        if (tid == kIssuer && has_next) {
            load_A(nxt);
            ++na;
        }
        ok = mbar_wait(&bars[1], ph, err, 1) && ok;  // Q, K (read by epilogue 1)
        // ---- epilogue 1
        {
            const float Gr = Gs[r];
            if (urow) {  // dMqk row r, columns cb .. cb+15 -> E1 row / column sums, dQK
                float dm[16], e1[16], dq[16];
                float rsum = 0.f;
                tmem_load16f(tDM + lanebase + cb, dm);
                const uint32_t mw[8] = {mqv[0].x, mqv[0].y, mqv[0].z, mqv[0].w,
                                        mqv[1].x, mqv[1].y, mqv[1].z, mqv[1].w};
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int i = cb + j;
                    const float mq = (j & 1) ? bf_hi(mw[j >> 1]) : bf_lo(mw[j >> 1]);
                    e1[j] = dm[j] * mq;
                    rsum += e1[j];
                    // rows past the chunk's tokens (a packed batch's ragged chunk reads
                    // the next sequence's dO) are zero
                    dq[j] = (i <= r && (!kPacked || r < nv)) ? __expf(Gr - Gs[i]) * dm[j] : 0.f;
                }
                tile_put16(sm + qk::DQK, 64, r, cb, dq);
                rE1[qtr * 64 + r] = rsum;
                const float csum = warp_colsum16(e1);
                if (lane < 16) cE1[(sub * 4 + qtr) * 16 + lane] = csum;
                if (has_next) load_mq(nxt);
            }
            const int k = lanerow;
            // -dW^T row k, columns cb .. cb+15 -> the dW^T tile (stored to scratch by TMA)
            {
                float w[16];
                tmem_load16f(tDW + lanebase + cb, w);
#pragma unroll
                for (int j = 0; j < 16; ++j) w[j] = -w[j];
                unsigned char* wt = sm + qk::DWT + (k >> 6) * 8192;
                *(uint4*)(wt + sw128_off(k & 63, cb)) = pack8(w);
                *(uint4*)(wt + sw128_off(k & 63, cb + 8)) = pack8(w + 8);
            }
            // dG1_t = sum_k Q_tk dQ1_tk and eR_t = sum_k K_tk dK'_tk for this quarter's
            // 16 tokens t: products over this warp's 32 rows k, then column sums
            {
                float q1[16], dk[16], pq[16], pk[16];
                tmem_load16f2(tQ1 + lanebase + cb, tDK + lanebase + cb, q1, dk);
                const unsigned char* qt = sm + qk::Q + (k >> 6) * 8192;
                const unsigned char* kt = sm + qk::K + (k >> 6) * 8192;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const uint32_t off = sw128_off(cb + j, k & 63);
                    pq[j] = __bfloat162float(*(const bf16*)(qt + off)) * q1[j];
                    pk[j] = __bfloat162float(*(const bf16*)(kt + off)) * dk[j];
                }
                const float sq = warp_colsum16(pq);
                const float sk = warp_colsum16(pk);
                if (lane < 16) {
                    dG1p[sub * 64 + cb + lane] = sq;
                    eRp[sub * 64 + cb + lane] = sk;
                }
            }
        }
        fence_proxy_async();
        fence_before_sync();
        ok = __syncthreads_and(ok);
        fence_after_sync();
        if (!ok) break;
        if (kRaw && warp == kIssuer / 32) {
            // The normalisation's chain rule needs q . dq per token, which epilogue 1
            // already holds: q . dQ1 = dG1 and q . dQ2 = sum_t' dQK q.k = the row sum of
            // dMqk .* Mqk (E1).  diag(-q . dq) goes on the diagonal tile, and phase 2
            // adds Q^T diag(-q . dq) to dQ2^T (dq_raw = (dq - q (q . dq)) / |q_raw|).
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int t = lane + 32 * hh;
                const float g1 = dG1p[t] + dG1p[64 + t] + dG1p[128 + t] + dG1p[192 + t];
                const float e1 = rE1[t] + rE1[64 + t] + rE1[128 + t] + rE1[192 + t];
                *(bf16*)(sm + qk::DD + sw128_off(t, t)) = __float2bfloat16_rn(-(gs[t] * g1 + e1));
            }
            fence_proxy_async();
            __syncwarp();
        }
        // ---- phase 2 (K over tokens): dQ2^T = K^T dQK^T;  Q^T dQK  (M=128, N=64)
        if (tid == kIssuer) {
            for (int j = 0; j < 2; ++j) tma_store_2d(&tm_dWt, sm + qk::DWT + j * 8192, 0, krow0 + 64 * j);
            bulk_commit();
            const uint32_t idq = idesc_bf16(128, 64, true, false);
            const uint32_t idk = idesc_bf16(128, 64, true, true);
            const uint64_t dkm = sdesc(sK, 8192, 1024, SW_128B), dqm = sdesc(sQ, 8192, 1024, SW_128B);
            const uint64_t dqk = sdesc(sDQK, 16, 1024, SW_128B), dqkm = sdesc(sDQK, 8192, 1024, SW_128B);
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2) {
                mma_bf16_ss(tQ2, desc_add(dkm, s2 * 2048), desc_add(dqk, s2 * 32), idq, s2 > 0);
                mma_bf16_ss(tQK, desc_add(dqm, s2 * 2048), desc_add(dqkm, s2 * 2048), idk, s2 > 0);
            }
            if (kRaw) {  // dQ2^T += Q^T diag(-q . dq)
                const uint64_t ddd = sdesc(smem_u32(sm + qk::DD), 16, 1024, SW_128B);
#pragma unroll
                for (int s2 = 0; s2 < 4; ++s2)
                    mma_bf16_ss(tQ2, desc_add(dqm, s2 * 2048), desc_add(ddd, s2 * 32), idq, 1u);
            }
            mma_commit(&bars[3]);
            ++n2;
        }
        // sums over the chunk while phase 2 runs: <dS1, S0> (warp 2) and
        // sum_i exp(G_C - G_i) eR_i (warp 5)
        if (warp == 2) {
            float ip = 0.f;
            for (int i = lane; i < 512; i += 32) ip += red[i];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ip += __shfl_xor_sync(0xffffffffu, ip, off);
            if (lane == 0) fin[0] = ip;
        } else if (warp == 5) {
            const float GC = Gs[63];
            float es = 0.f;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int t = lane + 32 * hh;
                es += expf(GC - Gs[t]) * (eRp[t] + eRp[64 + t] + eRp[128 + t] + eRp[192 + t]);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) es += __shfl_xor_sync(0xffffffffu, es, off);
            if (lane == 0) fin[1] = es;
        }
        ok = mbar_wait(&bars[3], ph, err, 8) && ok;
        __syncwarp();
        fence_after_sync();
        fence_before_sync();
        ok = __syncthreads_and(ok);  // Q, K, dQK free; fin visible
        fence_after_sync();
        if (!ok) break;
        if (tid == kIssuer && has_next) {
            load_B(nxt);
            ++nb;
        }
        // ---- epilogue 2: dq (transposed into the dq tile), the dK^T part, dG
        {
            const int k = lanerow;
            const float GC = Gs[63];
            float q1[16], q2[16];
            tmem_load16f2(tQ1 + lanebase + cb, tQ2 + lanebase + cb, q1, q2);
            unsigned char* dqt = sm + qk::DQ;
            // dq of the normalised row; with the raw prologue dQ2 already carries
            // -q (q . dq), so dq_raw is one scaling by 1 / |q_raw|
#pragma unroll
            for (int j = 0; j < 16; ++j)
                q1[j] = kRaw ? rqs[cb + j] * (gs[cb + j] * q1[j] + q2[j]) : gs[cb + j] * q1[j] + q2[j];
#pragma unroll
            for (int j = 0; j < 16; ++j) *(bf16*)(dqt + tile_off(64, cb + j, k)) = __float2bfloat16_rn(q1[j]);
            float dk[16], qkv[16];
            tmem_load16f2(tDK + lanebase + cb, tQK + lanebase + cb, dk, qkv);
#pragma unroll
            for (int j = 0; j < 16; ++j) dk[j] = expf(GC - Gs[cb + j]) * dk[j] + qkv[j];
            unsigned char* kp = sm + qk::DKP + (k >> 6) * 8192;
            *(uint4*)(kp + sw128_off(k & 63, cb)) = pack8(dk);
            *(uint4*)(kp + sw128_off(k & 63, cb + 8)) = pack8(dk + 8);
        }
        if (tid < 64) {
            const int t = tid;
            const float GC = Gs[63], gC = gs[63];
            const float dG1 = dG1p[t] + dG1p[64 + t] + dG1p[128 + t] + dG1p[192 + t];
            const float eR = eRp[t] + eRp[64 + t] + eRp[128 + t] + eRp[192 + t];
            const float re = rE1[t] + rE1[64 + t] + rE1[128 + t] + rE1[192 + t];
            const int qq = t >> 4, col = t & 15;
            const float ce = cE1[(0 * 4 + qq) * 16 + col] + cE1[(1 * 4 + qq) * 16 + col];
            // per-token terms only for the chunk's tokens (past them, dQ1 carries the
            // next sequence's dO in a packed batch's ragged chunk); the chunk-level
            // terms (gamma_C in S1, exp(G_C - G) in Khat) sit at position 63, from
            // where the reverse cumsum carries them to every token of the chunk
            float g = (!kPacked || t < nv) ? gs[t] * dG1 + re - ce - expf(GC - Gs[t]) * eR : 0.f;
            if (t == 63) g += gC * fin[0] + fin[1];
            dGp[(int64_t)row0 + t] = g;
            // k . (the dK part written here) = exp(G_C - G_t) eR_t + the column sum of E1
            if (kRaw) raw.kdot[(int64_t)row0 + t] = expf(GC - Gs[t]) * eR + ce;
        }
        fence_proxy_async();
        fence_before_sync();
        ok = __syncthreads_and(ok);
        fence_after_sync();
        const bool dq_tma = !kPacked || nv == kC;
        if (tid == kIssuer && ok) {
            for (int j = 0; j < 2; ++j) {
                if (dq_tma && 64 * j < d.K) tma_store_4d(&tm_dq, sm + qk::DQ + j * 8192, 64 * j, h, t0, b);
                tma_store_2d(&tm_dKp, sm + qk::DKP + j * 8192, 0, krow0 + 64 * j);
            }
            bulk_commit();
        }
        if constexpr (kPacked) {
            if (!dq_tma && ok && warp == kIssuer / 32) {
                // the last chunk of a packed sequence, fewer than 64 tokens: the valid
                // rows of dq (the rows after them belong to the next sequence)
                for (int i = lane; i < nv * (kD / 8); i += 32) {
                    const int t = i / (kD / 8), k8 = 8 * (i % (kD / 8));
                    if (k8 < d.K)
                        *(uint4*)(dq_rows + ((int64_t)(t0 + t) * d.H + h) * d.K + k8) =
                            *(const uint4*)(sm + qk::DQ + (k8 >> 6) * 8192 + sw128_off(t, k8 & 63));
                }
            }
        }
        if (!ok) break;
    }
    if (tid == kIssuer) {
        if (!ok) {  // the last loads and MMAs issued may still be in flight (bounded waits)
            if (na > 0) mbar_wait(&bars[0], (na - 1) & 1, nullptr, 0);
            if (nb > 0) mbar_wait(&bars[1], (nb - 1) & 1, nullptr, 0);
            if (n1 > 0) mbar_wait(&bars[2], (n1 - 1) & 1, nullptr, 0);
            if (n2 > 0) mbar_wait(&bars[3], (n2 - 1) & 1, nullptr, 0);
        }
        bulk_wait_read0();  // stores have read their tiles; their writes complete on their own
    }
    __syncwarp();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ====================================================== chunk gradients (2)
namespace wy {
// inputs: K | V | dU ([64 x 128] each) | dW^T [128 x 64] | T [64 x 64]
constexpr int K = 0, V = 16384, DU = 32768, DWT = 49152, T = 65536;
constexpr int T1 = 73728, T2 = 81920, DT = 90112, Y = 98304;  // [64 x 64]
constexpr int E = DT;      // dT is dead once Y is formed
constexpr int ID = Y;      // identity [64 x 64], written once Y has been read
constexpr int KP = V;      // dK partial [128 x 64], loaded once V has been read
constexpr int DV = DU;     // outputs [64 x 128] into dead slots
constexpr int DK = DT;     // dT / E and Y / ID: dead once phase 4's MMA is done, not
                           // rewritten before the next chunk's first MMA completes
constexpr int VEC = Y + 8192;  // per-token and partial-sum vectors
constexpr int NVEC = 18 * 64;  // 15 x 64, then (raw prologue) sigmoid(a), 1/|k_raw|, k . dK part
constexpr int BAR = VEC + NVEC * 4;
constexpr size_t SMEM = BAR + 64 + 1024;
static_assert(2 * (SMEM + 1024) <= 233472, "two CTAs per SM");
// the M=128 operands whose rows 0-63 are not used read the 8 KB before their tile
static_assert(T1 - 8192 == T && T2 - 8192 == T1 && E - 8192 == T2 && ID - 8192 == DT, "tile order");
static_assert(DK + 16384 == VEC, "the dK tile spans the dT and Y tiles");
}  // namespace wy

// Persistent, two CTAs per SM (each one's epilogues overlap the other's MMAs and
// loads), 256 threads: CTA i starts with chunk i and takes further chunks from a
// work counter (lane 0 of warp 3 claims each one a chunk ahead), so that faster SMs
// take more chunks.  Warps w and w+4
// reach TMEM lanes 32*(w%4) and split columns.  Rows of the 64 x 64 products land
// in lanes 0-63 (threads with warp % 4 < 2); dV and dK are formed with tokens on
// lanes 64-127 and 128 columns, so the other half of the threads writes them as
// whole rows.  dK is staged in the dT and Y tiles, so every input slot is free once
// phase 4's MMA is done: the next chunk's tiles are requested then, and warp 3
// reads the next chunk's per-token values into registers a chunk ahead.
template <bool kRaw, bool kPacked>
__global__ void __launch_bounds__(256, 2)
grad_wy_tc(Dims d, const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
           const __grid_constant__ CUtensorMap tm_dWt, const __grid_constant__ CUtensorMap tm_dU,
           const __grid_constant__ CUtensorMap tm_T, const __grid_constant__ CUtensorMap tm_dk,
           const __grid_constant__ CUtensorMap tm_dv, const __grid_constant__ CUtensorMap tm_dKp,
           const bf16* __restrict__ alpha, const bf16* __restrict__ beta, const float* __restrict__ G,
           const float* __restrict__ dGp, bf16* __restrict__ dalpha, bf16* __restrict__ dbeta, RawPrologue raw,
           bf16* __restrict__ dk_rows, bf16* __restrict__ dv_rows, int* err) {
    extern __shared__ unsigned char smraw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    float* vec = (float*)(sm + wy::VEC);
    float* Gs = vec;            // 64
    float* gs = vec + 64;
    float* bs = vec + 128;
    float* as_ = vec + 192;
    float* dGq = vec + 256;
    float* cB12 = vec + 320;    // [2 row groups][64]
    float* cGw = vec + 448;     // [2][64]
    float* dB3p = vec + 576;    // [2 column halves][64]
    float* rE2p = vec + 704;    // [2][64]
    float* cE2 = vec + 832;     // [2][64]
    float* sas = vec + 960;     // raw prologue: sigmoid(a) = 1 - alpha
    float* rks = vec + 1024;    // raw prologue: 1 / |k_raw|
    float* kds = vec + 1088;    // raw prologue: k . dK part (from grad_qk_tc)
    uint64_t* bars = (uint64_t*)(sm + wy::BAR);  // [0] loads, [1] MMA, [2] dK partial
    uint32_t* tslot = (uint32_t*)(sm + wy::BAR + 32);
    int* s_next = (int*)(sm + wy::BAR + 40);  // the chunk after this one

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sub = warp & 3, half = warp >> 2;
    const int lanerow = 32 * sub + lane;
    const bool urow = sub < 2;
    const int r = urow ? lanerow : lanerow - 64;  // row of the 64-row results (both sides)
    const int cb = half * 32;                     // this warp's 32 columns of a 64-column result
    const int64_t nchunks = d.NS() * d.NC;

    // chunk index = (b * H + h) * NC + c; its first token (a packed batch: from the
    // chunk-token map)
    auto decode = [&](int64_t ch, int& b, int& h, int& t0) {
        t0 = chunk_tok<kPacked>(d, (int)(ch % d.NC));
        h = (int)((ch / d.NC) % d.H);
        b = (int)(ch / d.NC / d.H);
    };
    auto load_inputs = [&](int64_t ch) {
        int b, h, t0;
        decode(ch, b, h, t0);
        const int row0 = (int)(ch * kC), krow0 = (int)(ch * kD);
        mbar_arrive_expect_tx(&bars[0], 9 * 8192);
        for (int j = 0; j < 2; ++j) {
            tma_load_4d(sm + wy::K + j * 8192, &tm_k, &bars[0], 64 * j, h, t0, b);
            tma_load_4d(sm + wy::V + j * 8192, &tm_v, &bars[0], 64 * j, h, t0, b);
            tma_load_2d(sm + wy::DU + j * 8192, &tm_dU, &bars[0], 64 * j, row0);
            tma_load_2d(sm + wy::DWT + j * 8192, &tm_dWt, &bars[0], 0, krow0 + 64 * j);
        }
        tma_load_2d(sm + wy::T, &tm_T, &bars[0], 0, row0);
    };
    // warp 3: G, the dG partial and the gates of tokens 2 lane, 2 lane + 1 of a chunk
    // (padding: alpha = 1, beta = 0), held in registers until the chunk starts
    // (with the raw prologue: the gate logits, padding a = b = -inf, and 1 / |k_raw|)
    float2 gv = make_float2(0.f, 0.f), qv = gv, kv = gv, dv2 = gv;
    bf16 ga[2], gb[2];
    auto load_vec = [&](int64_t ch) {
        int b, h, t0;
        decode(ch, b, h, t0);
        const int64_t row0 = ch * kC;
        gv = *(const float2*)(G + row0 + 2 * lane);
        qv = *(const float2*)(dGp + row0 + 2 * lane);
        if (kRaw) dv2 = *(const float2*)(raw.kdot + row0 + 2 * lane);
        float kr[2] = {0.f, 0.f};
        const int nv = chunk_valid<kPacked>(d, (int)(ch % d.NC));
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int t = t0 + 2 * lane + e;
            ga[e] = __float2bfloat16_rn(kRaw ? -INFINITY : 1.f);
            gb[e] = __float2bfloat16_rn(kRaw ? -INFINITY : 0.f);
            if (kPacked ? 2 * lane + e < nv : t < d.T) {
                const int64_t gi = ((int64_t)b * d.T + t) * d.H + h;
                ga[e] = alpha[gi];
                gb[e] = beta[gi];
                if (kRaw) kr[e] = raw.rk[gi];
            }
        }
        kv = make_float2(kr[0], kr[1]);
    };

    const int64_t first = blockIdx.x;
    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        if (first < nchunks) load_inputs(first);
    }
    if (warp == 1) {
        tmem_alloc(tslot, 256);
        tmem_relinquish();
    }
    int claimed = 0;  // lane 0 of warp 3: the next chunk, claimed a chunk ahead
    if (warp == 3 && first < nchunks) {
        load_vec(first);
        if (lane == 0) claimed = (int)gridDim.x + atomicAdd(err + kSchedWy, 1);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t lanebase = (uint32_t)(sub * 32) << 16;
    // TMEM columns: Qm 0-63, P 64-127, Y 128-191, KK 192-255; then dA over Y,
    // dV over Qm/P (128 columns), dK over dV (128 columns)
    const uint32_t tQm = tmem, tP = tmem + 64, tY = tmem + 128, tKK = tmem + 192;
    const uint32_t tDA = tY, tDV = tmem, tDK = tmem;
    const uint32_t sK = smem_u32(sm + wy::K), sV = smem_u32(sm + wy::V), sDU = smem_u32(sm + wy::DU);
    const uint32_t sDWT = smem_u32(sm + wy::DWT), sT = smem_u32(sm + wy::T);
    const uint32_t sT1 = smem_u32(sm + wy::T1), sT2 = smem_u32(sm + wy::T2), sDT = smem_u32(sm + wy::DT);
    const uint32_t sY = smem_u32(sm + wy::Y), sE = smem_u32(sm + wy::E), sID = smem_u32(sm + wy::ID);
    const uint32_t sKP = smem_u32(sm + wy::KP);


    bool ok = true;
    int n = 0;
    // thread 0, this chunk: bit 0 the next chunk's inputs requested, bit 1 the dK
    // partial requested, bits 2+ MMA commits
    int trk = 0;
    int64_t nxt = first;
#pragma unroll 1
    for (int64_t ch = first; ch < nchunks; ch = nxt, ++n) {
        const int ph = n & 1;
        int b, h, t0;
        decode(ch, b, h, t0);
        const int nv = chunk_valid<kPacked>(d, (int)(ch % d.NC));  // tokens of the chunk
        // a packed sequence's last chunk of fewer than 64 tokens: dk and dv rows are
        // copied by warp 0 (the rows after them belong to the next sequence)
        const bool out_tma = !kPacked || nv == kC;
        auto copy_rows = [&](bf16* dst, int width, const unsigned char* tile) {
            if constexpr (kPacked) {
                for (int i = lane; i < nv * (kD / 8); i += 32) {
                    const int t = i / (kD / 8), c8 = 8 * (i % (kD / 8));
                    if (c8 < width)
                        *(uint4*)(dst + ((int64_t)(t0 + t) * d.H + h) * width + c8) =
                            *(const uint4*)(tile + (c8 >> 6) * 8192 + sw128_off(t, c8 & 63));
                }
            }
        };
        const int krow0 = (int)(ch * kD);
        trk = 0;
        if (warp == 3) {
            const int nx = __shfl_sync(0xffffffffu, claimed, 0);
            if (lane == 0) {
                *s_next = nx;
                if (nx < nchunks) claimed = (int)gridDim.x + atomicAdd(err + kSchedWy, 1);
            }
            const float g2[2] = {gv.x, gv.y}, q2[2] = {qv.x, qv.y}, k2[2] = {kv.x, kv.y}, kd2[2] = {dv2.x, dv2.y};
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int p = 2 * lane + e;
                Gs[p] = g2[e];
                gs[p] = expf(g2[e]);
                dGq[p] = q2[e];
                if (kRaw) {  // alpha = sigmoid(-a), beta = sigmoid(b)
                    const float a = __bfloat162float(ga[e]), bl = __bfloat162float(gb[e]);
                    as_[p] = 1.f / (1.f + expf(a));
                    sas[p] = 1.f / (1.f + expf(-a));
                    bs[p] = 1.f / (1.f + expf(-bl));
                    rks[p] = k2[e];
                    kds[p] = kd2[e];
                } else {
                    bs[p] = __bfloat162float(gb[e]);
                    as_[p] = __bfloat162float(ga[e]);
                }
            }
            if (nx < nchunks) load_vec(nx);  // used next iteration
        }
        __syncthreads();  // per-token values and the next chunk's index visible
        fence_after_sync();
        nxt = *s_next;
        const bool has_next = nxt < nchunks;
        ok = mbar_wait(&bars[0], ph, err, 1, d.wait_ns) && ok;
        // ---- phase 1: Qm = dW K^T (K over k), P = dU V^T (K over v), KK = K K^T   (M=128: rows 64-127 unused)
        if (tid == 0 && ok) {
            const uint32_t idq = idesc_bf16(128, 64, true, false);
            const uint32_t id = idesc_bf16(128, 64, false, false);
            const uint64_t ddw = sdesc(sDWT, 16384, 1024, SW_128B);
            const uint64_t dk = sdesc(sK, 16, 1024, SW_128B), du = sdesc(sDU, 16, 1024, SW_128B);
            const uint64_t dv = sdesc(sV, 16, 1024, SW_128B);
#pragma unroll
            for (int s2 = 0; s2 < 8; ++s2) {
                const uint32_t o = (s2 >> 2) * 8192 + (s2 & 3) * 32;
                mma_bf16_ss(tQm, desc_add(ddw, s2 * 2048), desc_add(dk, o), idq, s2 > 0);
                mma_bf16_ss(tP, desc_add(du, o), desc_add(dv, o), id, s2 > 0);
                mma_bf16_ss(tKK, desc_add(dk, o), desc_add(dk, o), id, s2 > 0);
            }
            // the previous chunk's dK store has read the dT / Y tiles before anyone
            // sees this commit (dT is written after it)
            bulk_wait_read0();
            mma_commit(&bars[1]);
            trk += 4;
        }
        if (!urow) {
            // T1 = T diag(beta gamma), T2 = T diag(beta): rows r, this half of the columns
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float f[8], f1[8], f2[8];
                tile_get8(sm + wy::T, 64, r, cb + 8 * q, f);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int cc = cb + 8 * q + j;
                    f2[j] = f[j] * bs[cc];
                    f1[j] = f2[j] * gs[cc];
                }
                *(uint4*)(sm + wy::T1 + tile_off(64, r, cb + 8 * q)) = pack8(f1);
                *(uint4*)(sm + wy::T2 + tile_off(64, r, cb + 8 * q)) = pack8(f2);
            }
        }
        ok = mbar_wait(&bars[1], 0, err, 2, d.wait_ns) && ok;
        __syncwarp();
        fence_after_sync();
        // V is dead: bring in the dK partial of the first gradient kernel for phase 4
        if (tid == 0 && ok) {
            mbar_arrive_expect_tx(&bars[2], 2 * 8192);
            for (int j = 0; j < 2; ++j) tma_load_2d(sm + wy::KP + j * 8192, &tm_dKp, &bars[2], 0, krow0 + 64 * j);
            trk |= 2;
        }
        if (urow) {
            // rows s = r: column sums of T (P + Qm diag(gamma)) and T Qm over this warp's 32
            // rows; dT (strictly lower) for the Y product
#pragma unroll
            for (int c0 = 0; c0 < 32; c0 += 16) {
                float qm[16], p[16], t8a[8], t8b[8], dt[16], c1[16], c2[16];
                tmem_load16f2(tQm + lanebase + cb + c0, tP + lanebase + cb + c0, qm, p);
                tile_get8(sm + wy::T, 64, r, cb + c0, t8a);
                tile_get8(sm + wy::T, 64, r, cb + c0 + 8, t8b);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int rc = cb + c0 + j;
                    const float tsr = j < 8 ? t8a[j] : t8b[j - 8];
                    const float pv = p[j] + gs[rc] * qm[j];
                    c1[j] = tsr * pv;
                    c2[j] = tsr * qm[j];
                    dt[j] = (rc < r) ? bs[rc] * pv : 0.f;
                }
                tile_put16(sm + wy::DT, 64, r, cb + c0, dt);
                const float s1 = warp_colsum16(c1), s2 = warp_colsum16(c2);
                if (lane < 16) {
                    cB12[sub * 64 + cb + c0 + lane] = s1;
                    cGw[sub * 64 + cb + c0 + lane] = s2;
                }
            }
        }
        fence_proxy_async();
        fence_before_sync();
        ok = __syncthreads_and(ok);
        fence_after_sync();
        // ---- phase 2: Y = dT T^T  (M=128, K over tokens); then dV = T2^T dU (N=128,
        // tokens on rows 64-127: T2 and dU are ready and Qm / P, whose columns it
        // takes, were read before the barrier), which runs during the Y epilogue
        // and is covered by phase 3's commit
        if (tid == 0 && ok) {
            const uint32_t id = idesc_bf16(128, 64, false, false);
            const uint64_t ddt = sdesc(sDT, 16, 1024, SW_128B), dt = sdesc(sT, 16, 1024, SW_128B);
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2) mma_bf16_ss(tY, desc_add(ddt, s2 * 32), desc_add(dt, s2 * 32), id, s2 > 0);
            mma_commit(&bars[1]);
            trk += 4;
            const uint32_t idv = idesc_bf16(128, 128, true, true);
            const uint64_t dt2m = sdesc(sT2 - 8192, 8192, 1024, SW_128B), dum = sdesc(sDU, 8192, 1024, SW_128B);
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2)
                mma_bf16_ss(tDV, desc_add(dt2m, s2 * 2048), desc_add(dum, s2 * 2048), idv, s2 > 0);
        }
        if (ok) ok = mbar_wait(&bars[1], 1, err, 4, d.wait_ns);
        __syncwarp();
        fence_after_sync();
        if (urow) {
            float y[16], y2[16];
            tmem_load16f2(tY + lanebase + cb, tY + lanebase + cb + 16, y, y2);
            tile_put16(sm + wy::Y, 64, r, cb, y);
            tile_put16(sm + wy::Y, 64, r, cb + 16, y2);
        }
        fence_proxy_async();
        fence_before_sync();
        ok = __syncthreads_and(ok);
        fence_after_sync();
        // ---- phase 3: dA = -T^T Y (N=64, rows 0-63); its commit also covers dV
        if (tid == 0 && ok) {
            const uint32_t ida = idesc_bf16(128, 64, true, true, true);
            const uint64_t dtm = sdesc(sT, 8192, 1024, SW_128B), dym = sdesc(sY, 8192, 1024, SW_128B);
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2)
                mma_bf16_ss(tDA, desc_add(dtm, s2 * 2048), desc_add(dym, s2 * 2048), ida, s2 > 0);
            mma_commit(&bars[1]);
            trk += 4;
        }
        if (ok) ok = mbar_wait(&bars[1], 0, err, 8, d.wait_ns);
        __syncwarp();
        fence_after_sync();
        if (urow) {
            // rows a = r: dbeta3, E = beta_a Gam .* dA (strictly lower) -> E tile, E2 = E .* KK
            const float Ga = Gs[r], ba = bs[r];
            float b3 = 0.f, re2 = 0.f;
#pragma unroll
            for (int c0 = 0; c0 < 32; c0 += 16) {
                float da[16], kk[16], ev[16], e2[16];
                tmem_load16f2(tDA + lanebase + cb + c0, tKK + lanebase + cb + c0, da, kk);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int bc = cb + c0 + j;
                    const float gam = (bc < r) ? __expf(Ga - Gs[bc]) : 0.f;
                    const float m = gam * da[j];
                    b3 += m * kk[j];
                    ev[j] = ba * m;
                    e2[j] = ev[j] * kk[j];
                    re2 += e2[j];
                }
                tile_put16(sm + wy::E, 64, r, cb + c0, ev);
                const float s3 = warp_colsum16(e2);
                if (lane < 16) cE2[sub * 64 + cb + c0 + lane] = s3;
            }
            dB3p[half * 64 + r] = b3;
            rE2p[half * 64 + r] = re2;
            // the identity for adding the dK partial by an MMA (Y is dead); with the raw
            // prologue also the zeros of diag(-k . dk) in the dead T2 tile
            if (half == 0) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float f[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) f[j] = (8 * q + j == r) ? 1.f : 0.f;
                    *(uint4*)(sm + wy::ID + sw128_off(r, 8 * q)) = pack8(f);
                }
            } else if (kRaw) {
#pragma unroll
                for (int q = 0; q < 8; ++q) *(uint4*)(sm + wy::T2 + sw128_off(r, 8 * q)) = make_uint4(0u, 0u, 0u, 0u);
            }
        } else {
            // dV row a = r (token), columns 64*half .. +64 -> dv tile (dU is dead)
            unsigned char* dvt = sm + wy::DV + half * 8192;
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                float x[32];
                tmem_cols<32>(tDV + lanebase + 64 * half + 32 * g, x);
#pragma unroll
                for (int q = 0; q < 4; ++q) *(uint4*)(dvt + sw128_off(r, 32 * g + 8 * q)) = pack8(x + 8 * q);
            }
        }
        fence_proxy_async();
        fence_before_sync();
        ok = __syncthreads_and(ok);
        fence_after_sync();
        if (kRaw && warp == 0) {
            // k . dk per token from sums this chunk already holds: k . dK part (grad_qk_tc),
            // k . T1^T dW = beta gamma (column sum of T .* Qm), k . (E + E^T) K = row and
            // column sums of E .* KK^T.  diag(-k . dk) on the diagonal tile; phase 4 adds
            // diag(-k . dk) K, so dk_raw = (dk - k (k . dk)) / |k_raw| is one row scaling.
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int t = lane + 32 * hh;
                const float sd = kds[t] + bs[t] * gs[t] * (cGw[t] + cGw[64 + t]) + (rE2p[t] + rE2p[64 + t]) +
                                 (cE2[t] + cE2[64 + t]);
                *(bf16*)(sm + wy::T2 + sw128_off(t, t)) = __float2bfloat16_rn(-sd);
            }
            fence_proxy_async();
            __syncwarp();
        }
        // ---- phase 4: dK = T1^T dW + E K + E^T K + dK_partial (N=128, tokens on rows 64-127)
        if (!out_tma && warp == 0 && ok) copy_rows(dv_rows, d.V, sm + wy::DV);
        if (tid == 0 && ok) {
            if (out_tma) {
                for (int j = 0; j < 2; ++j)
                    if (64 * j < d.V) tma_store_4d(&tm_dv, sm + wy::DV + j * 8192, 64 * j, h, t0, b);
                bulk_commit();
            }
            ok = mbar_wait(&bars[2], ph, err, 16, d.wait_ns);
            if (ok) {
                const uint32_t id_mk = idesc_bf16(128, 128, true, false);   // A MN-major, B K-major
                const uint32_t id_km = idesc_bf16(128, 128, false, true);   // A K-major, B MN-major
                const uint32_t id_mm = idesc_bf16(128, 128, true, true);
                const uint32_t id_kk = idesc_bf16(128, 128, false, false);
                const uint64_t dt1m = sdesc(sT1 - 8192, 8192, 1024, SW_128B), ddw = sdesc(sDWT, 16, 1024, SW_128B);
                const uint64_t dek = sdesc(sE - 8192, 16, 1024, SW_128B), dem = sdesc(sE - 8192, 8192, 1024, SW_128B);
                const uint64_t dkm = sdesc(sK, 8192, 1024, SW_128B);
                const uint64_t did = sdesc(sID - 8192, 16, 1024, SW_128B), dkp = sdesc(sKP, 16, 1024, SW_128B);
#pragma unroll
                for (int s2 = 0; s2 < 4; ++s2) {
                    mma_bf16_ss(tDK, desc_add(dt1m, s2 * 2048), desc_add(ddw, s2 * 32), id_mk, s2 > 0);
                    mma_bf16_ss(tDK, desc_add(dek, s2 * 32), desc_add(dkm, s2 * 2048), id_km, 1u);
                    mma_bf16_ss(tDK, desc_add(dem, s2 * 2048), desc_add(dkm, s2 * 2048), id_mm, 1u);
                    mma_bf16_ss(tDK, desc_add(did, s2 * 32), desc_add(dkp, s2 * 32), id_kk, 1u);
                }
                if (kRaw) {  // + diag(-k . dk) K (rows 0-63 of this A are the T1 tile, unused)
                    const uint64_t dsk = sdesc(smem_u32(sm + wy::T2 - 8192), 16, 1024, SW_128B);
#pragma unroll
                    for (int s2 = 0; s2 < 4; ++s2)
                        mma_bf16_ss(tDK, desc_add(dsk, s2 * 32), desc_add(dkm, s2 * 2048), id_km, 1u);
                }
                mma_commit(&bars[1]);
                trk += 4;
            }
        }
        if (warp == 1) {
            // dG, dlog alpha = reverse within-chunk cumsum (lane l holds positions 63-2l and
            // 62-2l), dalpha = dlog alpha / alpha, dbeta = dbeta12 + dbeta3
            auto dg = [&](int p) {
                return dGq[p] + bs[p] * gs[p] * (cGw[p] + cGw[64 + p]) + (rE2p[p] + rE2p[64 + p]) -
                       (cE2[p] + cE2[64 + p]);
            };
            const int p1 = 63 - 2 * lane, p0 = 62 - 2 * lane;
            const float g1 = dg(p1), g0 = dg(p0);
            const float pair = g1 + g0;
            float incl = pair;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            const float run1 = incl - pair + g1, run0 = run1 + g0;
            const int pos[2] = {p1, p0};
            const float run[2] = {run1, run0};
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = t0 + pos[e];
                if (kPacked ? pos[e] < nv : t < d.T) {
                    const int64_t gi = ((int64_t)b * d.T + t) * d.H + h;
                    const int p = pos[e];
                    const float dbv = cB12[p] + cB12[64 + p] + dB3p[p] + dB3p[64 + p];
                    if (kRaw) {  // d log alpha / da = -sigmoid(a); d beta / db = beta (1 - beta)
                        dalpha[gi] = __float2bfloat16_rn(-run[e] * sas[p]);
                        dbeta[gi] = __float2bfloat16_rn(dbv * bs[p] * (1.f - bs[p]));
                    } else {
                        dalpha[gi] = __float2bfloat16_rn(run[e] / as_[p]);
                        dbeta[gi] = __float2bfloat16_rn(dbv);
                    }
                }
            }
        }
        ok = __syncthreads_and(ok);  // the issuer's load wait is every thread's
        if (ok) ok = mbar_wait(&bars[1], 1, err, 16, d.wait_ns);
        __syncwarp();
        fence_after_sync();
        // every input slot is free (the dV store has read the dU slot): the next chunk's
        if (tid == 0 && ok && has_next) {
            bulk_wait_read0();
            load_inputs(nxt);
            trk |= 1;
        }
        if (!urow) {
            // dK row a = r (token), columns 64*half .. +64 -> dk tile (dT / E and Y / ID are dead)
            unsigned char* dkt = sm + wy::DK + half * 8192;
            const float rr = kRaw ? rks[r] : 1.f;  // dk_raw = (dk - k (k . dk)) / |k_raw|
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                float x[32];
                tmem_cols<32>(tDK + lanebase + 64 * half + 32 * g, x);
                if (kRaw) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) x[j] *= rr;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) *(uint4*)(dkt + sw128_off(r, 32 * g + 8 * q)) = pack8(x + 8 * q);
            }
        }
        fence_proxy_async();
        fence_before_sync();
        ok = __syncthreads_and(ok);
        fence_after_sync();
        if (tid == 0 && ok && out_tma) {
            for (int j = 0; j < 2; ++j)
                if (64 * j < d.K) tma_store_4d(&tm_dk, sm + wy::DK + j * 8192, 64 * j, h, t0, b);
            bulk_commit();
        }
        if (!out_tma && warp == 0 && ok) copy_rows(dk_rows, d.K, sm + wy::DK);
        if (!ok) break;
    }
    if (tid == 0) {
        if (!ok) {  // bounded waits for the copies and MMAs still in flight
            mbar_wait(&bars[0], n & 1, nullptr, 0);
            if (trk & 1) mbar_wait(&bars[0], (n + 1) & 1, nullptr, 0);
            if (trk & 2) mbar_wait(&bars[2], n & 1, nullptr, 0);
            if (trk >= 4) mbar_wait(&bars[1], ((trk >> 2) - 1) & 1, nullptr, 0);  // 4 commits per chunk
        }
        bulk_wait_read0();  // stores have read their tiles; their writes complete on their own
    }
    __syncwarp();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem, 256);
}

template <int Vt>
cudaError_t launch_scan_bwd_vt(const Dims& d, const void* q, const void* k, const void* d_o, const TcBufs& tb,
                               const float* dsT, const TcBwdBufs& bb, float* ds0, cudaStream_t st,
                               const SeqMap* sq) {
    using P = BScan<Vt>;
    CUtensorMap mq, mk, mW, mM, mdo, mdU, mdS1;
    const int64_t rows = d.NS() * d.NC * kC;
    if (!tmap_bthd(&mq, q, d.B, d.T, d.H, d.K) || !tmap_bthd(&mk, k, d.B, d.T, d.H, d.K) ||
        !tmap_rows(&mW, tb.W, rows, kD) || !tmap_rows(&mM, tb.Mqk, rows, kC) ||
        !tmap_core8_bthd(&mdo, d_o, d.B, d.T, d.H, d.V, Vt / 8) ||
        !tmap_core8_rows(&mdU, bb.dU, rows, kD, kC, Vt / 8) ||
        !tmap_core8_rows(&mdS1, bb.dS1, d.NS() * d.NC * kD, kD, kD, Vt / 8))
        return cudaErrorInvalidValue;
    auto kern = d.tok ? scan_bwd_tc<Vt, true> : scan_bwd_tc<Vt, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid((kD + Vt - 1) / Vt, d.H, sq ? sq->nseq : d.B);
    kern<<<grid, 320, P::SMEM, st>>>(d, mq, mk, mW, mM, mdo, mdU, mdS1, tb.G, dsT, ds0,
                                     sq ? sq->chunk_off : nullptr, (sq && sq->mode == 0) ? sq->order : nullptr,
                                     tb.err);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scan_bwd_tc(const Dims& d, const void* q, const void* k, const void* d_o, const TcBufs& tb,
                               const float* dsT, const TcBwdBufs& bb, float* ds0, cudaStream_t st,
                               const SeqMap* sq) {
    switch (tc_scan_vt_for(d, sq, sq ? (int64_t)sq->nseq * d.H : d.NS())) {
        case 16: return launch_scan_bwd_vt<16>(d, q, k, d_o, tb, dsT, bb, ds0, st, sq);
        case 32: return launch_scan_bwd_vt<32>(d, q, k, d_o, tb, dsT, bb, ds0, st, sq);
        case 48: return launch_scan_bwd_vt<48>(d, q, k, d_o, tb, dsT, bb, ds0, st, sq);
        default: return launch_scan_bwd_vt<64>(d, q, k, d_o, tb, dsT, bb, ds0, st, sq);
    }
}

cudaError_t launch_grad_qk_tc(const Dims& d, const void* q, const void* k, const void* d_o, const TcBufs& tb,
                              const __nv_bfloat16* states, const TcBwdBufs& bb, void* dq, cudaStream_t st,
                              const RawPrologue* rp) {
    // tb.Ut holds U: the forward scan that wrote the chunk-start states wrote U over U~
    CUtensorMap mq, mk, mdo, mU, mdU, mS0, mdS1, mdq, mdKp, mdWt;
    const int64_t rows = d.NS() * d.NC * kC;
    const int64_t krows = d.NS() * d.NC * kD;
    if (!tmap_bthd(&mq, q, d.B, d.T, d.H, d.K) || !tmap_bthd(&mk, k, d.B, d.T, d.H, d.K) ||
        !tmap_bthd(&mdo, d_o, d.B, d.T, d.H, d.V) || !tmap_rows(&mU, tb.Ut, rows, kD) ||
        !tmap_rows(&mdU, bb.dU, rows, kD) || !tmap_rows(&mS0, states, krows, kD) ||
        !tmap_rows(&mdS1, bb.dS1, krows, kD) || !tmap_bthd(&mdq, dq, d.B, d.T, d.H, d.K) ||
        !tmap_rows(&mdKp, bb.dKp, krows, kC) || !tmap_rows(&mdWt, bb.dWt, krows, kC))
        return cudaErrorInvalidValue;
    RawPrologue raw{};
    if (rp && rp->on) raw = *rp;
    auto kern = d.tok ? grad_qk_tc<false, true> : (raw.on ? grad_qk_tc<true, false> : grad_qk_tc<false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)qk::SMEM);
    if (e != cudaSuccess) return e;
    const int64_t nchunks = d.NS() * d.NC;
    dim3 grid((unsigned)std::min<int64_t>(nchunks, sm_count()));
    kern<<<grid, 512, qk::SMEM, st>>>(d, mq, mk, mdo, mU, mdU, mS0, mdS1, mdq, mdKp, mdWt, tb.Mqk, tb.G,
                                            bb.dGp, raw, (bf16*)dq, tb.err);
    return cudaGetLastError();
}

cudaError_t launch_grad_wy_tc(const Dims& d, const void* k, const void* v, const void* alpha, const void* beta,
                              const TcBufs& tb, const TcBwdBufs& bb, void* dk, void* dv, void* dalpha, void* dbeta,
                              cudaStream_t st, const RawPrologue* rp) {
    CUtensorMap mk, mv, mdWt, mdU, mT, mdk, mdv, mdKp;
    const int64_t rows = d.NS() * d.NC * kC;
    const int64_t krows = d.NS() * d.NC * kD;
    if (!tmap_bthd(&mk, k, d.B, d.T, d.H, d.K) || !tmap_bthd(&mv, v, d.B, d.T, d.H, d.V) ||
        !tmap_rows(&mdWt, bb.dWt, krows, kC) || !tmap_rows(&mdU, bb.dU, rows, kD) ||
        !tmap_rows(&mT, tb.T, rows, kC) || !tmap_bthd(&mdk, dk, d.B, d.T, d.H, d.K) ||
        !tmap_bthd(&mdv, dv, d.B, d.T, d.H, d.V) || !tmap_rows(&mdKp, bb.dKp, krows, kC))
        return cudaErrorInvalidValue;
    RawPrologue raw{};
    if (rp && rp->on) raw = *rp;
    auto kern = d.tok ? grad_wy_tc<false, true> : (raw.on ? grad_wy_tc<true, false> : grad_wy_tc<false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wy::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)std::min<int64_t>(d.NS() * d.NC, 2 * sm_count()));
    kern<<<grid, 256, wy::SMEM, st>>>(d, mk, mv, mdWt, mdU, mT, mdk, mdv, mdKp, (const bf16*)alpha,
                                            (const bf16*)beta, tb.G, bb.dGp, (bf16*)dalpha, (bf16*)dbeta, raw,
                                            (bf16*)dk, (bf16*)dv, tb.err);
    return cudaGetLastError();
}

}  // namespace gdn
