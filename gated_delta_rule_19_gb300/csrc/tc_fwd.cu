// tc_fwd.cu -- tensor-core (tcgen05 + TMA) forward for bf16 inputs, chunk 64, K and V
// of 16 to 128 (tiles and buffers 128 wide; TMA fills the columns past K or V with
// zeros).  Dense tensors, or a packed batch read in place (kPacked).
//
// prep_fwd_tc (chunk-parallel; persistent, two CTAs per SM; "Sparse Delta Memory:
// layer and kernels", "What the layer computes", Phase 1 and Solve):
//   TMA loads of the chunk's K, Q, V tiles (128B-swizzled, K-major), the next
//   chunk's requested as the current one's MMAs release them;
//   one M=128 MMA gives [K;Q] K^T = [K K^T ; Q K^T] in TMEM;
//   A = strict_lower(beta_r Gam_ri (K K^T)_ri) -> fp32 solve T = (I + A)^-1
//   (16x16 diagonal blocks in registers, off-diagonal blocks in shared memory);
//   Mqk = lower(Gam .* Q K^T) -> bf16;
//   T1 = T diag(beta gamma), T2 = T diag(beta) (bf16), then one M=128, N=256 MMA
//   [T1; T2] [K | V] whose rows 0-63 of columns 0-127 are W = T1 K and rows 64-127
//   of columns 128-255 are Ut = T2 V (K and V read MN-major from their tiles);
//   W, Ut, Mqk leave through TMA stores as bf16 [rows = chunk*64 + r][...].
//
// scan_fwd_tc (one CTA per (V-slice of Vt rows, head, batch); Phase 2):
//   the state slice S^T [K=128, Vt] lives in registers (fp32, thread k = row k) and
//   as a bf16 MMA operand in shared memory; per chunk
//     [X; Y] = [W; Q] S0^T            (one M=128 MMA)
//     U = Ut - X,  Uh = diag(exp(G_C - G)) U
//     S1^T = gamma_C S0^T + K^T Uh    (M=128 MMA, on the chunk-to-chunk chain)
//     O = diag(gamma) Y + Mqk U       (M=128 MMA, rows 64-127)
//   with warps 0-7 on the epilogues, warp 8 issuing the MMAs and warp 9 the TMA
//   copies, and the next chunks' tiles prefetched NS stages ahead.  A scan that
//   writes the chunk-start states for the backward also writes U (bf16) in place
//   over its U~ slice: the backward's chunk gradients read U, never U~.
//
// Every wait is bounded (2 s unless a test sets a shorter limit); a wait that gives
// up raises the error flag, and the block leaves its loop together (block-wide
// vote) after draining its copies.

#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>

#include "gdn_internal.h"
#include "tc.cuh"

namespace gdn {
namespace {

using namespace tc;
using bf16 = __nv_bfloat16;

constexpr int kC = 64;
constexpr int kD = 128;  // tile width of K and V (narrower K, V: zero columns)

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNormEps = 1e-6f;  // q, k normalisation: x / sqrt(sum x^2 + eps)

constexpr int kAS = 68;  // fp32 row stride of A and T in shared memory (16-byte aligned rows)
constexpr int kXS = 36;  // fp32 row stride of the solve's scratch block

// T = (I + A)^-1 for strictly lower A (64 x 64 fp32, rows kAS floats apart), by
// 256 threads in five steps separated by barriers:
//   1. the four 16x16 diagonal blocks T_II by forward substitution, one column
//      per thread (threads 0-63), zeros stored above their diagonals;
//   2-3. T_10 = -T_11 A_10 T_00 and T_32 = -T_33 A_32 T_22;
//   4-5. the lower-left 32x32 block -T_bb A_ba T_aa, where T_aa and T_bb are the
//      two 32x32 diagonal blocks finished by steps 1-3.
// Entries above the diagonal outside the 16x16 diagonal blocks stay unwritten.
__device__ void solve_unit_lower_64(const float* A, float* Tf, float* X) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid < 64) {
        const int bo = (tid >> 4) * 16, c = tid & 15;
        float t[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const float* ar = A + (bo + r) * kAS + bo;
            float acc = 0.f;
#pragma unroll
            for (int i4 = 0; i4 < r; i4 += 4) {
                const float4 a = *(const float4*)(ar + i4);
                acc = fmaf(a.x, t[i4], acc);
                if (i4 + 1 < r) acc = fmaf(a.y, t[i4 + 1], acc);
                if (i4 + 2 < r) acc = fmaf(a.z, t[i4 + 2], acc);
                if (i4 + 3 < r) acc = fmaf(a.w, t[i4 + 3], acc);
            }
            t[r] = (r == c) ? 1.f : ((r < c) ? 0.f : -acc);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) Tf[(bo + r) * kAS + bo + c] = t[r];
    }
    __syncthreads();
    // steps 2-3: warps 0-3 block I = 1, warps 4-7 block I = 3; this warp's 4
    // columns start at cq, lane -> row r and a column pair
    const int blk = warp >> 2, I = 1 + 2 * blk, cq = (warp & 3) * 4;
    const int r16 = lane & 15, cp = cq + 2 * (lane >> 4);
    {
        const float* ar = A + (16 * I + r16) * kAS + 16 * (I - 1);
        const float* tc = Tf + 16 * (I - 1) * kAS + 16 * (I - 1) + cp;
        float x0 = 0.f, x1 = 0.f;
#pragma unroll
        for (int m4 = 0; m4 < 16; m4 += 4) {
            if (m4 + 3 < cq) continue;  // T_{I-1,I-1}[m][c] = 0 for m < c (warp-uniform)
            const float4 a = *(const float4*)(ar + m4);
            const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 tv = *(const float2*)(tc + (m4 + e) * kAS);
                x0 = fmaf(av[e], tv.x, x0);
                x1 = fmaf(av[e], tv.y, x1);
            }
        }
        *(float2*)(X + (16 * blk + r16) * kXS + cp) = make_float2(x0, x1);
    }
    __syncthreads();
    {
        const float* tr = Tf + (16 * I + r16) * kAS + 16 * I;  // zeros above the diagonal
        const float* xc = X + 16 * blk * kXS + cp;
        float y0 = 0.f, y1 = 0.f;
#pragma unroll
        for (int m4 = 0; m4 < 16; m4 += 4) {
            const float4 a = *(const float4*)(tr + m4);
            const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 xv = *(const float2*)(xc + (m4 + e) * kXS);
                y0 = fmaf(av[e], xv.x, y0);
                y1 = fmaf(av[e], xv.y, y1);
            }
        }
        *(float2*)(Tf + (16 * I + r16) * kAS + 16 * (I - 1) + cp) = make_float2(-y0, -y1);
    }
    __syncthreads();
    // steps 4-5: lane -> row r of the lower-left block, warp -> 4 columns c0
    const int r = lane, c0 = warp * 4;
    {
        const float* ar = A + (32 + r) * kAS;
        float x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
        for (int m4 = c0; m4 < 32; m4 += 4) {  // T_aa[m][c] = 0 for m < c
            const float4 a = *(const float4*)(ar + m4);
            const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 tv = *(const float4*)(Tf + (m4 + e) * kAS + c0);
                x[0] = fmaf(av[e], tv.x, x[0]);
                x[1] = fmaf(av[e], tv.y, x[1]);
                x[2] = fmaf(av[e], tv.z, x[2]);
                x[3] = fmaf(av[e], tv.w, x[3]);
            }
        }
        *(float4*)(X + r * kXS + c0) = make_float4(x[0], x[1], x[2], x[3]);
    }
    __syncthreads();
    {
        const float* tr = Tf + (32 + r) * kAS + 32;
        float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
        for (int m4 = 0; m4 <= r; m4 += 4) {  // T_bb[r][m] = 0 for m > r; m4 + 3 stays in r's 16-block
            const float4 a = *(const float4*)(tr + m4);
            const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 xv = *(const float4*)(X + (m4 + e) * kXS + c0);
                y[0] = fmaf(av[e], xv.x, y[0]);
                y[1] = fmaf(av[e], xv.y, y[1]);
                y[2] = fmaf(av[e], xv.z, y[2]);
                y[3] = fmaf(av[e], xv.w, y[3]);
            }
        }
        *(float4*)(Tf + (32 + r) * kAS + c0) = make_float4(-y[0], -y[1], -y[2], -y[3]);
    }
    __syncthreads();
}

// Shared-memory plan of prep_fwd_tc (offsets from a 1024-aligned base).  The Gram
// MMA reads [K_0; Q_0] and [K_1; Q_1] as M=128 K-major operands (rows 64-127 of a
// K-major tile lie 8 KB after rows 0-63); the W / Ut MMA reads K_0, K_1, V_0, V_1
// as one N=256 MN-major operand (64-wide blocks 16 KB apart).  W and Ut are staged
// for their stores in the fp32 T and A regions, dead by then, so that the input
// slots can take the next chunk's tiles as soon as the MMAs reading them are done.
constexpr int P_K0 = 0, P_Q0 = 8192, P_K1 = 16384, P_Q1 = 24576;
constexpr int P_V0 = 32768, P_M = 40960;   // V_1 at P_V0 + 16384; P_M: the Mqk output tile
constexpr int P_AF = 57344;                // fp32 A [64][kAS], dead before T1 / T2 exist
constexpr int P_T1 = 65536, P_T2 = 73728;  // [T1; T2]: one M=128 K-major operand
constexpr int P_TF = 81920;                // fp32 T [64][kAS]
constexpr int P_US = P_AF, P_WS = P_TF;    // Ut / W output tiles [64 x 128] (two 8 KB halves)
constexpr int P_X = P_TF + 64 * kAS * 4;   // fp32 [32][kXS] solve scratch
constexpr int P_VEC = P_X + 32 * kXS * 4;  // G (log2 units), gamma, beta
constexpr int P_BAR = P_VEC + 3 * 64 * 4;
constexpr int P_END = P_BAR + 64;
constexpr size_t kPrepSmem = P_END + 1024;
static_assert(P_K1 == P_K0 + 16384 && P_Q1 == P_Q0 + 16384, "64-column halves 16 KB apart");
static_assert(P_AF + 64 * kAS * 4 <= P_T2 + 8192, "A overlaps only T1 / T2");
static_assert(P_WS + 16384 <= P_X && P_US + 16384 <= P_T2 + 8192, "output tiles fit the dead regions");
static_assert(2 * (kPrepSmem + 1024) <= 228 * 1024, "two CTAs per SM");

// Persistent, two CTAs per SM, 256 threads: CTA i takes chunks i, i + gridDim.x, ...
// Warps w and w+4 read the same TMEM lane quarter (w % 4) and split its columns.
// A chunk's Q tiles are replaced by the next chunk's once the Gram MMA is done, its
// K and V tiles once the W / Ut MMA is done (both requested by thread 128, whose
// warp has no Gram epilogue work); warp 2 keeps the next chunk's gates in registers.
template <bool kRaw, bool kPacked>
__global__ void __launch_bounds__(256, 2)
prep_fwd_tc(Dims d, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_W,
            const __grid_constant__ CUtensorMap tm_U, const __grid_constant__ CUtensorMap tm_M,
            const bf16* __restrict__ alpha, const bf16* __restrict__ beta, float* __restrict__ Gout,
            bf16* __restrict__ Tout, RawPrologue raw, int* err) {
    extern __shared__ unsigned char smraw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    float* Af = (float*)(sm + P_AF);
    float* Tf = (float*)(sm + P_TF);
    float* G2s = (float*)(sm + P_VEC);  // within-chunk cumsum of log2(alpha)
    float* gs = G2s + 64;               // gamma = alpha_1 ... alpha_r
    float* bs = gs + 64;
    // [0] Q loads, [1] K loads, [2] Gram MMA, [3] W / Ut MMA, [4] V loads
    uint64_t* bars = (uint64_t*)(sm + P_BAR);
    uint32_t* tslot = (uint32_t*)(sm + P_BAR + 40);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sub = warp & 3, half = warp >> 2;
    const int64_t nchunks = d.NS() * d.NC;
    constexpr int kLoader = 128;

    // chunk index = (b * H + h) * NC + c; its first token (a packed batch: from the
    // chunk-token map)
    auto decode = [&](int64_t ch, int& b, int& h, int& t0) {
        t0 = chunk_tok<kPacked>(d, (int)(ch % d.NC));
        const int64_t bh = ch / d.NC;
        h = (int)(bh % d.H);
        b = (int)(bh / d.H);
    };
    auto load_q = [&](int64_t ch) {
        int b, h, t0;
        decode(ch, b, h, t0);
        mbar_arrive_expect_tx(&bars[0], 2 * 8192);
        for (int j = 0; j < 2; ++j) tma_load_4d(sm + P_Q0 + j * 16384, &tm_q, &bars[0], 64 * j, h, t0, b);
    };
    // K (the next Gram MMA waits for it) and V (only the W / Ut MMA reads it)
    auto load_k = [&](int64_t ch) {
        int b, h, t0;
        decode(ch, b, h, t0);
        mbar_arrive_expect_tx(&bars[1], 2 * 8192);
        for (int j = 0; j < 2; ++j) tma_load_4d(sm + P_K0 + j * 16384, &tm_k, &bars[1], 64 * j, h, t0, b);
    };
    auto load_v = [&](int64_t ch) {
        int b, h, t0;
        decode(ch, b, h, t0);
        mbar_arrive_expect_tx(&bars[4], 2 * 8192);
        for (int j = 0; j < 2; ++j) tma_load_4d(sm + P_V0 + j * 16384, &tm_v, &bars[4], 64 * j, h, t0, b);
    };
    // warp 2: gates of tokens 2 lane, 2 lane + 1 of a chunk; padding (alpha = 1,
    // beta = 0) leaves the state unchanged
    bf16 ga[2], gb[2];
    // (with kRaw the gate logits; padding a = b = -inf gives alpha = 1, beta = 0)
    auto load_gates = [&](int64_t ch) {
        int b, h, t0;
        decode(ch, b, h, t0);
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
            }
        }
    };

    // chunks position-major, descending: the forward scan starts with every stream's
    // chunk 0, which is then the last one written (still in L2)
    const int64_t first = d.chunk_of(blockIdx.x, true);
    if (tid == 0) {
        for (int i = 0; i < 5; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        if (first < nchunks) {
            load_q(first);
            load_k(first);
            load_v(first);
        }
    }
    if (warp == 1) {
        tmem_alloc(tslot, 256);
        tmem_relinquish();
    }
    if (warp == 2 && first < nchunks) load_gates(first);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    bool ok = true;
    int n = 0;
    int nq = first < nchunks ? 1 : 0, nk = nq, nv = nq;  // load batches issued (thread kLoader's count)
    int g_last = -1, w_last = -1;               // chunks whose MMAs were issued (thread 0)
#pragma unroll 1
    for (int64_t wi = blockIdx.x; wi < nchunks; wi += gridDim.x, ++n) {
        const int ph = n & 1;
        const int64_t ch = d.chunk_of(wi, true);
        const int64_t nxt = d.chunk_of(wi + gridDim.x, true);
        const bool has_next = nxt < nchunks;
        const int row0 = (int)(ch * kC);
        if (kRaw) {
            // Raw q, k rows to unit length as they land, before the Gram MMA reads them
            // (q = q_raw (sum q_raw^2 + 1e-6)^-1/2, the same for k): 16 consecutive lanes
            // hold the 16-byte pieces of one row (both 64-column halves), so every access
            // is conflict-free; rows 0-63 are the K tile's, 64-127 the Q tile's.
            int b, h, t0;
            decode(ch, b, h, t0);
            ok = mbar_wait(&bars[0], ph, err, 1, d.wait_ns) && ok;
            ok = mbar_wait(&bars[1], ph, err, 1, d.wait_ns) && ok;
            const int pc = tid & 15, hf = pc >> 3, p = pc & 7;
#pragma unroll 2
            for (int it = 0; it < 8; ++it) {
                const int rowid = it * 16 + (tid >> 4);
                const bool isq = rowid >= 64;
                const int rr = rowid & 63;
                unsigned char* ptr = sm + (isq ? P_Q0 : P_K0) + hf * 16384 + rr * 128 + p * 16;
                const uint4 x = *(const uint4*)ptr;
                const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) ss += bf_lo(w4[e]) * bf_lo(w4[e]) + bf_hi(w4[e]) * bf_hi(w4[e]);
#pragma unroll
                for (int off = 1; off < 16; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                const float rn = rsqrtf(ss + kNormEps);
                uint32_t o4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) o4[e] = pack_bf16(rn * bf_lo(w4[e]), rn * bf_hi(w4[e]));
                const uint4 y = make_uint4(o4[0], o4[1], o4[2], o4[3]);
                *(uint4*)ptr = y;
                // the normalised row's global copy, for the scan and the backward: smem piece
                // p holds columns 8 (p ^ (rr % 8)) .. +8 of its 128B-swizzled half row
                const int t = t0 + rr;
                const int col = 64 * hf + 8 * (p ^ (rr & 7));  // K is a multiple of 8
                if (t < d.T && col < d.K)
                    *(uint4*)((isq ? raw.qn : raw.kn) + (((int64_t)b * d.T + t) * d.H + h) * d.K + col) = y;
                if (pc == 0 && t < d.T) (isq ? raw.rq : raw.rk)[((int64_t)b * d.T + t) * d.H + h] = rn;
            }
            fence_proxy_async();
            fence_before_sync();
            ok = __syncthreads_and(ok);
            fence_after_sync();
            if (!ok) break;
        }
        if (tid == 0) {
            ok = mbar_wait(&bars[0], ph, err, 1, d.wait_ns) && ok;
            ok = mbar_wait(&bars[1], ph, err, 1, d.wait_ns) && ok;
            if (ok) {
                // [K; Q] K^T = [K K^T ; Q K^T] into columns 0-63 (M=128, N=64, K over k)
                const uint32_t id = idesc_bf16(128, 64, false, false);
                const uint32_t base = smem_u32(sm + P_K0);
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t a = base + (s >> 2) * 16384 + (s & 3) * 32;
                    mma_bf16_ss(tmem, sdesc(a, 16, 1024, SW_128B), sdesc(a, 16, 1024, SW_128B), id, s > 0);
                }
                mma_commit(&bars[2]);
                g_last = n;
            }
            bulk_wait_read0();  // the previous chunk's stores have read the A, T and Mqk tiles
        }
        if (warp == 2) {
            // log2 alpha, beta; from the logits: log alpha = -softplus(a), beta = sigmoid(b)
            float l[2], bv[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                if (kRaw) {
                    const float a = __bfloat162float(ga[e]), bl = __bfloat162float(gb[e]);
                    const float sp = a > 0.f ? a + log1pf(expf(-a)) : log1pf(expf(a));
                    l[e] = -sp * kLog2e;
                    bv[e] = 1.f / (1.f + expf(-bl));
                } else {
                    l[e] = log2f(__bfloat162float(ga[e]));
                    bv[e] = __bfloat162float(gb[e]);
                }
            }
            const float pair = l[0] + l[1];
            float incl = pair;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            const float g0 = incl - pair + l[0], g1 = incl;
            G2s[2 * lane] = g0;
            G2s[2 * lane + 1] = g1;
            gs[2 * lane] = exp2f(g0);
            gs[2 * lane + 1] = exp2f(g1);
            bs[2 * lane] = bv[0];
            bs[2 * lane + 1] = bv[1];
            constexpr float kLn2 = 0.693147180559945309f;
            *(float2*)(Gout + (int64_t)row0 + 2 * lane) = make_float2(g0 * kLn2, g1 * kLn2);
            if (has_next) load_gates(nxt);  // consumed next iteration
        }
        __syncthreads();  // gates visible; the output tiles are writable
        ok = mbar_wait(&bars[2], ph, err, 2, d.wait_ns) && ok;
        __syncwarp();
        fence_after_sync();
        if (tid == kLoader && ok && has_next) {  // the Q tiles are free
            load_q(nxt);
            ++nq;
        }
        // Gram epilogue: lanes 0-63 hold rows of K K^T -> A (fp32), lanes 64-127 rows of
        // Q K^T -> Mqk (bf16 tile); this warp takes columns cb .. cb+31.  Rows past the
        // chunk's tokens (a packed batch's ragged chunk reads the next sequence's rows)
        // are zero in Mqk; in A their beta is 0.
        {
            const int rr = 32 * (sub & 1) + lane;
            const int nv_rows = kPacked ? chunk_valid<true>(d, (int)(ch % d.NC)) : kC;
            const int cb = 32 * half;
            const bool any = cb <= 32 * (sub & 1) + 31;  // warp-uniform: some column on or below the diagonal
            const float G2r = G2s[rr];
            if (sub < 2) {
                if (any) {
                    uint32_t v[32];
                    tmem_ld32(tmem + ((uint32_t)(32 * sub) << 16) + cb, v);
                    tmem_wait_ld(v);
                    const float br = bs[rr];
                    float* arow = Af + rr * kAS + cb;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        float f[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i = cb + 4 * q + e;
                            f[e] = (i < rr) ? br * fast_exp2(G2r - G2s[i]) * __uint_as_float(v[4 * q + e]) : 0.f;
                        }
                        *(float4*)(arow + 4 * q) = make_float4(f[0], f[1], f[2], f[3]);
                    }
                }
            } else {
                unsigned char* mt = sm + P_M;
                if (any) {
                    uint32_t v[32];
                    tmem_ld32(tmem + ((uint32_t)(32 * sub) << 16) + cb, v);
                    tmem_wait_ld(v);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t pk[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i = cb + 8 * q + 2 * e;
                            const bool live = !kPacked || rr < nv_rows;
                            const float m0 =
                                (live && i <= rr) ? fast_exp2(G2r - G2s[i]) * __uint_as_float(v[8 * q + 2 * e]) : 0.f;
                            const float m1 = (live && i + 1 <= rr)
                                                 ? fast_exp2(G2r - G2s[i + 1]) * __uint_as_float(v[8 * q + 2 * e + 1])
                                                 : 0.f;
                            pk[e] = pack_bf16(m0, m1);
                        }
                        *(uint4*)(mt + sw128_off(rr, cb + 8 * q)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q) *(uint4*)(mt + sw128_off(rr, cb + 8 * q)) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
        }
        fence_proxy_async();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        if (tid == 0) {
            tma_store_2d(&tm_M, sm + P_M, 0, row0);
            bulk_commit();
        }
        solve_unit_lower_64(Af, Tf, (float*)(sm + P_X));  // ends with __syncthreads
        // B operands of W / Ut: T1 = T diag(beta gamma), T2 = T diag(beta), bf16 K-major
        // [r][i], zero above the diagonal; T itself to global memory when asked for.
        {
            const int r = tid >> 2, i0 = (tid & 3) * 16;
            const float* trow = Tf + r * kAS + i0;
            uint32_t p0[8], p1[8], p2[8];
#pragma unroll
            for (int e4 = 0; e4 < 16; e4 += 4) {
                const float4 t4 = *(const float4*)(trow + e4);
                float tv[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (i0 + e4 + e > r) tv[e] = 0.f;
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int i = i0 + e4 + e;
                    const float b0 = bs[i], b1 = bs[i + 1];
                    p0[(e4 + e) >> 1] = pack_bf16(tv[e], tv[e + 1]);
                    p1[(e4 + e) >> 1] = pack_bf16(tv[e] * b0 * gs[i], tv[e + 1] * b1 * gs[i + 1]);
                    p2[(e4 + e) >> 1] = pack_bf16(tv[e] * b0, tv[e + 1] * b1);
                }
            }
            if (Tout) {
                uint4* tg = (uint4*)(Tout + ((int64_t)row0 + r) * kC + i0);
                tg[0] = make_uint4(p0[0], p0[1], p0[2], p0[3]);
                tg[1] = make_uint4(p0[4], p0[5], p0[6], p0[7]);
            }
            *(uint4*)(sm + P_T1 + sw128_off(r, i0)) = make_uint4(p1[0], p1[1], p1[2], p1[3]);
            *(uint4*)(sm + P_T1 + sw128_off(r, i0 + 8)) = make_uint4(p1[4], p1[5], p1[6], p1[7]);
            *(uint4*)(sm + P_T2 + sw128_off(r, i0)) = make_uint4(p2[0], p2[1], p2[2], p2[3]);
            *(uint4*)(sm + P_T2 + sw128_off(r, i0 + 8)) = make_uint4(p2[4], p2[5], p2[6], p2[7]);
        }
        fence_proxy_async();
        fence_before_sync();
        ok = __syncthreads_and(ok);
        fence_after_sync();
        if (tid == 0) ok = mbar_wait(&bars[4], ph, err, 1, d.wait_ns) && ok;
        if (tid == 0 && ok) {
            // [T1; T2] [K | V] (M=128, N=256, K over tokens): rows 0-63 of columns 0-127
            // are W = T1 K, rows 64-127 of columns 128-255 are Ut = T2 V.
            const uint32_t id = idesc_bf16(128, 256, false, true);
            const uint64_t da = sdesc(smem_u32(sm + P_T1), 16, 1024, SW_128B);
            const uint64_t db = sdesc(smem_u32(sm + P_K0), 16384, 1024, SW_128B);
#pragma unroll
            for (int s = 0; s < 4; ++s) mma_bf16_ss(tmem, desc_add(da, s * 32), desc_add(db, s * 2048), id, s > 0);
            mma_commit(&bars[3]);
            w_last = n;
        }
        if (ok) ok = mbar_wait(&bars[3], ph, err, 4, d.wait_ns);
        __syncwarp();
        fence_after_sync();
        if (tid == kLoader && ok && has_next) {  // the K and V tiles are free
            load_k(nxt);
            load_v(nxt);
            ++nk;
            ++nv;
        }
        // Epilogue: row rr of W (lanes 0-63) or Ut (lanes 64-127), 64 columns per warp,
        // into the dead T (W) and A (Ut) regions as 128B-swizzled K-major tiles.
        {
            const int rr = 32 * (sub & 1) + lane;
            const bool isw = sub < 2;
            unsigned char* dst = sm + (isw ? P_WS : P_US) + half * 8192;
            const uint32_t taddr = tmem + ((uint32_t)(32 * sub) << 16) + (isw ? 0 : 128) + 64 * half;
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                uint32_t v[32];
                tmem_ld32(taddr + 32 * g, v);
                tmem_wait_ld(v);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        pk[e] = pack_bf16(__uint_as_float(v[8 * q + 2 * e]), __uint_as_float(v[8 * q + 2 * e + 1]));
                    *(uint4*)(dst + sw128_off(rr, 32 * g + 8 * q)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
            }
        }
        fence_proxy_async();
        fence_before_sync();
        ok = __syncthreads_and(ok);
        fence_after_sync();
        if (tid == 0 && ok) {
            tma_store_2d(&tm_W, sm + P_WS, 0, row0);
            tma_store_2d(&tm_W, sm + P_WS + 8192, 64, row0);
            tma_store_2d(&tm_U, sm + P_US, 0, row0);
            tma_store_2d(&tm_U, sm + P_US + 8192, 64, row0);
            bulk_commit();
        }
        if (!ok) break;
    }
    if (!ok) {  // bounded waits for what is still in flight before the CTA leaves
        if (tid == kLoader) {
            for (int i = n; i < nq; ++i) mbar_wait(&bars[0], i & 1, nullptr, 0);
            for (int i = n; i < nk; ++i) mbar_wait(&bars[1], i & 1, nullptr, 0);
            for (int i = n; i < nv; ++i) mbar_wait(&bars[4], i & 1, nullptr, 0);
        }
        if (tid == 0) {
            if (g_last == n) mbar_wait(&bars[2], n & 1, nullptr, 0);
            if (w_last == n) mbar_wait(&bars[3], n & 1, nullptr, 0);
        }
    }
    if (tid == 0) bulk_wait_read0();  // stores have read their tiles; their writes complete on their own
    __syncwarp();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------------------
template <int Vt>
struct ScanPlan {
    // TMA stages: three (two chunks of lead) where they fit, up to 48-column slices
    static constexpr int NS = Vt <= 48 ? 3 : 2;
    // stage: [W_0 | Q_0 | W_1 | Q_1] (stacked A of one M=128 MMA) | K_0 | K_1 | Mqk | Ut slice
    static constexpr int OFF_WQ = 0, OFF_K = 32768, OFF_M = 49152, OFF_UT = 57344;
    static constexpr int STAGE = 57344 + kC * Vt * 2;  // a multiple of 1024 (swizzled operands)
    static constexpr int S_OP = NS * STAGE;          // S0^T [Vt/8][128 k][8] (MN-major, no swizzle)
    static constexpr int U_OP = S_OP + kD * Vt * 2;  // U  [Vt/8][64 tok][8]
    static constexpr int UH_OP = U_OP + kC * Vt * 2; // Uh
    static constexpr int O_OP = UH_OP + kC * Vt * 2; // output tiles of chunk c in buffer c & 1, same layout
    static constexpr int BAR = O_OP + 2 * kC * Vt * 2;  // tma[NS], XY, S, O, then the TMEM slot at +48
    static constexpr int END = BAR + 64;
    static constexpr size_t SMEM = END + 1024;
    // TMEM: [X;Y] (two buffers), O2, DS, each Vt columns
    static constexpr uint32_t TMEM_COLS = (4 * Vt <= 32) ? 32 : (4 * Vt <= 64 ? 64 : (4 * Vt <= 128 ? 128 : 256));
};

// Loads W consecutive fp32 TMEM columns (W = 16, 24 or 32) of this thread's lane;
// 24 columns are three 8-column loads (each starting on a multiple of 8).
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
// Two W-column groups, one wait.
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

// 320 threads: warps 0-7 run the epilogues, warp 8 issues the MMAs and warp 9 the
// TMA copies (lane 0 of each), so no epilogue waits behind an instruction issue
// and the two issue streams run side by side.  Warp w < 8 reaches TMEM lanes
// 32*(w%4) ..; warps w and w+4 split the columns.  Lanes 0-63 hold X = W S0^T
// (rows of U), lanes 64-127 hold Y = Q S0^T and the output term; the state update
// uses all 128 lanes (rows k).  The three roles run separate loops with the same
// two block-wide barriers per chunk.
template <int Vt, bool kPacked>
__global__ void __launch_bounds__(320, 1)
scan_fwd_tc(Dims d, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_W, const __grid_constant__ CUtensorMap tm_M,
            const __grid_constant__ CUtensorMap tm_Ut, const __grid_constant__ CUtensorMap tm_o,
            const __grid_constant__ CUtensorMap tm_st, const float* __restrict__ G, const float* s0,
            float* sT, int write_o, int write_states, const int* __restrict__ chunk_off, int nseq, int tmode,
            float* trans, const int* __restrict__ order, bf16* __restrict__ o_rows, int* err) {
    using P = ScanPlan<Vt>;
    constexpr int HV = Vt / 2;  // columns per thread
    constexpr int NS = P::NS;
    extern __shared__ unsigned char smraw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    uint64_t* tbar = (uint64_t*)(sm + P::BAR);
    uint64_t* barXY = tbar + NS;
    uint64_t* barS = tbar + NS + 1;
    uint64_t* barO = tbar + NS + 2;
    uint32_t* tslot = (uint32_t*)(sm + P::BAR + 48);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool mma_warp = warp == 8, tma_warp = warp == 9, epi = warp < 8;
    const bool mma_issuer = tid == 256, tma_issuer = tid == 288;
    const int sub = warp & 3, half = (warp >> 2) & 1;
    const int lanerow = 32 * sub + lane;  // TMEM lane of this thread (epilogue warps)
    const int cb = half * HV;             // first column of this thread
    const int v0 = blockIdx.x * Vt, h = blockIdx.y;
    // Stream (b = blockIdx.z, h) runs chunks 0 .. d.NC-1 of its row of chunks.  With
    // packed sequences (chunk_off) the data is one row of chunks per head (B = 1):
    // sequence s = blockIdx.z runs chunks chunk_off[s] .. chunk_off[s+1]-1 of it
    // and keeps its state in slot s*H + h.  c below counts this CTA's chunks.
    // A transition CTA (tmode) starts from S0 = I, reads U~ as 0 and writes its
    // final state, the product of its chunks' maps, to `trans`.  `order` (or NULL)
    // maps grid row z to the sequence it runs.
    int b = blockIdx.z, c0 = 0, NC = d.NC;
    bool tr = tmode == 2;
    if (tmode == 1 && b >= nseq) {
        tr = true;
        b -= nseq;
    }
    if (order) b = order[b];
    const int64_t sidx = (int64_t)b * d.H + h;  // state slot
    if (chunk_off) {
        c0 = chunk_off[b];
        NC = chunk_off[b + 1] - c0;
        b = 0;
    }
    const int64_t cbase = ((int64_t)b * d.H + h) * d.NC + c0;  // global index of chunk c = 0
    const float ut_w = tr ? 0.f : 1.f;
    float* const s_out = tr ? trans : sT;
    // a slice wholly past the caller's V (V = 64) has no output columns
    const bool wr_o = write_o && !tr && v0 < d.V, wr_states = write_states && !tr;

    // Chunk c's tiles into stage c % NS (the n-th use of a stage completes phase n & 1).
    auto issue_loads = [&](int c) {
        unsigned char* st = sm + (c % NS) * P::STAGE;
        const int row = (int)((cbase + c) * kC);
        const int t0 = chunk_tok<kPacked>(d, c0 + c);
        uint64_t* bar = &tbar[c % NS];
        mbar_arrive_expect_tx(bar, 7 * 8192 + kC * Vt * 2);
        for (int j = 0; j < 2; ++j) {
            tma_load_2d(st + P::OFF_WQ + j * 16384, &tm_W, bar, 64 * j, row);
            tma_load_4d(st + P::OFF_WQ + j * 16384 + 8192, &tm_q, bar, 64 * j, h, t0, b);
            tma_load_4d(st + P::OFF_K + j * 8192, &tm_k, bar, 64 * j, h, t0, b);
        }
        tma_load_2d(st + P::OFF_M, &tm_M, bar, 0, row);
        tma_load_3d(st + P::OFF_UT, &tm_Ut, bar, 0, row, v0 / 8);
    };

    int issued = 0;  // chunks whose loads were issued (TMA issuer)
    if (tma_issuer) {
        for (int i = 0; i < NS + 3; ++i) mbar_init(&tbar[i], 1);
        fence_mbar_init();
        for (; issued < NS - 1 && issued < NC; ++issued) issue_loads(issued);
    }
    if (warp == 0) {
        tmem_alloc(tslot, P::TMEM_COLS);
        tmem_relinquish();
    }
    // State: thread holds S[v0 + cb + j][k = lanerow], j < HV.
    const int k = lanerow;
    float s[HV];
#pragma unroll
    for (int j = 0; j < HV; ++j) {
        const int v = v0 + cb + j;  // a 48-wide slice runs past V = 128 (zero columns)
        // the caller's state is [V, K] (K, V <= 128); rows and columns past them are zero
        const bool vok = (kD % Vt == 0) || v < kD;
        const bool uok = v < d.V && k < d.K;
        s[j] = (!epi || !vok) ? 0.f
                              : (tr ? (v == k ? 1.f : 0.f) : ((s0 && uok) ? s0[(sidx * d.V + v) * d.K + k] : 0.f));
    }
    auto write_state_operand = [&]() {
        // MN-major, no swizzle: element (v, k) at (v/8)*2048 + k*16 + (v%8)*2
#pragma unroll
        for (int g = 0; g < HV / 8; ++g)
            *(uint4*)(sm + P::S_OP + (cb / 8 + g) * 2048 + k * 16) =
                make_uint4(pack_bf16(s[8 * g + 0], s[8 * g + 1]), pack_bf16(s[8 * g + 2], s[8 * g + 3]),
                           pack_bf16(s[8 * g + 4], s[8 * g + 5]), pack_bf16(s[8 * g + 6], s[8 * g + 7]));
    };
    if (epi) write_state_operand();
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

    float GC_n = (NC > 0 && epi) ? G[cbase * kC + kC - 1] : 0.f;
    float Gr_n = (NC > 0 && epi) ? G[cbase * kC + r] : 0.f;
    float gr_prev = 0.f;

    // Output of chunk cc (threads on lanes 64-127): O = gamma Y + Mqk U.
    auto output_epilogue = [&](int cc, bool& okk) {
        okk = mbar_wait(barO, cc & 1, err, 64, d.wait_ns) && okk;
        __syncwarp();
        fence_after_sync();
        float y[HV], ov[HV];
        if constexpr (HV == 8) {
            // two 8-column halves through the x16 loader would over-read; use the
            // x16 load on a 16-column window and keep our half
            uint32_t wa[16], wb[16];
            tmem_ld16(tXY0 + (uint32_t)((cc & 1) * Vt) + lanebase, wa);
            tmem_ld16(tO + lanebase, wb);
            tmem_wait_ld(wa);
            tmem_wait_ld(wb);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                y[j] = __uint_as_float(half ? wa[8 + j] : wa[j]);
                ov[j] = __uint_as_float(half ? wb[8 + j] : wb[j]);
            }
        } else {
            tmem_cols2<HV>(tXY0 + (uint32_t)((cc & 1) * Vt) + lanebase + cb, tO + lanebase + cb, y, ov);
        }
#pragma unroll
        for (int g = 0; g < HV / 8; ++g) {
            float f[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = gr_prev * y[8 * g + j] + ov[8 * g + j];
            *(uint4*)(sm + P::O_OP + (cc & 1) * (kC * Vt * 2) + (cb / 8 + g) * 1024 + r * 16) =
                make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]),
                           pack_bf16(f[6], f[7]));
        }
    };

    // Output tile of chunk cc to o: one TMA store, except the last chunk of a packed
    // sequence with fewer than 64 tokens, whose valid rows the TMA warp copies (the
    // rows after them belong to the next sequence).  Called by the whole TMA warp.
    auto store_o = [&](int cc) {
        const unsigned char* tile = sm + P::O_OP + (cc & 1) * (kC * Vt * 2);
        const int t0 = chunk_tok<kPacked>(d, c0 + cc);
        if (!kPacked || chunk_valid<true>(d, c0 + cc) == kC) {
            if (tma_issuer) {
                tma_store_5d(&tm_o, tile, 0, t0, v0 / 8, h, b);
                bulk_commit();
            }
            return;
        }
        if constexpr (kPacked) {
            // core-matrix tile: 8 columns of row r at (group) * 1024 + r * 16
            const int nv = chunk_valid<true>(d, c0 + cc);
            for (int i = lane; i < nv * (Vt / 8); i += 32) {
                const int r = i / (Vt / 8), g = i % (Vt / 8);
                if (v0 + 8 * g < d.V)
                    *(uint4*)(o_rows + ((int64_t)(t0 + r) * d.H + h) * d.V + v0 + 8 * g) =
                        *(const uint4*)(tile + g * 1024 + r * 16);
            }
        }
    };

    bool ok = true;
    int c = 0;
    int xy_last = -1, o_last = -1;  // last chunk whose [X;Y] / output MMAs were committed (MMA issuer)
    if (mma_warp) {
#pragma unroll 1
        for (; c < NC; ++c) {
            const int stg = c % NS;
            unsigned char* st = sm + stg * P::STAGE;
            if (mma_issuer) {
                ok = mbar_wait(&tbar[stg], (c / NS) & 1, err, 8, d.wait_ns) && ok;
                if (ok) {
                    // [X; Y] = [W; Q] S0^T in one M=128 MMA chain
                    const uint64_t dWQ = sdesc(smem_u32(st + P::OFF_WQ), 16, 1024, SW_128B);
#pragma unroll
                    for (int s2 = 0; s2 < 8; ++s2)
                        mma_bf16_ss(tXY0 + (uint32_t)((c & 1) * Vt),
                                    desc_add(dWQ, (s2 >> 2) * 16384 + (s2 & 3) * 32), desc_add(dS, s2 * 256), id,
                                    s2 > 0);
                    mma_commit(barXY);
                    xy_last = c;
                }
            }
            __syncwarp();
            fence_before_sync();
            ok = __syncthreads_and(ok);  // 1: U and Uh written, X / Y read
            if (!ok) break;
            fence_after_sync();
            if (mma_issuer) {
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
                o_last = c;
            }
            __syncwarp();
            fence_before_sync();
            ok = __syncthreads_and(ok);  // 2: the state operand S1^T written
            if (!ok) break;
            fence_after_sync();
        }
    } else if (tma_warp) {
#pragma unroll 1
        for (; c < NC; ++c) {
            if (tma_issuer) {
                if (wr_states) {  // chunk-start state -> saved boundary states
                    tma_store_3d(&tm_st, sm + P::S_OP, 0, (int)((cbase + c) * kD), v0 / 8);
                    bulk_commit();
                }
                // chunk c + NS - 1 into the stage chunk c - 1 used, once its last
                // MMAs (the output term) have read it
                if (ok && issued < NC) {
                    if (c > 0) ok = mbar_wait(barO, (c - 1) & 1, err, 64, d.wait_ns) && ok;
                    if (ok) issue_loads(issued++);
                }
                bulk_wait_read0();  // the states store has read S0^T (rewritten after barrier 1)
            }
            __syncwarp();
            fence_before_sync();
            ok = __syncthreads_and(ok);  // 1
            if (!ok) break;
            fence_after_sync();
            if (tma_issuer) {
                // U of this chunk, in place over its U~ slice (read by this CTA only,
                // and already consumed), for the backward's chunk gradients
                if (wr_states) {
                    tma_store_3d(&tm_Ut, sm + P::U_OP, 0, (int)((cbase + c) * kC), v0 / 8);
                    bulk_commit();
                }
            }
            if (c > 0 && wr_o) store_o(c - 1);  // output tile of the previous chunk
            if (tma_issuer) {
                if (c > 0 && wr_o && (!kPacked || chunk_valid<true>(d, c0 + c - 1) == kC)) {
                    // the store issued a chunk earlier has read its tile, which the
                    // next output epilogue rewrites; so has the U store (older group)
                    bulk_wait_read1();
                } else {
                    // no output store this chunk (or rows copied by the warp): every
                    // store so far has read its tile (the U tile is rewritten next)
                    bulk_wait_read0();
                }
            }
            __syncwarp();
            fence_before_sync();
            ok = __syncthreads_and(ok);  // 2
            if (!ok) break;
            fence_after_sync();
        }
    } else {
#pragma unroll 1
        for (; c < NC; ++c) {
            const int stg = c % NS;
            unsigned char* st = sm + stg * P::STAGE;
            const int64_t chunk = cbase + c;
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
                ok = mbar_wait(&tbar[stg], (c / NS) & 1, err, 8, d.wait_ns) && ok;  // Ut slice is read below
                ok = mbar_wait(barXY, c & 1, err, 16, d.wait_ns) && ok;
                __syncwarp();
                fence_after_sync();
                // U = Ut - X, Uh = e_r U  (row r, columns cb .. cb+HV)
                float xg[HV];
                if constexpr (HV == 8) {
                    uint32_t w16[16];
                    tmem_ld16(tXY0 + (uint32_t)((c & 1) * Vt) + lanebase, w16);
                    tmem_wait_ld(w16);
#pragma unroll
                    for (int j = 0; j < 8; ++j) xg[j] = __uint_as_float(half ? w16[8 + j] : w16[j]);
                } else {
                    tmem_cols<HV>(tXY0 + (uint32_t)((c & 1) * Vt) + lanebase + cb, xg);
                }
#pragma unroll
                for (int g = 0; g < HV / 8; ++g) {
                    const int gg = cb / 8 + g;
                    const uint4 uq = *(const uint4*)(st + P::OFF_UT + gg * 1024 + r * 16);
                    const uint32_t uw4[4] = {uq.x, uq.y, uq.z, uq.w};
                    float u[8], uh[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {  // ut_w = 1 gives exactly Ut - X
                        u[2 * e] = fmaf(ut_w, bf_lo(uw4[e]), -xg[8 * g + 2 * e]);
                        u[2 * e + 1] = fmaf(ut_w, bf_hi(uw4[e]), -xg[8 * g + 2 * e + 1]);
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) uh[j] = er * u[j];
                    // MN-major, no swizzle: element (v, r) at (v/8)*1024 + r*16 + (v%8)*2
                    *(uint4*)(sm + P::U_OP + gg * 1024 + r * 16) = make_uint4(
                        pack_bf16(u[0], u[1]), pack_bf16(u[2], u[3]), pack_bf16(u[4], u[5]), pack_bf16(u[6], u[7]));
                    *(uint4*)(sm + P::UH_OP + gg * 1024 + r * 16) =
                        make_uint4(pack_bf16(uh[0], uh[1]), pack_bf16(uh[2], uh[3]), pack_bf16(uh[4], uh[5]),
                                   pack_bf16(uh[6], uh[7]));
                }
            }
            fence_proxy_async();
            fence_before_sync();
            ok = __syncthreads_and(ok);  // 1
            if (!ok) break;
            fence_after_sync();
            ok = mbar_wait(barS, c & 1, err, 32, d.wait_ns) && ok;
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
            ok = __syncthreads_and(ok);  // 2
            if (!ok) break;
            fence_after_sync();
        }
    }
    // `ok` is the value of the last block-wide vote here, the same in every thread
    if (ok && NC > 0) {
        if (epi && !urow) output_epilogue(NC - 1, ok);
        fence_proxy_async();
        fence_before_sync();
        ok = __syncthreads_and(ok);
        if (tma_warp && ok && wr_o) store_o(NC - 1);
    }
    if (ok && s_out && epi) {
#pragma unroll
        for (int j = 0; j < HV; ++j)
            if (v0 + cb + j < d.V && k < d.K) s_out[(sidx * d.V + v0 + cb + j) * d.K + k] = s[j];
    }
    if (tma_issuer) {
        // on an error, the loads still in flight (bounded waits) before leaving
        if (!ok)
            for (int cc = c; cc < issued; ++cc) mbar_wait(&tbar[cc % NS], (cc / NS) & 1, nullptr, 0);
        bulk_wait_read0();  // stores have read their tiles; their writes complete on their own
    }
    if (mma_issuer && !ok) {  // the MMAs still in flight, before the TMEM is freed
        if (xy_last >= 0) mbar_wait(barXY, xy_last & 1, nullptr, 0);
        if (o_last >= 0) mbar_wait(barO, o_last & 1, nullptr, 0);
    }
    __syncwarp();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, P::TMEM_COLS);
}

template <int Vt>
cudaError_t launch_scan_vt(const Dims& d, const void* q, const void* k, const TcBufs& tb, const float* s0,
                           void* o, float* sT, bf16* states, cudaStream_t st, const SeqMap* sq) {
    using P = ScanPlan<Vt>;
    CUtensorMap mq, mk, mW, mM, mUt, mo, mst;
    const int64_t rows = d.NS() * d.NC * kC;
    if (!tmap_bthd(&mq, q, d.B, d.T, d.H, d.K) || !tmap_bthd(&mk, k, d.B, d.T, d.H, d.K) ||
        !tmap_rows(&mW, tb.W, rows, kD) || !tmap_rows(&mM, tb.Mqk, rows, kC) ||
        !tmap_core8_rows(&mUt, tb.Ut, rows, kD, kC, Vt / 8))
        return cudaErrorInvalidValue;
    memset(&mo, 0, sizeof(mo));
    memset(&mst, 0, sizeof(mst));
    if (o && !tmap_core8_bthd(&mo, o, d.B, d.T, d.H, d.V, Vt / 8)) return cudaErrorInvalidValue;
    if (states && !tmap_core8_rows(&mst, states, d.NS() * d.NC * kD, kD, kD, Vt / 8))
        return cudaErrorInvalidValue;
    auto kern = d.tok ? scan_fwd_tc<Vt, true> : scan_fwd_tc<Vt, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P::SMEM);
    if (e != cudaSuccess) return e;
    const int mode = sq ? sq->mode : 0;
    const int nseq = sq ? sq->nseq : d.B;
    dim3 grid((kD + Vt - 1) / Vt, d.H, mode == 1 ? 2 * nseq : nseq);
    const bool tr_only = mode == 2;
    kern<<<grid, 320, P::SMEM, st>>>(d, mq, mk, mW, mM, mUt, mo, mst, tb.G, s0, sT, (o != nullptr && !tr_only),
                                     (states != nullptr && !tr_only), sq ? sq->chunk_off : nullptr, nseq, mode,
                                     sq ? sq->trans : nullptr, (sq && mode == 0) ? sq->order : nullptr,
                                     (bf16*)o, tb.err);
    return cudaGetLastError();
}

}  // namespace

// bf16 with 64-token chunks and K, V of 16, 32, 64 or 128: the kernels work on 128
// columns and TMA fills the columns past a narrower K or V with zeros on every load
// (they contribute nothing to any product) and clips them on every store.
bool tc_fwd_supported(const Dims& d, InType ty) {
    auto w = [](int x) { return x == 16 || x == 32 || x == 64 || x == kD; };
    return ty == InType::BF16 && d.C == kC && w(d.K) && w(d.V);
}

// The narrowest V-slice whose CTAs (one per slice and stream) fit one wave.
int tc_scan_vt(int64_t streams) {
    const int64_t sms = sm_count();
    for (int vt : {16, 32, 48, 64})
        if (streams * ((kD + vt - 1) / vt) <= sms) return vt;
    return 64;
}

// Packed sequences of unequal length: the CTAs do not finish together, so the
// waves interleave and the scan takes about max(longest chain, chunk-slices per
// SM) chunks, each at a cost that grows with the slice width (measured on GB300
// at about 2.1K, 2.4K, 2.75K and 3.2K cycles per chunk for 16, 32, 48 and 64
// columns); the longest sequences start first (SeqMap::order).
int tc_scan_vt_for(const Dims& d, const SeqMap* sq, int64_t streams) {
    if (!sq || sq->mode != 0 || sq->max_nc <= 0) return tc_scan_vt(streams);
    const double sms = (double)sm_count();
    const int vts[4] = {16, 32, 48, 64};
    const double cost[4] = {2.1, 2.4, 2.75, 3.2};
    int best = 64;
    double best_t = 0.0;
    for (int i = 0; i < 4; ++i) {
        const int slices = (kD + vts[i] - 1) / vts[i];
        const double work = (double)d.NC * d.H * slices / sms;  // flat chunk rows bound the total
        const double t = cost[i] * (work > sq->max_nc ? work : (double)sq->max_nc);
        if (i == 0 || t < best_t) {
            best = vts[i];
            best_t = t;
        }
    }
    return best;
}

cudaError_t launch_prep_tc(const Dims& d, const void* q, const void* k, const void* v, const void* alpha,
                           const void* beta, const TcBufs& tb, cudaStream_t st, const RawPrologue* rp) {
    CUtensorMap mq, mk, mv, mW, mU, mM;
    const int64_t rows = d.NS() * d.NC * kC;
    if (!tmap_bthd(&mq, q, d.B, d.T, d.H, d.K) || !tmap_bthd(&mk, k, d.B, d.T, d.H, d.K) ||
        !tmap_bthd(&mv, v, d.B, d.T, d.H, d.V) || !tmap_rows(&mW, tb.W, rows, kD) ||
        !tmap_rows(&mU, tb.Ut, rows, kD) || !tmap_rows(&mM, tb.Mqk, rows, kC))
        return cudaErrorInvalidValue;
    RawPrologue raw{};
    if (rp && rp->on) raw = *rp;
    auto kern = d.tok ? prep_fwd_tc<false, true> : (raw.on ? prep_fwd_tc<true, false> : prep_fwd_tc<false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrepSmem);
    if (e != cudaSuccess) return e;
    const int64_t nchunks = d.NS() * d.NC;
    dim3 grid((unsigned)std::min<int64_t>(nchunks, 2 * sm_count()));
    kern<<<grid, 256, kPrepSmem, st>>>(d, mq, mk, mv, mW, mU, mM, (const bf16*)alpha, (const bf16*)beta,
                                              tb.G, tb.T, raw, tb.err);
    return cudaGetLastError();
}

cudaError_t launch_scan_fwd_tc(const Dims& d, const void* q, const void* k, const TcBufs& tb, const float* s0,
                               void* o, float* sT, __nv_bfloat16* states, cudaStream_t st, const SeqMap* sq) {
    const int64_t streams = sq ? (int64_t)sq->nseq * d.H * (sq->mode == 1 ? 2 : 1) : d.NS();
    switch (tc_scan_vt_for(d, sq, streams)) {
        case 16: return launch_scan_vt<16>(d, q, k, tb, s0, o, sT, states, st, sq);
        case 32: return launch_scan_vt<32>(d, q, k, tb, s0, o, sT, states, st, sq);
        case 48: return launch_scan_vt<48>(d, q, k, tb, s0, o, sT, states, st, sq);
        default: return launch_scan_vt<64>(d, q, k, tb, s0, o, sT, states, st, sq);
    }
}

}  // namespace gdn
