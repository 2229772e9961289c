// simt.cu -- CUDA-core (float32) kernels of the chunkwise gated delta rule.
//
// These kernels compute every step of the path in float32 with plain FMAs: the
// float32 input path (whose tolerance rules out single-pass TF32/bf16 tensor-core
// products) and the reference schedule the tensor-core kernels are checked
// against.  Templated on the input type (float or bf16); state, gates, solve and
// accumulation are float32 either way.
//
// Chunk algebra (per (b,h) stream, chunk of C tokens, start state S0 [V,K]):
//   G_r = sum_{i<=r} log alpha_i,  gamma_r = exp(G_r),  Gam_ri = exp(G_r - G_i), r>=i
//   A   = strict_lower(diag(beta)(Gam .* K K^T)),  T = (I + A)^-1
//   Ut  = T diag(beta) V,  W = T diag(beta gamma) K,  Mqk = lower(Gam .* Q K^T)
//   U   = Ut - W S0^T,  O = diag(gamma) Q S0^T + Mqk U
//   S1  = gamma_C S0 + U^T diag(exp(G_C - G)) K
// ("Sparse Delta Memory: layer and kernels", "What the layer computes": Phase 1
// builds the decay-weighted Gram matrices, the Solve inverts (I + tril(beta A,-1)),
// Phase 2 walks the chunks in order; the backward walks them in reverse.)
// Only differences G_r - G_i with r >= i are exponentiated, so nothing overflows
// for 0 < alpha <= 1.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float* p, float x) { *p = x; }
__device__ __forceinline__ void stf(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ int64_t row_qk(const Dims& d, int b, int t, int h) {
    return (((int64_t)b * d.T + t) * d.H + h) * d.K;
}
__device__ __forceinline__ int64_t row_v(const Dims& d, int b, int t, int h) {
    return (((int64_t)b * d.T + t) * d.H + h) * d.V;
}
__device__ __forceinline__ int64_t gate(const Dims& d, int b, int t, int h) {
    return ((int64_t)b * d.T + t) * d.H + h;
}

// In-place inclusive prefix sum of x[0..n) by one full warp (n <= 32 * 8).
__device__ void warp_cumsum(float* x, int n) {
    const int lane = threadIdx.x & 31;
    const int per = (n + 31) / 32;
    const int lo = lane * per;
    const int hi = min(lo + per, n);
    float run = 0.f;
    for (int i = lo; i < hi; ++i) {
        run += x[i];
        x[i] = run;
    }
    float incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    const float excl = incl - run;
    for (int i = lo; i < hi; ++i) x[i] += excl;
}

// T = (I + A)^-1 for a strictly lower triangular A (C x C, row stride CP, C a
// multiple of 16): 16x16 diagonal blocks by column-wise forward substitution, then
// block rows in order, T_IJ = -T_II * sum_{J<=L<I} A_IL T_LJ.  X holds
// (C/16 - 1) * 256 floats.  Contains __syncthreads(); call from the whole block.
__device__ void tril_inverse(const float* A, float* Tm, float* X, int C, int CP) {
    const int tid = threadIdx.x, nt = blockDim.x;
    for (int idx = tid; idx < C * C; idx += nt) {
        const int r = idx / C, i = idx - r * C;
        Tm[r * CP + i] = 0.f;
    }
    __syncthreads();
    const int nb = C / 16;
    for (int w = tid; w < nb * 16; w += nt) {
        const int base = (w >> 4) * 16, j = w & 15;
        Tm[(base + j) * CP + base + j] = 1.f;
        for (int r = j + 1; r < 16; ++r) {
            float acc = 0.f;
            for (int i = j; i < r; ++i) acc += A[(base + r) * CP + base + i] * Tm[(base + i) * CP + base + j];
            Tm[(base + r) * CP + base + j] = -acc;
        }
    }
    __syncthreads();
    for (int I = 1; I < nb; ++I) {
        const int n = I * 256;
        for (int idx = tid; idx < n; idx += nt) {
            const int J = idx >> 8, r = (idx >> 4) & 15, cc = idx & 15;
            float acc = 0.f;
            for (int L = J; L < I; ++L)
                for (int m = 0; m < 16; ++m)
                    acc += A[(I * 16 + r) * CP + L * 16 + m] * Tm[(L * 16 + m) * CP + J * 16 + cc];
            X[idx] = acc;
        }
        __syncthreads();
        for (int idx = tid; idx < n; idx += nt) {
            const int J = idx >> 8, r = (idx >> 4) & 15, cc = idx & 15;
            float acc = 0.f;
            for (int m = 0; m <= r; ++m)
                acc += Tm[(I * 16 + r) * CP + I * 16 + m] * X[(J << 8) + (m << 4) + cc];
            Tm[(I * 16 + r) * CP + J * 16 + cc] = -acc;
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Chunk-parallel step: one CTA per (chunk, head, batch).
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
prep_kernel(Dims d, const Tin* __restrict__ k, const Tin* __restrict__ q,
            const Tin* __restrict__ v, const Tin* __restrict__ alpha,
            const Tin* __restrict__ beta, ChunkBufs cb, int write_T) {
    extern __shared__ float sm[];
    const int C = d.C, K = d.K, V = d.V, KP = K + 1, CP = C + 1;
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, nt = blockDim.x;
    float* Ks = sm;
    float* Qs = Ks + C * KP;
    float* Vs = Qs + C * KP;
    float* As = Vs + C * V;
    float* Ts = As + C * CP;
    float* Xs = Ts + C * CP;
    float* Gs = Xs + C * 16;
    float* bs = Gs + C;
    float* gs = bs + C;
    const int t0 = c * C;
    const int64_t chunk = ((int64_t)b * d.H + h) * d.NC + c;

    for (int idx = tid; idx < C * K; idx += nt) {
        const int r = idx / K, j = idx - r * K, t = t0 + r;
        float kv = 0.f, qv = 0.f;
        if (t < d.T) {
            const int64_t o = row_qk(d, b, t, h) + j;
            kv = ldf(k + o);
            qv = ldf(q + o);
        }
        Ks[r * KP + j] = kv;
        Qs[r * KP + j] = qv;
    }
    for (int idx = tid; idx < C * V; idx += nt) {
        const int r = idx / V, j = idx - r * V, t = t0 + r;
        Vs[r * V + j] = (t < d.T) ? ldf(v + row_v(d, b, t, h) + j) : 0.f;
    }
    if (tid < C) {
        const int t = t0 + tid;
        float a = 1.f, be = 0.f;  // padding: alpha = 1, beta = 0 keeps the state
        if (t < d.T) {
            a = ldf(alpha + gate(d, b, t, h));
            be = ldf(beta + gate(d, b, t, h));
        }
        Gs[tid] = logf(a);
        bs[tid] = be;
    }
    __syncthreads();
    if (tid < 32) warp_cumsum(Gs, C);
    __syncthreads();
    if (tid < C) gs[tid] = expf(Gs[tid]);

    float* Mg = cb.Mqk + chunk * C * C;
    for (int idx = tid; idx < C * C; idx += nt) {
        const int r = idx / C, i = idx - r * C;
        float a_ = 0.f, m_ = 0.f;
        if (i <= r) {
            float dkk = 0.f, dqk = 0.f;
            for (int j = 0; j < K; ++j) {
                const float ki = Ks[i * KP + j];
                dkk += Ks[r * KP + j] * ki;
                dqk += Qs[r * KP + j] * ki;
            }
            const float gam = expf(Gs[r] - Gs[i]);
            if (i < r) a_ = bs[r] * gam * dkk;
            m_ = gam * dqk;
        }
        As[r * CP + i] = a_;
        Mg[r * C + i] = m_;
    }
    __syncthreads();
    tril_inverse(As, Ts, Xs, C, CP);

    float* Utg = cb.Ut + chunk * C * V;
    for (int idx = tid; idx < C * V; idx += nt) {
        const int r = idx / V, j = idx - r * V;
        float acc = 0.f;
        for (int i = 0; i <= r; ++i) acc += Ts[r * CP + i] * bs[i] * Vs[i * V + j];
        Utg[r * V + j] = acc;
    }
    float* Wg = cb.W + chunk * C * K;
    for (int idx = tid; idx < C * K; idx += nt) {
        const int r = idx / K, j = idx - r * K;
        float acc = 0.f;
        for (int i = 0; i <= r; ++i) acc += Ts[r * CP + i] * (bs[i] * gs[i]) * Ks[i * KP + j];
        Wg[r * K + j] = acc;
    }
    if (write_T) {
        float* Tg = cb.Tm + chunk * C * C;
        for (int idx = tid; idx < C * C; idx += nt) {
            const int r = idx / C, i = idx - r * C;
            Tg[r * C + i] = Ts[r * CP + i];
        }
    }
    if (tid < C) cb.G[chunk * C + tid] = Gs[tid];
}

// ---------------------------------------------------------------------------
// Sequential forward scan: one CTA per (V-slice of Vt rows, head, batch) walks the
// chunks in order with its slice of the state in shared memory.
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
scan_fwd_kernel(Dims d, int Vt, const Tin* __restrict__ q, const Tin* __restrict__ k,
                ChunkBufs cb, const float* s0, Tin* __restrict__ o, float* sT,
                float* __restrict__ states, int write_o) {
    extern __shared__ float sm[];
    const int C = d.C, K = d.K, V = d.V, KP = K + 1, CP = C + 1, VtP = Vt + 1;
    const int v0 = blockIdx.x * Vt, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, nt = blockDim.x;
    float* S = sm;
    float* Ws = S + Vt * KP;
    float* Qs = Ws + C * KP;
    float* Ks = Qs + C * KP;
    float* Ms = Ks + C * KP;
    float* Us = Ms + C * CP;
    float* Ys = Us + C * VtP;
    float* Gs = Ys + C * VtP;
    float* gs = Gs + C;
    float* es = gs + C;
    const int64_t s = (int64_t)b * d.H + h;

    for (int idx = tid; idx < Vt * K; idx += nt) {
        const int vv = idx / K, j = idx - vv * K;
        S[vv * KP + j] = s0 ? s0[(s * V + v0 + vv) * K + j] : 0.f;
    }
    for (int c = 0; c < d.NC; ++c) {
        __syncthreads();
        const int64_t chunk = s * d.NC + c;
        const int t0 = c * C;
        const float* Wg = cb.W + chunk * C * K;
        const float* Utg = cb.Ut + chunk * C * V;
        for (int idx = tid; idx < C * K; idx += nt) {
            const int r = idx / K, j = idx - r * K, t = t0 + r;
            Ws[r * KP + j] = Wg[idx];
            float kv = 0.f, qv = 0.f;
            if (t < d.T) {
                const int64_t off = row_qk(d, b, t, h) + j;
                kv = ldf(k + off);
                if (write_o) qv = ldf(q + off);
            }
            Ks[r * KP + j] = kv;
            Qs[r * KP + j] = qv;
        }
        if (write_o) {
            const float* Mg = cb.Mqk + chunk * C * C;
            for (int idx = tid; idx < C * C; idx += nt) {
                const int r = idx / C, i = idx - r * C;
                Ms[r * CP + i] = Mg[idx];
            }
        }
        for (int idx = tid; idx < C * Vt; idx += nt) {
            const int r = idx / Vt, vv = idx - r * Vt;
            Us[r * VtP + vv] = Utg[r * V + v0 + vv];
        }
        if (tid < C) Gs[tid] = cb.G[chunk * C + tid];
        if (states) {
            float* St = states + chunk * V * K;
            for (int idx = tid; idx < Vt * K; idx += nt) {
                const int vv = idx / K, j = idx - vv * K;
                St[(int64_t)(v0 + vv) * K + j] = S[vv * KP + j];
            }
        }
        __syncthreads();
        if (tid < C) {
            gs[tid] = expf(Gs[tid]);
            es[tid] = expf(Gs[C - 1] - Gs[tid]);
        }
        // U = Ut - W S0^T ; Y = Q S0^T
        for (int idx = tid; idx < C * Vt; idx += nt) {
            const int r = idx / Vt, vv = idx - r * Vt;
            float x = 0.f, y = 0.f;
            for (int j = 0; j < K; ++j) {
                const float sv = S[vv * KP + j];
                x += Ws[r * KP + j] * sv;
                y += Qs[r * KP + j] * sv;
            }
            Us[r * VtP + vv] -= x;
            Ys[r * VtP + vv] = y;
        }
        __syncthreads();
        if (write_o) {
            for (int idx = tid; idx < C * Vt; idx += nt) {
                const int r = idx / Vt, vv = idx - r * Vt, t = t0 + r;
                if (t >= d.T) continue;
                float acc = gs[r] * Ys[r * VtP + vv];
                for (int i = 0; i <= r; ++i) acc += Ms[r * CP + i] * Us[i * VtP + vv];
                stf(o + row_v(d, b, t, h) + v0 + vv, acc);
            }
        }
        const float gC = gs[C - 1];
        for (int idx = tid; idx < Vt * K; idx += nt) {
            const int vv = idx / K, j = idx - vv * K;
            float acc = gC * S[vv * KP + j];
            for (int r = 0; r < C; ++r) acc += Us[r * VtP + vv] * (es[r] * Ks[r * KP + j]);
            S[vv * KP + j] = acc;
        }
    }
    __syncthreads();
    if (sT) {
        for (int idx = tid; idx < Vt * K; idx += nt) {
            const int vv = idx / K, j = idx - vv * K;
            sT[(s * V + v0 + vv) * K + j] = S[vv * KP + j];
        }
    }
}

// ---------------------------------------------------------------------------
// Reverse scan: one CTA per (V-slice, head, batch) walks the chunks backwards,
// carrying dS (the gradient of the current chunk's end state):
//   U  = Ut - W S0^T,   dU = Mqk^T dO + diag(exp(G_C - G)) K dS1^T
//   dS0 = gamma_C dS1 + dO^T diag(gamma) Q - dU^T W
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
scan_bwd_kernel(Dims d, int Vt, const Tin* __restrict__ q, const Tin* __restrict__ k,
                const Tin* __restrict__ d_o, ChunkBufs cb, const float* __restrict__ states,
                const float* dsT, BwdBufs bb, float* ds0) {
    extern __shared__ float sm[];
    const int C = d.C, K = d.K, V = d.V, KP = K + 1, CP = C + 1, VtP = Vt + 1;
    const int v0 = blockIdx.x * Vt, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, nt = blockDim.x;
    float* dS = sm;
    float* S0 = dS + Vt * KP;
    float* Ws = S0 + Vt * KP;
    float* Qs = Ws + C * KP;
    float* Ks = Qs + C * KP;
    float* Ms = Ks + C * KP;
    float* dOs = Ms + C * CP;
    float* Us = dOs + C * VtP;
    float* dUs = Us + C * VtP;
    float* Gs = dUs + C * VtP;
    float* gs = Gs + C;
    float* es = gs + C;
    const int64_t s = (int64_t)b * d.H + h;

    for (int idx = tid; idx < Vt * K; idx += nt) {
        const int vv = idx / K, j = idx - vv * K;
        dS[vv * KP + j] = dsT ? dsT[(s * V + v0 + vv) * K + j] : 0.f;
    }
    for (int c = d.NC - 1; c >= 0; --c) {
        __syncthreads();
        const int64_t chunk = s * d.NC + c;
        const int t0 = c * C;
        const float* Wg = cb.W + chunk * C * K;
        const float* Utg = cb.Ut + chunk * C * V;
        const float* Mg = cb.Mqk + chunk * C * C;
        const float* St = states + chunk * V * K;
        for (int idx = tid; idx < C * K; idx += nt) {
            const int r = idx / K, j = idx - r * K, t = t0 + r;
            Ws[r * KP + j] = Wg[idx];
            float kv = 0.f, qv = 0.f;
            if (t < d.T) {
                const int64_t off = row_qk(d, b, t, h) + j;
                kv = ldf(k + off);
                qv = ldf(q + off);
            }
            Ks[r * KP + j] = kv;
            Qs[r * KP + j] = qv;
        }
        for (int idx = tid; idx < C * C; idx += nt) {
            const int r = idx / C, i = idx - r * C;
            Ms[r * CP + i] = Mg[idx];
        }
        for (int idx = tid; idx < C * Vt; idx += nt) {
            const int r = idx / Vt, vv = idx - r * Vt, t = t0 + r;
            Us[r * VtP + vv] = Utg[r * V + v0 + vv];
            dOs[r * VtP + vv] = (t < d.T) ? ldf(d_o + row_v(d, b, t, h) + v0 + vv) : 0.f;
        }
        float* dSt = bb.dS1 + chunk * V * K;
        for (int idx = tid; idx < Vt * K; idx += nt) {
            const int vv = idx / K, j = idx - vv * K;
            S0[vv * KP + j] = St[(int64_t)(v0 + vv) * K + j];
            dSt[(int64_t)(v0 + vv) * K + j] = dS[vv * KP + j];
        }
        if (tid < C) Gs[tid] = cb.G[chunk * C + tid];
        __syncthreads();
        if (tid < C) {
            gs[tid] = expf(Gs[tid]);
            es[tid] = expf(Gs[C - 1] - Gs[tid]);
        }
        __syncthreads();
        float* Ug = bb.U + chunk * C * V;
        float* dUg = bb.dU + chunk * C * V;
        for (int idx = tid; idx < C * Vt; idx += nt) {
            const int r = idx / Vt, vv = idx - r * Vt;
            float x = 0.f, kd = 0.f;
            for (int j = 0; j < K; ++j) {
                x += Ws[r * KP + j] * S0[vv * KP + j];
                kd += Ks[r * KP + j] * dS[vv * KP + j];
            }
            float du = es[r] * kd;
            for (int s2 = r; s2 < C; ++s2) du += Ms[s2 * CP + r] * dOs[s2 * VtP + vv];
            const float u = Us[r * VtP + vv] - x;
            Us[r * VtP + vv] = u;
            dUs[r * VtP + vv] = du;
            Ug[r * V + v0 + vv] = u;
            dUg[r * V + v0 + vv] = du;
        }
        __syncthreads();
        const float gC = gs[C - 1];
        for (int idx = tid; idx < Vt * K; idx += nt) {
            const int vv = idx / K, j = idx - vv * K;
            float acc = gC * dS[vv * KP + j];
            for (int r = 0; r < C; ++r)
                acc += dOs[r * VtP + vv] * (gs[r] * Qs[r * KP + j]) - dUs[r * VtP + vv] * Ws[r * KP + j];
            dS[vv * KP + j] = acc;
        }
    }
    __syncthreads();
    if (ds0) {
        for (int idx = tid; idx < Vt * K; idx += nt) {
            const int vv = idx / K, j = idx - vv * K;
            ds0[(s * V + v0 + vv) * K + j] = dS[vv * KP + j];
        }
    }
}

// ---------------------------------------------------------------------------
// Chunk-local gradients: one CTA per (chunk, head, batch), full K and V.
// Given S0, dS1, U, dU of the chunk (from the reverse scan):
//   dMqk = lower(dO U^T), dQK = Gam .* dMqk
//   dQ   = diag(gamma) dO S0 + dQK K
//   dW   = -dU S0,  dT = dU (beta V)^T + dW (beta gamma K)^T  (strict lower part)
//   dV   = diag(beta) T^T dU,  dA = strict_lower(-T^T dT T^T)
//   E    = diag(beta)(Gam .* dA)
//   dK   = dQK^T Q + diag(exp(G_C-G)) U dS1 + diag(beta gamma) T^T dW + (E + E^T) K
//   dbeta, dG from every place beta, gamma, Gam and exp(G_C - G) enter;
//   dlog alpha = reverse within-chunk cumsum of dG,  dalpha = dlog alpha / alpha.
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
grad_kernel(Dims d, const Tin* __restrict__ q, const Tin* __restrict__ k,
            const Tin* __restrict__ v, const Tin* __restrict__ alpha,
            const Tin* __restrict__ beta, const Tin* __restrict__ d_o, ChunkBufs cb,
            const float* __restrict__ states, BwdBufs bb, Tin* __restrict__ dq,
            Tin* __restrict__ dk, Tin* __restrict__ dv, Tin* __restrict__ dalpha,
            Tin* __restrict__ dbeta) {
    extern __shared__ float sm[];
    const int C = d.C, K = d.K, V = d.V, KP = K + 1, CP = C + 1;
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, nt = blockDim.x;
    float* Qs = sm;
    float* Ks = Qs + C * KP;
    float* Ts = Ks + C * KP;
    float* Ms = Ts + C * CP;
    float* dQKs = Ms + C * CP;
    float* E1s = dQKs + C * CP;
    float* KKs = E1s + C * CP;
    float* M2s = KKs + C * CP;
    float* M4s = M2s + C * CP;
    float* Gs = M4s + C * CP;
    float* gs = Gs + C;
    float* es = gs + C;
    float* as_ = es + C;
    float* bs = as_ + C;
    float* dB12 = bs + C;
    float* dGw = dB12 + C;
    float* dB3 = dGw + C;
    float* rE2 = dB3 + C;
    float* cE2 = rE2 + C;
    float* rE1 = cE2 + C;
    float* cE1 = rE1 + C;
    float* eR = cE1 + C;
    float* dG1 = eR + C;
    float* red = dG1 + C;  // kThreads floats

    const int t0 = c * C;
    const int64_t chunk = ((int64_t)b * d.H + h) * d.NC + c;
    const float* S0 = states + chunk * V * K;
    const float* dS1 = bb.dS1 + chunk * V * K;
    const float* Ug = bb.U + chunk * C * V;
    const float* dUg = bb.dU + chunk * C * V;
    float* dWg = bb.dW + chunk * C * K;
    float* dQ1g = bb.dQ1 + chunk * C * K;
    float* dKhg = bb.dKh + chunk * C * K;

    for (int idx = tid; idx < C * K; idx += nt) {
        const int r = idx / K, j = idx - r * K, t = t0 + r;
        float kv = 0.f, qv = 0.f;
        if (t < d.T) {
            const int64_t off = row_qk(d, b, t, h) + j;
            kv = ldf(k + off);
            qv = ldf(q + off);
        }
        Ks[r * KP + j] = kv;
        Qs[r * KP + j] = qv;
    }
    {
        const float* Tg = cb.Tm + chunk * C * C;
        const float* Mg = cb.Mqk + chunk * C * C;
        for (int idx = tid; idx < C * C; idx += nt) {
            const int r = idx / C, i = idx - r * C;
            Ts[r * CP + i] = Tg[idx];
            Ms[r * CP + i] = Mg[idx];
        }
    }
    if (tid < C) {
        const int t = t0 + tid;
        Gs[tid] = cb.G[chunk * C + tid];
        float a = 1.f, be = 0.f;
        if (t < d.T) {
            a = ldf(alpha + gate(d, b, t, h));
            be = ldf(beta + gate(d, b, t, h));
        }
        as_[tid] = a;
        bs[tid] = be;
    }
    __syncthreads();
    if (tid < C) {
        gs[tid] = expf(Gs[tid]);
        es[tid] = expf(Gs[C - 1] - Gs[tid]);
    }
    __syncthreads();

    // P1: C x C products and the [C,K] / [C,V] terms that read S0, dS1, U, dU.
    for (int idx = tid; idx < C * C; idx += nt) {
        const int r = idx / C, i = idx - r * C, t = t0 + r;
        float dm = 0.f, kk = 0.f, p = 0.f, gam = 0.f;
        if (i <= r) {
            gam = expf(Gs[r] - Gs[i]);
            if (t < d.T) {
                const Tin* dor = d_o + row_v(d, b, t, h);
                for (int vv = 0; vv < V; ++vv) dm += ldf(dor + vv) * Ug[i * V + vv];
            }
            const int ti = t0 + i;
            if (ti < d.T) {
                const Tin* vr = v + row_v(d, b, ti, h);
                for (int vv = 0; vv < V; ++vv) p += dUg[r * V + vv] * ldf(vr + vv);
            }
            if (i < r)
                for (int j = 0; j < K; ++j) kk += Ks[r * KP + j] * Ks[i * KP + j];
        }
        dQKs[r * CP + i] = gam * dm;
        E1s[r * CP + i] = dm * Ms[r * CP + i];
        KKs[r * CP + i] = kk;
        M2s[r * CP + i] = p;  // P[s][r'] = sum_v dU[s][v] V[r'][v]
    }
    for (int idx = tid; idx < C * K; idx += nt) {
        const int r = idx / K, j = idx - r * K, t = t0 + r;
        float dw = 0.f, dq1 = 0.f, dkh = 0.f;
        const Tin* dor = (t < d.T) ? d_o + row_v(d, b, t, h) : nullptr;
        for (int vv = 0; vv < V; ++vv) {
            const float s0v = S0[(int64_t)vv * K + j];
            dw -= dUg[r * V + vv] * s0v;
            if (dor) dq1 += ldf(dor + vv) * s0v;
            dkh += Ug[r * V + vv] * dS1[(int64_t)vv * K + j];
        }
        dWg[idx] = dw;
        dQ1g[idx] = gs[r] * dq1;
        dKhg[idx] = dkh;
    }
    for (int idx = tid; idx < C * V; idx += nt) {
        const int r = idx / V, vv = idx - r * V, t = t0 + r;
        if (t >= d.T) continue;
        float acc = 0.f;
        for (int s2 = r; s2 < C; ++s2) acc += Ts[s2 * CP + r] * dUg[s2 * V + vv];
        stf(dv + row_v(d, b, t, h) + vv, bs[r] * acc);
    }
    __syncthreads();
    // P2: Qm = dW K^T (lower)
    for (int idx = tid; idx < C * C; idx += nt) {
        const int s2 = idx / C, r = idx - s2 * C;
        float qm = 0.f;
        if (r <= s2)
            for (int j = 0; j < K; ++j) qm += dWg[s2 * K + j] * Ks[r * KP + j];
        M4s[s2 * CP + r] = qm;
    }
    __syncthreads();
    if (tid < C) {
        const int r = tid;
        float b12 = 0.f, gw = 0.f, re = 0.f, ce = 0.f;
        for (int s2 = r; s2 < C; ++s2) {
            const float tsr = Ts[s2 * CP + r];
            b12 += tsr * (M2s[s2 * CP + r] + gs[r] * M4s[s2 * CP + r]);
            gw += tsr * M4s[s2 * CP + r];
        }
        for (int i = 0; i < C; ++i) {
            re += E1s[r * CP + i];
            ce += E1s[i * CP + r];
        }
        dB12[r] = b12;
        dGw[r] = bs[r] * gs[r] * gw;
        rE1[r] = re;
        cE1[r] = ce;
    }
    __syncthreads();
    // dT (strictly lower) in place of P
    for (int idx = tid; idx < C * C; idx += nt) {
        const int s2 = idx / C, r = idx - s2 * C;
        M2s[s2 * CP + r] = (r < s2) ? bs[r] * (M2s[s2 * CP + r] + gs[r] * M4s[s2 * CP + r]) : 0.f;
    }
    __syncthreads();
    // P3: Y = dT T^T
    for (int idx = tid; idx < C * C; idx += nt) {
        const int s2 = idx / C, bc = idx - s2 * C;
        float y = 0.f;
        const int rmax = min(s2 - 1, bc);
        for (int r = 0; r <= rmax; ++r) y += M2s[s2 * CP + r] * Ts[bc * CP + r];
        M4s[s2 * CP + bc] = y;
    }
    __syncthreads();
    // P4: dA = strict_lower(-T^T Y)
    for (int idx = tid; idx < C * C; idx += nt) {
        const int a = idx / C, bc = idx - a * C;
        float acc = 0.f;
        if (a > bc)
            for (int s2 = a; s2 < C; ++s2) acc += Ts[s2 * CP + a] * M4s[s2 * CP + bc];
        M2s[a * CP + bc] = -acc;
    }
    __syncthreads();
    if (tid < C) {
        const int a = tid;
        float b3 = 0.f, ce = 0.f;
        for (int bc = 0; bc < a; ++bc) b3 += expf(Gs[a] - Gs[bc]) * M2s[a * CP + bc] * KKs[a * CP + bc];
        for (int a2 = a + 1; a2 < C; ++a2)
            ce += bs[a2] * expf(Gs[a2] - Gs[a]) * M2s[a2 * CP + a] * KKs[a2 * CP + a];
        dB3[a] = b3;
        rE2[a] = bs[a] * b3;
        cE2[a] = ce;
    }
    __syncthreads();
    // E = diag(beta)(Gam .* dA) in place
    for (int idx = tid; idx < C * C; idx += nt) {
        const int a = idx / C, bc = idx - a * C;
        M2s[a * CP + bc] = (a > bc) ? bs[a] * expf(Gs[a] - Gs[bc]) * M2s[a * CP + bc] : 0.f;
    }
    __syncthreads();
    // P6: dQ, dK
    for (int idx = tid; idx < C * K; idx += nt) {
        const int r = idx / K, j = idx - r * K, t = t0 + r;
        if (t >= d.T) continue;
        float dkk = es[r] * dKhg[idx];
        float tw = 0.f;
        for (int s2 = r; s2 < C; ++s2) {
            dkk += dQKs[s2 * CP + r] * Qs[s2 * KP + j];
            tw += Ts[s2 * CP + r] * dWg[s2 * K + j];
        }
        dkk += bs[r] * gs[r] * tw;
        float dqq = dQ1g[idx];
        for (int i = 0; i < C; ++i) {
            const float ki = Ks[i * KP + j];
            dkk += (M2s[r * CP + i] + M2s[i * CP + r]) * ki;
            if (i <= r) dqq += dQKs[r * CP + i] * ki;
        }
        const int64_t off = row_qk(d, b, t, h) + j;
        stf(dq + off, dqq);
        stf(dk + off, dkk);
    }
    if (tid < C) {
        const int r = tid;
        float e = 0.f, g1 = 0.f;
        for (int j = 0; j < K; ++j) {
            e += dKhg[r * K + j] * Ks[r * KP + j];
            g1 += Qs[r * KP + j] * dQ1g[r * K + j];
        }
        eR[r] = es[r] * e;
        dG1[r] = g1;
    }
    {
        float part = 0.f;
        for (int idx = tid; idx < V * K; idx += nt) part += dS1[idx] * S0[idx];
        red[tid] = part;
    }
    __syncthreads();
    for (int w = nt / 2; w > 0; w >>= 1) {
        if (tid < w) red[tid] += red[tid + w];
        __syncthreads();
    }
    if (tid == 0) {
        float esum = 0.f;
        for (int r = 0; r < C; ++r) esum += eR[r];
        // dG per position, then the reverse within-chunk cumsum gives dlog alpha.
        float run = 0.f;
        for (int r = C - 1; r >= 0; --r) {
            float g = dG1[r] + dGw[r] + rE1[r] - cE1[r] + rE2[r] - cE2[r] - eR[r];
            if (r == C - 1) g += gs[C - 1] * red[0] + esum;
            run += g;
            const int t = t0 + r;
            if (t < d.T) {
                stf(dalpha + gate(d, b, t, h), run / as_[r]);
                stf(dbeta + gate(d, b, t, h), dB12[r] + dB3[r]);
            }
        }
    }
}

template <typename F>
cudaError_t set_smem(F* kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// The scans' V-slice: 32 columns (or V), halved down to 4 while the CTAs (one
// per slice and stream) would leave SMs idle; each slice's chunk loop reads the
// same per-chunk tiles, so narrower slices trade L2 reads for parallelism.
int pick_vt(const Dims& d) {
    int vt = d.V < 32 ? d.V : 32;
    const int64_t streams = (int64_t)d.B * d.H, sms = sm_count();
    while (vt > 4 && streams * (d.V / vt) < sms) vt /= 2;
    return vt;
}

}  // namespace

size_t prep_smem_bytes(const Dims& d) {
    const size_t C = d.C, KP = d.K + 1, CP = d.C + 1;
    return sizeof(float) * (2 * C * KP + C * d.V + 2 * C * CP + C * 16 + 3 * C);
}

cudaError_t launch_prep(const Dims& d, InType ty, const void* k, const void* q,
                        const void* v, const void* alpha, const void* beta,
                        const ChunkBufs& cb, bool write_T, cudaStream_t st) {
    dim3 grid(d.NC, d.H, d.B);
    const size_t sm = prep_smem_bytes(d);
    if (ty == InType::F32) {
        auto kern = prep_kernel<float>;
        cudaError_t e = set_smem(kern, sm);
        if (e != cudaSuccess) return e;
        kern<<<grid, kThreads, sm, st>>>(d, (const float*)k, (const float*)q, (const float*)v,
                                         (const float*)alpha, (const float*)beta, cb, write_T);
    } else {
        auto kern = prep_kernel<__nv_bfloat16>;
        cudaError_t e = set_smem(kern, sm);
        if (e != cudaSuccess) return e;
        kern<<<grid, kThreads, sm, st>>>(d, (const __nv_bfloat16*)k, (const __nv_bfloat16*)q,
                                         (const __nv_bfloat16*)v, (const __nv_bfloat16*)alpha,
                                         (const __nv_bfloat16*)beta, cb, write_T);
    }
    return cudaGetLastError();
}

cudaError_t launch_scan_fwd(const Dims& d, InType ty, const void* q, const void* k,
                            const ChunkBufs& cb, const float* s0, void* o, float* sT,
                            float* states, bool write_o, cudaStream_t st) {
    const int Vt = pick_vt(d);
    dim3 grid(d.V / Vt, d.H, d.B);
    const size_t C = d.C, KP = d.K + 1, CP = d.C + 1, VtP = Vt + 1;
    const size_t sm = sizeof(float) * (Vt * KP + 3 * C * KP + C * CP + 2 * C * VtP + 3 * C);
    if (ty == InType::F32) {
        auto kern = scan_fwd_kernel<float>;
        cudaError_t e = set_smem(kern, sm);
        if (e != cudaSuccess) return e;
        kern<<<grid, kThreads, sm, st>>>(d, Vt, (const float*)q, (const float*)k, cb, s0,
                                         (float*)o, sT, states, write_o);
    } else {
        auto kern = scan_fwd_kernel<__nv_bfloat16>;
        cudaError_t e = set_smem(kern, sm);
        if (e != cudaSuccess) return e;
        kern<<<grid, kThreads, sm, st>>>(d, Vt, (const __nv_bfloat16*)q, (const __nv_bfloat16*)k,
                                         cb, s0, (__nv_bfloat16*)o, sT, states, write_o);
    }
    return cudaGetLastError();
}

cudaError_t launch_scan_bwd(const Dims& d, InType ty, const void* q, const void* k,
                            const void* d_o, const ChunkBufs& cb, const float* states,
                            const float* dsT, const BwdBufs& bb, float* ds0,
                            cudaStream_t st) {
    const int Vt = pick_vt(d);
    dim3 grid(d.V / Vt, d.H, d.B);
    const size_t C = d.C, KP = d.K + 1, CP = d.C + 1, VtP = Vt + 1;
    const size_t sm = sizeof(float) * (2 * Vt * KP + 3 * C * KP + C * CP + 3 * C * VtP + 3 * C);
    if (ty == InType::F32) {
        auto kern = scan_bwd_kernel<float>;
        cudaError_t e = set_smem(kern, sm);
        if (e != cudaSuccess) return e;
        kern<<<grid, kThreads, sm, st>>>(d, Vt, (const float*)q, (const float*)k,
                                         (const float*)d_o, cb, states, dsT, bb, ds0);
    } else {
        auto kern = scan_bwd_kernel<__nv_bfloat16>;
        cudaError_t e = set_smem(kern, sm);
        if (e != cudaSuccess) return e;
        kern<<<grid, kThreads, sm, st>>>(d, Vt, (const __nv_bfloat16*)q, (const __nv_bfloat16*)k,
                                         (const __nv_bfloat16*)d_o, cb, states, dsT, bb, ds0);
    }
    return cudaGetLastError();
}

cudaError_t launch_grad(const Dims& d, InType ty, const void* q, const void* k,
                        const void* v, const void* alpha, const void* beta,
                        const void* d_o, const ChunkBufs& cb, const float* states,
                        const BwdBufs& bb, void* dq, void* dk, void* dv, void* dalpha,
                        void* dbeta, cudaStream_t st) {
    dim3 grid(d.NC, d.H, d.B);
    const size_t C = d.C, KP = d.K + 1, CP = d.C + 1;
    const size_t sm = sizeof(float) * (2 * C * KP + 7 * C * CP + 15 * C + kThreads);
    if (ty == InType::F32) {
        auto kern = grad_kernel<float>;
        cudaError_t e = set_smem(kern, sm);
        if (e != cudaSuccess) return e;
        kern<<<grid, kThreads, sm, st>>>(d, (const float*)q, (const float*)k, (const float*)v,
                                         (const float*)alpha, (const float*)beta,
                                         (const float*)d_o, cb, states, bb, (float*)dq,
                                         (float*)dk, (float*)dv, (float*)dalpha, (float*)dbeta);
    } else {
        using bf = __nv_bfloat16;
        auto kern = grad_kernel<bf>;
        cudaError_t e = set_smem(kern, sm);
        if (e != cudaSuccess) return e;
        kern<<<grid, kThreads, sm, st>>>(d, (const bf*)q, (const bf*)k, (const bf*)v,
                                         (const bf*)alpha, (const bf*)beta, (const bf*)d_o, cb,
                                         states, bb, (bf*)dq, (bf*)dk, (bf*)dv, (bf*)dalpha,
                                         (bf*)dbeta);
    }
    return cudaGetLastError();
}

}  // namespace gdn
