// api.cu -- the C ABI of libgdn.so (declared in include/gdn.h).
//
// Host-side only: argument checks (before any launch), workspace carving, and
// the launch sequence on the caller's stream.  Nothing here allocates device
// memory or synchronises.

#include <limits.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <vector>

#include "gdn.h"
#include "gdn_internal.h"

namespace {

thread_local char g_err[512] = "";

gdn_status fail(gdn_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return s;
}

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool supported_dim(int64_t x) { return x == 16 || x == 32 || x == 64 || x == 128; }

// Limit of the tensor-core kernels' bounded waits for calls made from now on, in
// nanoseconds (0: the kernels' default); see gdn_test_set_wait_limit.
uint32_t g_wait_limit_ns = 0;

// Checks the problem and fills Dims.  Returns GDN_OK or an error status.  With
// need_chunk false the chunk field is not used (gdn_decode, the prologue) and is
// not checked.
gdn_status check_problem(const gdn_problem* p, gdn::Dims* d, bool need_chunk = true) {
    if (!p) return fail(GDN_ERR_INVALID_ARG, "problem pointer is NULL");
    if (p->B < 0 || p->T < 0 || p->H < 0)
        return fail(GDN_ERR_INVALID_ARG, "negative size (B=%lld T=%lld H=%lld)",
                    (long long)p->B, (long long)p->T, (long long)p->H);
    if (p->dtype != GDN_F32 && p->dtype != GDN_BF16)
        return fail(GDN_ERR_UNSUPPORTED, "dtype %d is not GDN_F32 or GDN_BF16", (int)p->dtype);
    if (!supported_dim(p->K) || !supported_dim(p->V))
        return fail(GDN_ERR_UNSUPPORTED, "K=%lld V=%lld: each must be 16, 32, 64 or 128",
                    (long long)p->K, (long long)p->V);
    if (need_chunk && p->chunk != 16 && p->chunk != 32 && p->chunk != 64)
        return fail(GDN_ERR_UNSUPPORTED, "chunk=%d: must be 16, 32 or 64", (int)p->chunk);
    if (p->B > 65535 || p->H > 65535)
        return fail(GDN_ERR_UNSUPPORTED, "B=%lld H=%lld: each must be <= 65535",
                    (long long)p->B, (long long)p->H);
    if (p->T > (int64_t)1 << 30)
        return fail(GDN_ERR_UNSUPPORTED, "T=%lld exceeds 2^30", (long long)p->T);
    d->B = (int)p->B;
    d->T = (int)p->T;
    d->H = (int)p->H;
    d->K = (int)p->K;
    d->V = (int)p->V;
    d->C = need_chunk ? p->chunk : 64;
    d->NC = (int)((p->T + d->C - 1) / d->C);
    d->wait_ns = g_wait_limit_ns;
    // The tensor-core kernels address their buffers by row with 32-bit TMA
    // coordinates; the largest row is that of the last chunk's 128-row state, and a
    // packed batch of B sequences has at most B (NC + 1) chunks per head.
    if (need_chunk && p->dtype == GDN_BF16 && d->C == 64 &&
        (int64_t)d->B * d->H * (d->NC + 1) * 128 > (int64_t)INT32_MAX)
        return fail(GDN_ERR_UNSUPPORTED, "B*H*(ceil(T/64)+1)*128 = %lld exceeds 2^31-1 (32-bit row coordinates)",
                    (long long)((int64_t)d->B * d->H * (d->NC + 1) * 128));
    return GDN_OK;
}

// Workspace carving.  With base == nullptr only the size is computed.
struct Carver {
    char* base;
    size_t off = 0;
    template <typename T>
    T* take(size_t count) {
        T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
        off += round_up(count * sizeof(T));
        return p;
    }
};

size_t carve_chunk(const gdn::Dims& d, Carver& cv, gdn::ChunkBufs* cb, bool with_T) {
    const size_t nchunks = (size_t)d.NS() * d.NC;
    const size_t C = d.C;
    cb->G = cv.take<float>(nchunks * C);
    cb->W = cv.take<float>(nchunks * C * d.K);
    cb->Ut = cv.take<float>(nchunks * C * d.V);
    cb->Mqk = cv.take<float>(nchunks * C * C);
    cb->Tm = with_T ? cv.take<float>(nchunks * C * C) : nullptr;
    return cv.off;
}

// The tensor-core kernels keep K and V at 128 in their own buffers: a problem with
// K or V below 128 is read through TMA boxes that fill the missing columns with zeros,
// and every internal row is 128 wide (its extra columns hold zeros).
constexpr size_t kTcD = 128;

// Chunk results of the tensor-core path.  err is carved separately (it always
// lives in the workspace, even when the chunk results live in `saved`).
size_t carve_tc_chunk(const gdn::Dims& d, Carver& cv, gdn::TcBufs* tb, bool with_T) {
    const size_t rows = (size_t)d.NS() * d.NC * d.C;
    tb->G = cv.take<float>(rows);
    tb->W = cv.take<__nv_bfloat16>(rows * kTcD);
    tb->Ut = cv.take<__nv_bfloat16>(rows * kTcD);
    tb->Mqk = cv.take<__nv_bfloat16>(rows * d.C);
    tb->T = with_T ? cv.take<__nv_bfloat16>(rows * d.C) : nullptr;
    return cv.off;
}

// `saved` of the tensor-core path: bf16 chunk-start states [chunks*K, V] followed
// by the forward's chunk results (reused by the backward instead of recomputed).
size_t carve_tc_saved(const gdn::Dims& d, Carver& cv, __nv_bfloat16** states, gdn::TcBufs* tb) {
    *states = cv.take<__nv_bfloat16>((size_t)d.NS() * d.NC * kTcD * kTcD);
    return carve_tc_chunk(d, cv, tb, true);
}

size_t carve_tc(const gdn::Dims& d, Carver& cv, gdn::TcBufs* tb, bool with_T = false) {
    const size_t rows = (size_t)d.NS() * d.NC * d.C;
    tb->err = cv.take<int>(64);
    tb->G = cv.take<float>(rows);
    tb->W = cv.take<__nv_bfloat16>(rows * kTcD);
    tb->Ut = cv.take<__nv_bfloat16>(rows * kTcD);
    tb->Mqk = cv.take<__nv_bfloat16>(rows * d.C);
    tb->T = with_T ? cv.take<__nv_bfloat16>(rows * d.C) : nullptr;
    return cv.off;
}

size_t carve_tc_bwd(const gdn::Dims& d, Carver& cv, gdn::TcBufs* tb, gdn::TcBwdBufs* bb,
                    bool need_recompute) {
    if (need_recompute) {
        carve_tc(d, cv, tb, true);
    } else {
        tb->err = cv.take<int>(64);
    }
    const bool need_states = need_recompute;
    const size_t nchunks = (size_t)d.NS() * d.NC;
    const size_t rows = nchunks * d.C;
    bb->dU = cv.take<__nv_bfloat16>(rows * kTcD);
    bb->dS1 = cv.take<__nv_bfloat16>(nchunks * kTcD * kTcD);
    bb->dKp = cv.take<__nv_bfloat16>(nchunks * kTcD * d.C);
    bb->dWt = cv.take<__nv_bfloat16>(nchunks * kTcD * d.C);
    bb->dGp = cv.take<float>(rows);
    bb->states = need_states ? cv.take<__nv_bfloat16>(nchunks * kTcD * kTcD) : nullptr;
    return cv.off;
}

gdn::InType in_type(const gdn_problem* p) {
    return p->dtype == GDN_BF16 ? gdn::InType::BF16 : gdn::InType::F32;
}

size_t carve_bwd(const gdn::Dims& d, Carver& cv, gdn::ChunkBufs* cb, gdn::BwdBufs* bb,
                 bool need_states) {
    carve_chunk(d, cv, cb, true);
    const size_t nchunks = (size_t)d.NS() * d.NC;
    const size_t C = d.C, VK = (size_t)d.V * d.K;
    bb->states = need_states ? cv.take<float>(nchunks * VK) : nullptr;
    bb->U = cv.take<float>(nchunks * C * d.V);
    bb->dU = cv.take<float>(nchunks * C * d.V);
    bb->dS1 = cv.take<float>(nchunks * VK);
    bb->dW = cv.take<float>(nchunks * C * d.K);
    bb->dQ1 = cv.take<float>(nchunks * C * d.K);
    bb->dKh = cv.take<float>(nchunks * C * d.K);
    return cv.off;
}

struct Span {
    const void* p;
    size_t n;
    const char* name;
};

bool overlap(const Span& a, const Span& b) {
    if (!a.p || !b.p || a.n == 0 || b.n == 0) return false;
    const char* a0 = (const char*)a.p;
    const char* b0 = (const char*)b.p;
    return a0 < b0 + b.n && b0 < a0 + a.n;
}

gdn_status check_ptr(const Span& s, bool required) {
    if (!s.p) {
        if (required && s.n > 0) return fail(GDN_ERR_INVALID_ARG, "%s is NULL", s.name);
        return GDN_OK;
    }
    if (((uintptr_t)s.p) % 16 != 0)
        return fail(GDN_ERR_INVALID_ARG, "%s is not 16-byte aligned", s.name);
    return GDN_OK;
}

// Every output must be disjoint from every input and from every other output;
// `allow_same` lists (output, input) pairs that may be the identical buffer.
gdn_status check_overlaps(const Span* ins, int nin, const Span* outs, int nout,
                          const void* same_out, const void* same_in) {
    for (int i = 0; i < nout; ++i) {
        for (int j = 0; j < nin; ++j) {
            if (outs[i].p && outs[i].p == same_out && ins[j].p == same_in) continue;
            if (overlap(outs[i], ins[j]))
                return fail(GDN_ERR_INVALID_ARG, "output %s overlaps input %s", outs[i].name,
                            ins[j].name);
        }
        for (int j = i + 1; j < nout; ++j)
            if (overlap(outs[i], outs[j]))
                return fail(GDN_ERR_INVALID_ARG, "outputs %s and %s overlap", outs[i].name,
                            outs[j].name);
    }
    return GDN_OK;
}

gdn_status cuda_fail(cudaError_t e, const char* what) {
    return fail(GDN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Optional launch timer: while on, each launch is bracketed by two CUDA events
// recorded on the launch's own stream.
struct Profiler {
    bool on = false;
    int n = 0;
    std::vector<cudaEvent_t> ev;  // 2 per record
    std::vector<int> kid;
};
Profiler g_prof;

const char* const kKernelNames[gdn::KID_COUNT] = {
    "prep_kernel(fwd)", "scan_fwd_kernel", "prep_kernel(bwd)",
    "scan_fwd_kernel(state-only)", "scan_bwd_kernel", "grad_kernel",
    "prep_fwd_tc", "scan_fwd_tc", "prep_fwd_tc(bwd)", "scan_fwd_tc(state-only)",
    "scan_bwd_tc", "grad_qk_tc", "grad_wy_tc", "decode_kernel", "prologue_fwd_kernel",
    "prologue_bwd_kernel", "varlen_offsets", "varlen_gather", "varlen_scatter", "scan_fwd_tc(split pass 1)",
    "scan_bwd_tc(split pass 1)", "scan_fwd_tc(transitions)", "split_combine", "count_nonfinite_kernel"};

template <typename F>
cudaError_t timed(int kid, cudaStream_t st, F&& launch) {
    if (!g_prof.on || g_prof.n >= (int)g_prof.kid.size()) return launch();
    const int i = g_prof.n++;
    g_prof.kid[i] = kid;
    cudaEventRecord(g_prof.ev[2 * i], st);
    cudaError_t e = launch();
    cudaEventRecord(g_prof.ev[2 * i + 1], st);
    return e;
}

// Within-call sequence split (split.cu): every sequence's chunks are cut into P
// pieces whose scans run side by side; the pieces' affine maps are chained by
// the combine kernels and a second scan runs each piece from its true state.
struct SplitCfg {
    int P = 1;                     // pieces per sequence (1: no split)
    int nseq = 0;                  // sequences (dense: B)
    const int* seq_off = nullptr;  // chunk offsets of packed sequences, or NULL: rows of nc chunks
    int nc = 0;
};
struct SplitBufs {
    int* piece_off;
    float* R;  // zero-start final states (forward) / zero-start state gradients (backward)
    float* T;  // transitions
    float* X;  // piece input states (forward) / piece output state gradients (backward)
};

int g_split = 0;  // gdn_set_sequence_split: 0 automatic, 1 off, n >= 2 pieces

void carve_split(const gdn::Dims& fd, const SplitCfg& sp, Carver& cv, SplitBufs* sb) {
    const size_t slots = (size_t)sp.nseq * sp.P * fd.H;
    sb->piece_off = cv.take<int>((size_t)sp.nseq * sp.P + 1);
    sb->R = cv.take<float>(slots * fd.V * fd.K);
    sb->T = cv.take<float>(slots * fd.K * fd.K);
    sb->X = cv.take<float>(slots * fd.V * fd.K);
}

// Pieces per sequence: the knob, else (dense calls only) a power of two when the
// streams would leave most SMs idle, keeping >= 4 chunks per piece and the first
// pass (states and transitions, 64-column slices) within one wave.
int split_pieces(int64_t streams, int nc, bool automatic) {
    if (g_split == 1) return 1;
    if (g_split >= 2) return g_split;
    if (!automatic) return 1;
    const int64_t sms = gdn::sm_count();
    if (streams * 8 > sms / 2) return 1;
    int P = 1;
    while (2 * P <= nc / 4 && 4 * (2 * P) * streams <= sms) P *= 2;
    return P;
}

// The dims the tensor-core kernels run on, and the split of a dense call: a
// split needs one row of chunks per head (B = 1, or T a multiple of the chunk so
// that the batch rows lie back to back as whole chunks).
SplitCfg dense_split(const gdn::Dims& d, gdn::Dims* fd) {
    *fd = d;
    SplitCfg sp;
    if (d.B != 1 && d.T % d.C != 0) return sp;
    if (d.K != 128 || d.V != 128) return sp;  // the transitions are 128 x 128 maps
    const int P = split_pieces(d.NS(), d.NC, true);
    if (P < 2) return sp;
    fd->B = 1;
    fd->T = d.B * d.T;
    fd->NC = d.B * d.NC;
    sp.P = P;
    sp.nseq = d.B;
    sp.nc = d.NC;
    return sp;
}

// The tensor-core forward on dims d: the chunk kernel, then the scan.  The
// workspace holds carve_tc(d) (then carve_split with a split) and `saved` (or
// NULL) carve_tc_saved(d); `sq` (or NULL) runs packed sequences on the flat
// chunk layout; `sp` (or NULL, or P = 1) splits every sequence into pieces.
// With `raw` (gdn_fwd_raw), q, k are the raw rows and alpha, beta the gate logits:
// the chunk kernel normalises q, k into raw->qn, raw->kn, which the scans read.
gdn_status run_fwd_tc(const gdn::Dims& d, const void* q, const void* k, const void* v, const void* alpha,
                      const void* beta, const float* initial_state, void* o, float* final_state, void* saved,
                      void* workspace, const gdn::SeqMap* sq, const SplitCfg* sp, cudaStream_t cs,
                      const gdn::RawPrologue* raw = nullptr) {
    const void* qp = q;  // the rows the chunk kernel reads
    const void* kp = k;
    if (raw && raw->on) {  // the scans read the normalised rows
        q = raw->qn;
        k = raw->kn;
    }
    Carver cv{(char*)workspace};
    gdn::TcBufs tb;
    __nv_bfloat16* states = nullptr;
    carve_tc(d, cv, &tb);
    if (saved) {  // keep the chunk results for the backward
        Carver sv{(char*)saved};
        carve_tc_saved(d, sv, &states, &tb);
    }
    // Clears the error word and the persistent kernels' work counters.  gdn_fwd_noalloc
    // depends on this: its scratch array keeps the previous call's contents, and
    // these are the only scratch words read before the call writes them.
    cudaError_t e = cudaMemsetAsync(tb.err, 0, gdn::kErrWords * sizeof(int), cs);
    if (e != cudaSuccess) return cuda_fail(e, "error-flag reset");
    e = timed(gdn::KID_PREP_TC, cs, [&] { return gdn::launch_prep_tc(d, qp, kp, v, alpha, beta, tb, cs, raw); });
    if (e != cudaSuccess) return cuda_fail(e, "tensor-core chunk kernel");
    if (!sp || sp->P < 2) {
        e = timed(gdn::KID_SCAN_FWD_TC, cs, [&] {
            return gdn::launch_scan_fwd_tc(d, q, k, tb, initial_state, o, final_state, states, cs, sq);
        });
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core scan kernel");
        return GDN_OK;
    }
    SplitBufs sb;
    carve_split(d, *sp, cv, &sb);
    const int npieces = sp->nseq * sp->P;
    e = timed(gdn::KID_SPLIT_COMBINE, cs, [&] {
        return gdn::launch_split_pieces(sp->nseq, sp->P, sp->nc, sp->seq_off, sb.piece_off, cs);
    });
    if (e != cudaSuccess) return cuda_fail(e, "split pieces");
    const gdn::SeqMap both{sb.piece_off, npieces, 1, sb.T};
    e = timed(gdn::KID_SPLIT_FWD_P1, cs, [&] {
        return gdn::launch_scan_fwd_tc(d, q, k, tb, nullptr, nullptr, sb.R, nullptr, cs, &both);
    });
    if (e != cudaSuccess) return cuda_fail(e, "split pass 1");
    e = timed(gdn::KID_SPLIT_COMBINE, cs, [&] {
        return gdn::launch_combine_fwd(sp->nseq, sp->P, d.H, initial_state, sb.R, sb.T, sb.X, final_state, cs);
    });
    if (e != cudaSuccess) return cuda_fail(e, "split combine");
    const gdn::SeqMap pieces{sb.piece_off, npieces};
    e = timed(gdn::KID_SCAN_FWD_TC, cs, [&] {
        return gdn::launch_scan_fwd_tc(d, q, k, tb, sb.X, o, nullptr, states, cs, &pieces);
    });
    if (e != cudaSuccess) return cuda_fail(e, "tensor-core scan kernel");
    return GDN_OK;
}

// The tensor-core backward on dims d (same conventions as run_fwd_tc; the
// workspace holds carve_tc_bwd(d), then carve_split with a split).
// With `raw` (gdn_bwd_raw), q, k are the raw rows and alpha, beta the gate logits;
// raw->qn, kn, rq, rk hold the normalised rows and reciprocal norms (written by
// the forward into `saved`, or here by the chunk kernel when `saved` is NULL), and
// dq, dk, dalpha, dbeta receive the gradients of the raw inputs.
gdn_status run_bwd_tc(const gdn::Dims& d, const void* q, const void* k, const void* v, const void* alpha,
                      const void* beta, const float* initial_state, const void* saved, const void* d_o,
                      const float* d_final_state, void* dq, void* dk, void* dv, void* dalpha, void* dbeta,
                      float* d_initial_state, void* workspace, const gdn::SeqMap* sq, const SplitCfg* sp,
                      cudaStream_t cs, const gdn::RawPrologue* raw = nullptr) {
    const void* qp = q;  // the rows the chunk kernel reads
    const void* kp = k;
    if (raw && raw->on) {
        q = raw->qn;
        k = raw->kn;
    }
    Carver cv{(char*)workspace};
    gdn::TcBufs tb;
    gdn::TcBwdBufs tbb;
    carve_tc_bwd(d, cv, &tb, &tbb, saved == nullptr);
    const __nv_bfloat16* states = tbb.states;
    if (saved) {  // reuse the forward's states and chunk results
        Carver sv{(char*)const_cast<void*>(saved)};
        __nv_bfloat16* st = nullptr;
        int* err = tb.err;
        carve_tc_saved(d, sv, &st, &tb);
        tb.err = err;
        states = st;
    }
    const bool split = sp && sp->P >= 2;
    SplitBufs sb{};
    if (split) carve_split(d, *sp, cv, &sb);
    const int npieces = split ? sp->nseq * sp->P : 0;
    cudaError_t e = cudaMemsetAsync(tb.err, 0, gdn::kErrWords * sizeof(int), cs);
    if (e != cudaSuccess) return cuda_fail(e, "error-flag reset");
    if (split) {
        e = timed(gdn::KID_SPLIT_COMBINE, cs, [&] {
            return gdn::launch_split_pieces(sp->nseq, sp->P, sp->nc, sp->seq_off, sb.piece_off, cs);
        });
        if (e != cudaSuccess) return cuda_fail(e, "split pieces");
    }
    if (!saved) {
        e = timed(gdn::KID_PREP_TC_BWD, cs, [&] { return gdn::launch_prep_tc(d, qp, kp, v, alpha, beta, tb, cs, raw); });
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core chunk kernel");
        if (!split) {
            e = timed(gdn::KID_STATE_TC, cs, [&] {
                return gdn::launch_scan_fwd_tc(d, q, k, tb, initial_state, nullptr, nullptr, tbb.states, cs, sq);
            });
        } else {  // the chunk-start states by the split forward, states only
            const gdn::SeqMap both{sb.piece_off, npieces, 1, sb.T};
            e = timed(gdn::KID_SPLIT_FWD_P1, cs, [&] {
                return gdn::launch_scan_fwd_tc(d, q, k, tb, nullptr, nullptr, sb.R, nullptr, cs, &both);
            });
            if (e == cudaSuccess)
                e = timed(gdn::KID_SPLIT_COMBINE, cs, [&] {
                    return gdn::launch_combine_fwd(sp->nseq, sp->P, d.H, initial_state, sb.R, sb.T, sb.X, nullptr,
                                                   cs);
                });
            const gdn::SeqMap pieces{sb.piece_off, npieces};
            if (e == cudaSuccess)
                e = timed(gdn::KID_STATE_TC, cs, [&] {
                    return gdn::launch_scan_fwd_tc(d, q, k, tb, sb.X, nullptr, nullptr, tbb.states, cs, &pieces);
                });
        }
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core state recompute");
    } else if (split) {  // the pieces' transitions (the forward did not keep them)
        const gdn::SeqMap trans{sb.piece_off, npieces, 2, sb.T};
        e = timed(gdn::KID_SPLIT_TRANS, cs, [&] {
            return gdn::launch_scan_fwd_tc(d, q, k, tb, nullptr, nullptr, nullptr, nullptr, cs, &trans);
        });
        if (e != cudaSuccess) return cuda_fail(e, "split transitions");
    }
    if (!split) {
        e = timed(gdn::KID_SCAN_BWD_TC, cs, [&] {
            return gdn::launch_scan_bwd_tc(d, q, k, d_o, tb, d_final_state, tbb, d_initial_state, cs, sq);
        });
    } else {
        // pass 1: every piece from a zero end gradient; its dU, dS1 are rewritten by pass 2
        const gdn::SeqMap pieces{sb.piece_off, npieces};
        e = timed(gdn::KID_SPLIT_BWD_P1, cs, [&] {
            return gdn::launch_scan_bwd_tc(d, q, k, d_o, tb, nullptr, tbb, sb.R, cs, &pieces);
        });
        if (e == cudaSuccess)
            e = timed(gdn::KID_SPLIT_COMBINE, cs, [&] {
                return gdn::launch_combine_bwd(sp->nseq, sp->P, d.H, d_final_state, sb.R, sb.T, sb.X,
                                               d_initial_state, cs);
            });
        if (e == cudaSuccess)
            e = timed(gdn::KID_SCAN_BWD_TC, cs, [&] {
                return gdn::launch_scan_bwd_tc(d, q, k, d_o, tb, sb.X, tbb, nullptr, cs, &pieces);
            });
    }
    if (e != cudaSuccess) return cuda_fail(e, "tensor-core reverse scan");
    e = timed(gdn::KID_GRAD_QK_TC, cs, [&] { return gdn::launch_grad_qk_tc(d, q, k, d_o, tb, states, tbb, dq, cs, raw); });
    if (e != cudaSuccess) return cuda_fail(e, "tensor-core gradient kernel (q, k)");
    e = timed(gdn::KID_GRAD_WY_TC, cs, [&] {
        return gdn::launch_grad_wy_tc(d, k, v, alpha, beta, tb, tbb, dk, dv, dalpha, dbeta, cs, raw);
    });
    if (e != cudaSuccess) return cuda_fail(e, "tensor-core gradient kernel (WY)");
    return GDN_OK;
}

}  // namespace

namespace gdn {
// Lets other translation units of the library report a message through
// gdn_last_error().
void set_last_error(const char* msg) { snprintf(g_err, sizeof(g_err), "%s", msg); }
}  // namespace gdn

extern "C" {

int gdn_version(void) { return 100; }

const char* gdn_status_string(gdn_status s) {
    switch (s) {
        case GDN_OK: return "ok";
        case GDN_ERR_INVALID_ARG: return "invalid argument";
        case GDN_ERR_UNSUPPORTED: return "unsupported problem";
        case GDN_ERR_WORKSPACE: return "workspace too small";
        case GDN_ERR_CUDA: return "CUDA launch failed";
    }
    return "unknown status";
}

const char* gdn_last_error(void) { return g_err; }

gdn_status gdn_test_set_wait_limit(uint32_t ns) {
    g_wait_limit_ns = ns;
    return GDN_OK;
}

size_t gdn_fwd_workspace_bytes(const gdn_problem* p) {
    gdn::Dims d{};
    if (check_problem(p, &d) != GDN_OK) return 0;
    Carver cv{nullptr};
    if (d.NS() * d.NC == 0) return 0;
    if (gdn::tc_fwd_supported(d, p->dtype == GDN_BF16 ? gdn::InType::BF16 : gdn::InType::F32)) {
        gdn::TcBufs tb;
        gdn::Dims fd;
        const SplitCfg sp = dense_split(d, &fd);
        carve_tc(fd, cv, &tb);
        SplitBufs sb;
        if (sp.P >= 2) carve_split(fd, sp, cv, &sb);
        return cv.off;
    }
    gdn::ChunkBufs cb;
    return carve_chunk(d, cv, &cb, false);
}

size_t gdn_saved_bytes(const gdn_problem* p) {
    gdn::Dims d{};
    if (check_problem(p, &d) != GDN_OK) return 0;
    if (gdn::tc_fwd_supported(d, in_type(p))) {
        Carver cv{nullptr};
        __nv_bfloat16* st;
        gdn::TcBufs tb;
        return carve_tc_saved(d, cv, &st, &tb);
    }
    return (size_t)d.NS() * d.NC * d.V * d.K * sizeof(float);
}

size_t gdn_bwd_workspace_bytes(const gdn_problem* p) {
    gdn::Dims d{};
    if (check_problem(p, &d) != GDN_OK) return 0;
    Carver cv{nullptr};
    if (d.NS() * d.NC == 0) return 0;
    if (gdn::tc_fwd_supported(d, in_type(p))) {
        gdn::TcBufs tb;
        gdn::TcBwdBufs tbb;
        gdn::Dims fd;
        const SplitCfg sp = dense_split(d, &fd);
        carve_tc_bwd(fd, cv, &tb, &tbb, true);
        SplitBufs sb;
        if (sp.P >= 2) carve_split(fd, sp, cv, &sb);
        return cv.off;
    }
    gdn::ChunkBufs cb;
    gdn::BwdBufs bb;
    return carve_bwd(d, cv, &cb, &bb, true);
}

gdn_status gdn_fwd(const gdn_problem* p, const void* q, const void* k, const void* v,
                   const void* alpha, const void* beta, const float* initial_state,
                   void* o, float* final_state, void* saved, void* workspace,
                   size_t workspace_bytes, void* stream) {
    g_err[0] = 0;
    gdn::Dims d{};
    gdn_status st = check_problem(p, &d);
    if (st != GDN_OK) return st;
    const size_t es = p->dtype == GDN_BF16 ? 2 : 4;
    const size_t BTH = (size_t)d.B * d.T * d.H;
    const size_t nstate = (size_t)d.NS() * d.V * d.K * sizeof(float);
    const size_t need = gdn_fwd_workspace_bytes(p);
    const Span ins[] = {{q, BTH * d.K * es, "q"},       {k, BTH * d.K * es, "k"},
                        {v, BTH * d.V * es, "v"},       {alpha, BTH * es, "alpha"},
                        {beta, BTH * es, "beta"},       {initial_state, nstate, "initial_state"}};
    const Span outs[] = {{o, BTH * d.V * es, "o"},
                         {final_state, nstate, "final_state"},
                         {saved, gdn_saved_bytes(p), "saved"},
                         {workspace, need, "workspace"}};
    for (int i = 0; i < 6; ++i)  // initial_state is optional
        if ((st = check_ptr(ins[i], i != 5)) != GDN_OK) return st;
    for (int i = 0; i < 4; ++i)  // final_state and saved are optional
        if ((st = check_ptr(outs[i], i == 0 || i == 3)) != GDN_OK) return st;
    if (workspace_bytes < need)
        return fail(GDN_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes,
                    need);
    if ((st = check_overlaps(ins, 6, outs, 4, final_state, initial_state)) != GDN_OK) return st;

    cudaStream_t cs = (cudaStream_t)stream;
    if (d.NS() == 0) return GDN_OK;
    if (d.T == 0) {  // empty sequence: the final state is the initial state
        cudaError_t e = cudaSuccess;
        if (final_state && final_state != initial_state)
            e = initial_state ? cudaMemcpyAsync(final_state, initial_state, nstate,
                                                cudaMemcpyDeviceToDevice, cs)
                              : cudaMemsetAsync(final_state, 0, nstate, cs);
        return e == cudaSuccess ? GDN_OK : cuda_fail(e, "empty-sequence state copy");
    }
    const gdn::InType ty = p->dtype == GDN_BF16 ? gdn::InType::BF16 : gdn::InType::F32;
    if (gdn::tc_fwd_supported(d, ty)) {
        gdn::Dims fd;
        const SplitCfg sp = dense_split(d, &fd);
        return run_fwd_tc(fd, q, k, v, alpha, beta, initial_state, o, final_state, saved, workspace, nullptr, &sp,
                          cs);
    }
    Carver cv{(char*)workspace};
    gdn::ChunkBufs cb;
    carve_chunk(d, cv, &cb, false);
    cudaError_t e = timed(gdn::KID_PREP_FWD, cs, [&] {
        return gdn::launch_prep(d, ty, k, q, v, alpha, beta, cb, false, cs);
    });
    if (e != cudaSuccess) return cuda_fail(e, "chunk kernel");
    e = timed(gdn::KID_SCAN_FWD, cs, [&] {
        return gdn::launch_scan_fwd(d, ty, q, k, cb, initial_state, o, final_state,
                                    (float*)saved, true, cs);
    });
    if (e != cudaSuccess) return cuda_fail(e, "scan kernel");
    return GDN_OK;
}

// ---------------------------------------------------------------- varlen
// Packed sequences run on one of two layouts:
//  * flat (tensor-core path): the kernels read and write the packed tensors in
//    place, one row of chunks per head (B = 1), every sequence starting a new
//    chunk: nc_max = ceil(total / C) + S chunks bound the sum of ceil(len_s / C),
//    and the chunk-token map (Dims::tok, len) gives each chunk's first packed
//    token and its number of tokens; the scans take a SeqMap.  Workspace: the
//    tensor-core workspace (its error word, word 0, is the call's), then
//    chunk_off [S+1], order [S], tok [nc_max], len [nc_max] and an error int for
//    the offsets; with `saved` the four arrays live there instead (the backward
//    reuses them), followed by the chunk kernels' own results.
//  * padded (other shapes): [S, max_len] streams laid out in the workspace (the
//    error word, chunk_off, the inner workspace, the laid-out tensors), gdn_fwd /
//    gdn_bwd as they are.
namespace {
struct VarlenPlan {
    bool flat;
    int pieces;    // within-call split of every sequence (flat layout; 1: none)
    gdn::Dims pd;  // the problem the chunk kernels run on
    size_t off, inner, q, k, v, a, b, o, d_o, dq, dk, dv, da, db, total;
    size_t nints;  // flat: ints at `off` (chunk_off, order, tok, len, the offsets' error)
    // `saved` of the flat layout: chunk_off, order, tok, len, then the chunk
    // kernels' own results
    size_t s_off, s_tc, saved;
};

gdn_status varlen_plan(const gdn_problem* p, int64_t total, bool bwd, VarlenPlan* L) {
    gdn::Dims d{};
    gdn_status st = check_problem(p, &d);
    if (st != GDN_OK) return st;
    if (total < 0 || total > (int64_t)p->B * p->T)
        return fail(GDN_ERR_INVALID_ARG, "total=%lld must be in [0, B*T] (B sequences of at most T tokens)",
                    (long long)total);
    *L = VarlenPlan{};
    L->flat = gdn::tc_fwd_supported(d, in_type(p));
    L->pd = d;
    int64_t nc_max = 0;
    if (L->flat) {
        nc_max = (total + d.C - 1) / d.C + d.B;
        if (nc_max * d.C > ((int64_t)1 << 30))
            return fail(GDN_ERR_UNSUPPORTED, "total=%lld with B=%d sequences exceeds 2^30 chunk rows",
                        (long long)total, d.B);
        L->pd.B = 1;
        L->pd.NC = (int)nc_max;
        L->pd.T = (int)total;  // the packed tensors the kernels read in place
    }
    const gdn::Dims& q = L->pd;
    const size_t es = p->dtype == GDN_BF16 ? 2 : 4;
    size_t inner_bytes = 0;
    Carver cv{nullptr};
    L->pieces = (L->flat && d.K == 128 && d.V == 128) ? split_pieces((int64_t)d.B * d.H, 0, false) : 1;
    if (q.NS() * q.NC > 0) {
        if (L->flat) {
            gdn::TcBufs tb;
            gdn::TcBwdBufs tbb;
            inner_bytes = bwd ? carve_tc_bwd(q, cv, &tb, &tbb, true) : carve_tc(q, cv, &tb);
            if (L->pieces >= 2) {
                SplitBufs sb;
                SplitCfg sp;
                sp.P = L->pieces;
                sp.nseq = d.B;
                carve_split(q, sp, cv, &sb);
                inner_bytes = cv.off;
            }
        } else {
            inner_bytes = bwd ? gdn_bwd_workspace_bytes(p) : gdn_fwd_workspace_bytes(p);
        }
    }
    if (L->flat) {
        L->nints = (size_t)2 * d.B + 1 + (size_t)2 * nc_max + 1;
        L->inner = 0;
        L->off = round_up(inner_bytes > 0 ? inner_bytes : sizeof(int));
        L->total = L->off + round_up(L->nints * sizeof(int));
        Carver sv{nullptr};
        __nv_bfloat16* states;
        gdn::TcBufs tb;
        const size_t tc = q.NS() * q.NC > 0 ? carve_tc_saved(q, sv, &states, &tb) : 0;
        L->s_off = 0;
        L->s_tc = round_up((L->nints - 1) * sizeof(int));
        L->saved = L->s_tc + tc;
        return GDN_OK;
    }
    L->saved = gdn_saved_bytes(p);
    const size_t BTH = (size_t)q.B * q.T * q.H;
    size_t off = kAlign;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += round_up(bytes);
        return o;
    };
    L->off = take(((size_t)2 * d.B + 1) * sizeof(int));  // chunk_off [B+1], order [B]
    L->inner = take(inner_bytes);
    L->q = take(BTH * q.K * es);
    L->k = take(BTH * q.K * es);
    L->v = take(BTH * q.V * es);
    L->a = take(BTH * es);
    L->b = take(BTH * es);
    if (!bwd) {
        L->o = take(BTH * q.V * es);
    } else {
        L->d_o = take(BTH * q.V * es);
        L->dq = take(BTH * q.K * es);
        L->dk = take(BTH * q.K * es);
        L->dv = take(BTH * q.V * es);
        L->da = take(BTH * es);
        L->db = take(BTH * es);
    }
    L->total = off;
    return GDN_OK;
}

uint32_t one_bits(const gdn_problem* p) { return p->dtype == GDN_BF16 ? 0x3F80u : 0x3F800000u; }

// The padded layout: packed -> laid out (gather) or back (scatter) for one tensor
// of `width` bytes per (token, head).  `merge` (row moves only) is ORed into the
// error word.
cudaError_t varlen_move(const VarlenPlan& L, int64_t total, const int32_t* cu, char* ws,
                        int width, const void* src, void* dst, uint32_t fill, bool scatter, const int* merge,
                        cudaStream_t cs) {
    int* err = (int*)ws;
    const gdn::Dims& d = L.pd;
    return timed(scatter ? gdn::KID_VARLEN_SCATTER : gdn::KID_VARLEN_GATHER, cs, [&] {
        if (width % 16 == 0)
            return gdn::launch_varlen_rows(d, total, cu, width, src, dst, fill, scatter, err, merge, cs);
        return gdn::launch_varlen_elems(d, total, cu, width, src, dst, fill, scatter, err, cs);
    });
}

// The flat layout's maps: chunk_off, order, tok, len at `ints` (computed on the
// device when `compute`, else read from the forward's `saved`), and the dims with
// the chunk-token map.  The offsets' error int (in the workspace) is cleared and
// set by the offsets kernel.
struct FlatMaps {
    gdn::Dims d;
    gdn::SeqMap sq;
};
gdn_status flat_maps(const VarlenPlan& L, const gdn_problem* p, int64_t total, const int32_t* cu, char* ints_base,
                     char* ws, bool compute, cudaStream_t cs, FlatMaps* fm) {
    const int S = (int)p->B, nc = L.pd.NC;
    int* ints = (int*)ints_base;
    int* chunk_off = ints;
    int* order = ints + S + 1;
    int* tok = order + S;
    int* len = tok + nc;
    int* offerr = (int*)(ws + L.off) + (L.nints - 1);
    fm->d = L.pd;
    fm->d.tok = tok;
    fm->d.len = len;
    // longest sequences first; the longest has at most ceil(max_len / C) chunks
    fm->sq = gdn::SeqMap{chunk_off, S, 0, nullptr, order, (int)((p->T + L.pd.C - 1) / L.pd.C)};
    if (!compute) return GDN_OK;
    cudaError_t e = cudaMemsetAsync(offerr, 0, sizeof(int), cs);
    if (e == cudaSuccess)
        e = timed(gdn::KID_VARLEN_OFFSETS, cs, [&] {
            cudaError_t e2 = gdn::launch_varlen_offsets(S, total, (int)p->T, L.pd.C, nc, cu, chunk_off, order, offerr,
                                                        cs);
            if (e2 == cudaSuccess)
                e2 = gdn::launch_varlen_chunk_tokens(S, total, L.pd.C, nc, cu, chunk_off, tok, len, cs);
            return e2;
        });
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "varlen offsets");
}

// The offsets' error int joins the call's error word (word 0 of the workspace,
// the tensor-core kernels' own), after the kernels have run.
gdn_status flat_merge_error(const VarlenPlan& L, char* ws, cudaStream_t cs) {
    const int* offerr = (const int*)(ws + L.off) + (L.nints - 1);
    cudaError_t e = gdn::launch_route_states(0, 0, nullptr, nullptr, nullptr, offerr, (int*)ws, cs);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "varlen error word");
}

gdn_status check_cu(const gdn_problem* p, const int32_t* cu) {
    if (!cu && p->B > 0) return fail(GDN_ERR_INVALID_ARG, "cu_seqlens is NULL");
    if (((uintptr_t)cu) % 4 != 0) return fail(GDN_ERR_INVALID_ARG, "cu_seqlens is not 4-byte aligned");
    return GDN_OK;
}
}  // namespace

size_t gdn_varlen_fwd_workspace_bytes(const gdn_problem* p, int64_t total) {
    VarlenPlan L;
    return varlen_plan(p, total, false, &L) == GDN_OK ? L.total : 0;
}

size_t gdn_varlen_bwd_workspace_bytes(const gdn_problem* p, int64_t total) {
    VarlenPlan L;
    return varlen_plan(p, total, true, &L) == GDN_OK ? L.total : 0;
}

size_t gdn_varlen_saved_bytes(const gdn_problem* p, int64_t total) {
    VarlenPlan L;
    return varlen_plan(p, total, false, &L) == GDN_OK ? L.saved : 0;
}

gdn_status gdn_varlen_fwd(const gdn_problem* p, int64_t total, const int32_t* cu_seqlens, const void* q,
                          const void* k, const void* v, const void* alpha, const void* beta,
                          const float* initial_state, void* o, float* final_state, void* saved, void* workspace,
                          size_t workspace_bytes, void* stream) {
    g_err[0] = 0;
    VarlenPlan L;
    gdn_status st = varlen_plan(p, total, false, &L);
    if (st != GDN_OK) return st;
    if ((st = check_cu(p, cu_seqlens)) != GDN_OK) return st;
    const size_t es = p->dtype == GDN_BF16 ? 2 : 4;
    const size_t TH = (size_t)total * p->H;
    const size_t nstate = (size_t)p->B * p->H * p->K * p->V * sizeof(float);
    const Span ins[] = {{q, TH * p->K * es, "q"},         {k, TH * p->K * es, "k"},
                        {v, TH * p->V * es, "v"},         {alpha, TH * es, "alpha"},
                        {beta, TH * es, "beta"},         {initial_state, nstate, "initial_state"},
                        {cu_seqlens, ((size_t)p->B + 1) * 4, "cu_seqlens"}};
    const Span outs[] = {{o, TH * p->V * es, "o"},
                         {workspace, L.total, "workspace"},
                         {final_state, nstate, "final_state"},
                         {saved, L.saved, "saved"}};
    for (int i = 0; i < 6; ++i)
        if ((st = check_ptr(ins[i], i != 5)) != GDN_OK) return st;
    for (int i = 0; i < 4; ++i)
        if ((st = check_ptr(outs[i], i < 2)) != GDN_OK) return st;
    if (workspace_bytes < L.total)
        return fail(GDN_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, L.total);
    if ((st = check_overlaps(ins, 7, outs, 4, final_state, initial_state)) != GDN_OK) return st;
    cudaStream_t cs = (cudaStream_t)stream;
    char* ws = (char*)workspace;
    cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(int), cs);
    if (e != cudaSuccess) return cuda_fail(e, "error-word reset");
    if (p->B * p->H == 0) return GDN_OK;
    const int S = (int)p->B, kb = (int)(p->K * es), vb = (int)(p->V * es);
    if (L.flat) {
        if (total == 0) {  // no tokens: every state passes through
            if (final_state) {
                e = initial_state ? cudaMemcpyAsync(final_state, initial_state, nstate, cudaMemcpyDeviceToDevice, cs)
                                  : cudaMemsetAsync(final_state, 0, nstate, cs);
                if (e != cudaSuccess) return cuda_fail(e, "state copy");
            }
            return GDN_OK;
        }
        FlatMaps fm;
        if ((st = flat_maps(L, p, total, cu_seqlens, saved ? (char*)saved + L.s_off : ws + L.off, ws, true, cs, &fm)) !=
            GDN_OK)
            return st;
        SplitCfg sp;
        sp.P = L.pieces;
        sp.nseq = S;
        sp.seq_off = fm.sq.chunk_off;
        st = run_fwd_tc(fm.d, q, k, v, alpha, beta, initial_state, o, final_state,
                        saved ? (char*)saved + L.s_tc : nullptr, ws + L.inner, &fm.sq, &sp, cs);
        if (st != GDN_OK) return st;
        return flat_merge_error(L, ws, cs);
    }
    const void* src[5] = {q, k, v, alpha, beta};
    const size_t dst[5] = {L.q, L.k, L.v, L.a, L.b};
    const int width[5] = {kb, kb, vb, (int)es, (int)es};
    const uint32_t fill[5] = {0u, 0u, 0u, one_bits(p), 0u};
    for (int i = 0; i < 5 && e == cudaSuccess; ++i)
        e = varlen_move(L, total, cu_seqlens, ws, width[i], src[i], ws + dst[i], fill[i], false, nullptr, cs);
    if (e != cudaSuccess) return cuda_fail(e, "varlen gather");
    st = gdn_fwd(p, ws + L.q, ws + L.k, ws + L.v, ws + L.a, ws + L.b, initial_state, ws + L.o, final_state, saved,
                 ws + L.inner, L.q - L.inner, stream);
    if (st != GDN_OK) return st;
    e = varlen_move(L, total, cu_seqlens, ws, vb, ws + L.o, o, 0u, true, nullptr, cs);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "varlen scatter");
}

gdn_status gdn_varlen_bwd(const gdn_problem* p, int64_t total, const int32_t* cu_seqlens, const void* q,
                          const void* k, const void* v, const void* alpha, const void* beta,
                          const float* initial_state, const void* saved, const void* d_o,
                          const float* d_final_state, void* dq, void* dk, void* dv, void* dalpha, void* dbeta,
                          float* d_initial_state, void* workspace, size_t workspace_bytes, void* stream) {
    g_err[0] = 0;
    VarlenPlan L;
    gdn_status st = varlen_plan(p, total, true, &L);
    if (st != GDN_OK) return st;
    if ((st = check_cu(p, cu_seqlens)) != GDN_OK) return st;
    const size_t es = p->dtype == GDN_BF16 ? 2 : 4;
    const size_t TH = (size_t)total * p->H;
    const size_t nstate = (size_t)p->B * p->H * p->K * p->V * sizeof(float);
    const Span ins[] = {{q, TH * p->K * es, "q"},
                        {k, TH * p->K * es, "k"},
                        {v, TH * p->V * es, "v"},
                        {alpha, TH * es, "alpha"},
                        {beta, TH * es, "beta"},
                        {d_o, TH * p->V * es, "d_o"},
                        {initial_state, nstate, "initial_state"},
                        {d_final_state, nstate, "d_final_state"},
                        {saved, L.saved, "saved"},
                        {cu_seqlens, ((size_t)p->B + 1) * 4, "cu_seqlens"}};
    const Span outs[] = {{dq, TH * p->K * es, "dq"},
                         {dk, TH * p->K * es, "dk"},
                         {dv, TH * p->V * es, "dv"},
                         {dalpha, TH * es, "dalpha"},
                         {dbeta, TH * es, "dbeta"},
                         {workspace, L.total, "workspace"},
                         {d_initial_state, nstate, "d_initial_state"}};
    for (int i = 0; i < 9; ++i)
        if ((st = check_ptr(ins[i], i < 6)) != GDN_OK) return st;
    for (int i = 0; i < 7; ++i)
        if ((st = check_ptr(outs[i], i < 6)) != GDN_OK) return st;
    if (workspace_bytes < L.total)
        return fail(GDN_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, L.total);
    if ((st = check_overlaps(ins, 10, outs, 7, d_initial_state, d_final_state)) != GDN_OK) return st;
    cudaStream_t cs = (cudaStream_t)stream;
    char* ws = (char*)workspace;
    cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(int), cs);
    if (e != cudaSuccess) return cuda_fail(e, "error-word reset");
    if (p->B * p->H == 0) return GDN_OK;
    const int S = (int)p->B, kb = (int)(p->K * es), vb = (int)(p->V * es);
    if (L.flat) {
        if (total == 0) {  // no tokens: every state gradient passes through
            if (d_initial_state) {
                e = d_final_state
                        ? cudaMemcpyAsync(d_initial_state, d_final_state, nstate, cudaMemcpyDeviceToDevice, cs)
                        : cudaMemsetAsync(d_initial_state, 0, nstate, cs);
                if (e != cudaSuccess) return cuda_fail(e, "state copy");
            }
            return GDN_OK;
        }
        // the forward's maps when `saved` is given, else computed here
        FlatMaps fm;
        char* ints = saved ? (char*)const_cast<void*>(saved) + L.s_off : ws + L.off;
        if ((st = flat_maps(L, p, total, cu_seqlens, ints, ws, saved == nullptr, cs, &fm)) != GDN_OK) return st;
        SplitCfg sp;
        sp.P = L.pieces;
        sp.nseq = S;
        sp.seq_off = fm.sq.chunk_off;
        st = run_bwd_tc(fm.d, q, k, v, alpha, beta, initial_state, saved ? (const char*)saved + L.s_tc : nullptr,
                        d_o, d_final_state, dq, dk, dv, dalpha, dbeta, d_initial_state, ws + L.inner, &fm.sq, &sp,
                        cs);
        if (st != GDN_OK) return st;
        return saved ? GDN_OK : flat_merge_error(L, ws, cs);
    }
    const void* src[6] = {q, k, v, d_o, alpha, beta};
    const size_t dst[6] = {L.q, L.k, L.v, L.d_o, L.a, L.b};
    const int width[6] = {kb, kb, vb, vb, (int)es, (int)es};
    const uint32_t fill[6] = {0u, 0u, 0u, 0u, one_bits(p), 0u};
    for (int i = 0; i < 6 && e == cudaSuccess; ++i)
        e = varlen_move(L, total, cu_seqlens, ws, width[i], src[i], ws + dst[i], fill[i], false, nullptr, cs);
    if (e != cudaSuccess) return cuda_fail(e, "varlen gather");
    st = gdn_bwd(p, ws + L.q, ws + L.k, ws + L.v, ws + L.a, ws + L.b, initial_state, saved, ws + L.d_o,
                 d_final_state, ws + L.dq, ws + L.dk, ws + L.dv, ws + L.da, ws + L.db, d_initial_state,
                 ws + L.inner, L.q - L.inner, stream);
    if (st != GDN_OK) return st;
    const size_t gsrc[5] = {L.dq, L.dk, L.dv, L.da, L.db};
    void* gdst[5] = {dq, dk, dv, dalpha, dbeta};
    const int gw[5] = {kb, kb, vb, (int)es, (int)es};
    for (int i = 0; i < 5 && e == cudaSuccess; ++i)
        e = varlen_move(L, total, cu_seqlens, ws, gw[i], ws + gsrc[i], gdst[i], 0u, true, nullptr, cs);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "varlen scatter");
}

gdn_status gdn_prologue_fwd(const gdn_problem* p, const void* q_raw, const void* k_raw, const void* a_logit,
                            const void* b_logit, void* q, void* k, void* alpha, void* beta, void* stream) {
    g_err[0] = 0;
    gdn::Dims d{};
    gdn_status st = check_problem(p, &d, false);
    if (st != GDN_OK) return st;
    const size_t es = p->dtype == GDN_BF16 ? 2 : 4;
    const size_t BTH = (size_t)d.B * d.T * d.H;
    const Span ins[] = {{q_raw, BTH * d.K * es, "q_raw"}, {k_raw, BTH * d.K * es, "k_raw"},
                        {a_logit, BTH * es, "a_logit"},   {b_logit, BTH * es, "b_logit"}};
    const Span outs[] = {{q, BTH * d.K * es, "q"}, {k, BTH * d.K * es, "k"}, {alpha, BTH * es, "alpha"},
                         {beta, BTH * es, "beta"}};
    for (int i = 0; i < 4; ++i)
        if ((st = check_ptr(ins[i], true)) != GDN_OK || (st = check_ptr(outs[i], true)) != GDN_OK) return st;
    if ((st = check_overlaps(ins, 4, outs, 4, nullptr, nullptr)) != GDN_OK) return st;
    if (BTH == 0) return GDN_OK;
    cudaStream_t cs = (cudaStream_t)stream;
    const gdn::InType ty = p->dtype == GDN_BF16 ? gdn::InType::BF16 : gdn::InType::F32;
    cudaError_t e = timed(gdn::KID_PROLOGUE_FWD, cs, [&] {
        return gdn::launch_prologue_fwd(d, ty, q_raw, k_raw, a_logit, b_logit, q, k, alpha, beta, cs);
    });
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "prologue kernel");
}

gdn_status gdn_prologue_bwd(const gdn_problem* p, const void* q_raw, const void* k_raw, const void* a_logit,
                            const void* b_logit, const void* dq, const void* dk, const void* dalpha,
                            const void* dbeta, void* dq_raw, void* dk_raw, void* da_logit, void* db_logit,
                            void* stream) {
    g_err[0] = 0;
    gdn::Dims d{};
    gdn_status st = check_problem(p, &d, false);
    if (st != GDN_OK) return st;
    const size_t es = p->dtype == GDN_BF16 ? 2 : 4;
    const size_t BTH = (size_t)d.B * d.T * d.H;
    const Span ins[] = {{q_raw, BTH * d.K * es, "q_raw"}, {k_raw, BTH * d.K * es, "k_raw"},
                        {a_logit, BTH * es, "a_logit"},   {b_logit, BTH * es, "b_logit"},
                        {dq, BTH * d.K * es, "dq"},       {dk, BTH * d.K * es, "dk"},
                        {dalpha, BTH * es, "dalpha"},     {dbeta, BTH * es, "dbeta"}};
    const Span outs[] = {{dq_raw, BTH * d.K * es, "dq_raw"}, {dk_raw, BTH * d.K * es, "dk_raw"},
                         {da_logit, BTH * es, "da_logit"},   {db_logit, BTH * es, "db_logit"}};
    for (int i = 0; i < 8; ++i)
        if ((st = check_ptr(ins[i], true)) != GDN_OK) return st;
    for (int i = 0; i < 4; ++i)
        if ((st = check_ptr(outs[i], true)) != GDN_OK) return st;
    if ((st = check_overlaps(ins, 8, outs, 4, nullptr, nullptr)) != GDN_OK) return st;
    if (BTH == 0) return GDN_OK;
    cudaStream_t cs = (cudaStream_t)stream;
    const gdn::InType ty = p->dtype == GDN_BF16 ? gdn::InType::BF16 : gdn::InType::F32;
    cudaError_t e = timed(gdn::KID_PROLOGUE_BWD, cs, [&] {
        return gdn::launch_prologue_bwd(d, ty, q_raw, k_raw, a_logit, b_logit, dq, dk, dalpha, dbeta, dq_raw,
                                        dk_raw, da_logit, db_logit, cs);
    });
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "prologue backward kernel");
}

gdn_status gdn_decode(const gdn_problem* p, const void* q, const void* k, const void* v,
                      const void* alpha, const void* beta, float* state, void* o, void* stream) {
    g_err[0] = 0;
    gdn::Dims d{};
    gdn_status st = check_problem(p, &d, false);
    if (st != GDN_OK) return st;
    const size_t es = p->dtype == GDN_BF16 ? 2 : 4;
    const size_t BTH = (size_t)d.B * d.T * d.H;
    const size_t nstate = (size_t)d.NS() * d.V * d.K * sizeof(float);
    const Span ins[] = {{q, BTH * d.K * es, "q"},   {k, BTH * d.K * es, "k"}, {v, BTH * d.V * es, "v"},
                        {alpha, BTH * es, "alpha"}, {beta, BTH * es, "beta"}};
    const Span outs[] = {{o, BTH * d.V * es, "o"}, {state, nstate, "state"}};
    for (int i = 0; i < 5; ++i)
        if ((st = check_ptr(ins[i], true)) != GDN_OK) return st;
    for (int i = 0; i < 2; ++i)
        if ((st = check_ptr(outs[i], true)) != GDN_OK) return st;
    if ((st = check_overlaps(ins, 5, outs, 2, nullptr, nullptr)) != GDN_OK) return st;
    if (d.NS() == 0 || d.T == 0) return GDN_OK;
    cudaStream_t cs = (cudaStream_t)stream;
    const gdn::InType ty = p->dtype == GDN_BF16 ? gdn::InType::BF16 : gdn::InType::F32;
    cudaError_t e = timed(gdn::KID_DECODE, cs, [&] {
        return gdn::launch_decode(d, ty, q, k, v, alpha, beta, state, o, cs);
    });
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "decode kernel");
}

gdn_status gdn_count_nonfinite(const void* x, int64_t n, gdn_dtype dtype, int64_t* count, void* stream) {
    g_err[0] = 0;
    if (n < 0) return fail(GDN_ERR_INVALID_ARG, "n=%lld is negative", (long long)n);
    if (dtype != GDN_F32 && dtype != GDN_BF16)
        return fail(GDN_ERR_UNSUPPORTED, "dtype %d is not GDN_F32 or GDN_BF16", (int)dtype);
    if (!count) return fail(GDN_ERR_INVALID_ARG, "count is NULL");
    if (((uintptr_t)count) % 8 != 0) return fail(GDN_ERR_INVALID_ARG, "count is not 8-byte aligned");
    if (n > 0 && !x) return fail(GDN_ERR_INVALID_ARG, "x is NULL");
    if (x && ((uintptr_t)x) % 16 != 0) return fail(GDN_ERR_INVALID_ARG, "x is not 16-byte aligned");
    if (n == 0) return GDN_OK;
    cudaStream_t cs = (cudaStream_t)stream;
    const gdn::InType ty = dtype == GDN_BF16 ? gdn::InType::BF16 : gdn::InType::F32;
    cudaError_t e = timed(gdn::KID_COUNT_NONFINITE, cs, [&] { return gdn::launch_count_nonfinite(x, n, ty, count, cs); });
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "non-finite count kernel");
}

gdn_status gdn_bwd(const gdn_problem* p, const void* q, const void* k, const void* v,
                   const void* alpha, const void* beta, const float* initial_state,
                   const void* saved, const void* d_o, const float* d_final_state,
                   void* dq, void* dk, void* dv, void* dalpha, void* dbeta,
                   float* d_initial_state, void* workspace, size_t workspace_bytes,
                   void* stream) {
    g_err[0] = 0;
    gdn::Dims d{};
    gdn_status st = check_problem(p, &d);
    if (st != GDN_OK) return st;
    const size_t es = p->dtype == GDN_BF16 ? 2 : 4;
    const size_t BTH = (size_t)d.B * d.T * d.H;
    const size_t nstate = (size_t)d.NS() * d.V * d.K * sizeof(float);
    const size_t need = gdn_bwd_workspace_bytes(p);
    const Span ins[] = {{q, BTH * d.K * es, "q"},
                        {k, BTH * d.K * es, "k"},
                        {v, BTH * d.V * es, "v"},
                        {alpha, BTH * es, "alpha"},
                        {beta, BTH * es, "beta"},
                        {initial_state, nstate, "initial_state"},
                        {saved, gdn_saved_bytes(p), "saved"},
                        {d_o, BTH * d.V * es, "d_o"},
                        {d_final_state, nstate, "d_final_state"}};
    const Span outs[] = {{dq, BTH * d.K * es, "dq"},
                         {dk, BTH * d.K * es, "dk"},
                         {dv, BTH * d.V * es, "dv"},
                         {dalpha, BTH * es, "dalpha"},
                         {dbeta, BTH * es, "dbeta"},
                         {d_initial_state, nstate, "d_initial_state"},
                         {workspace, need, "workspace"}};
    for (int i = 0; i < 9; ++i) {
        const bool req = !(i == 5 || i == 6 || i == 8);
        if ((st = check_ptr(ins[i], req)) != GDN_OK) return st;
    }
    for (int i = 0; i < 7; ++i)
        if ((st = check_ptr(outs[i], i != 5)) != GDN_OK) return st;
    if (workspace_bytes < need)
        return fail(GDN_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes,
                    need);
    if ((st = check_overlaps(ins, 9, outs, 7, d_initial_state, d_final_state)) != GDN_OK)
        return st;

    cudaStream_t cs = (cudaStream_t)stream;
    if (d.NS() == 0) return GDN_OK;
    if (d.T == 0) {  // empty sequence: d(initial state) = d(final state)
        cudaError_t e = cudaSuccess;
        if (d_initial_state && d_initial_state != d_final_state)
            e = d_final_state ? cudaMemcpyAsync(d_initial_state, d_final_state, nstate,
                                                cudaMemcpyDeviceToDevice, cs)
                              : cudaMemsetAsync(d_initial_state, 0, nstate, cs);
        return e == cudaSuccess ? GDN_OK : cuda_fail(e, "empty-sequence state copy");
    }
    const gdn::InType ty = p->dtype == GDN_BF16 ? gdn::InType::BF16 : gdn::InType::F32;
    if (gdn::tc_fwd_supported(d, ty)) {
        gdn::Dims fd;
        const SplitCfg sp = dense_split(d, &fd);
        return run_bwd_tc(fd, q, k, v, alpha, beta, initial_state, saved, d_o, d_final_state, dq, dk, dv, dalpha,
                          dbeta, d_initial_state, workspace, nullptr, &sp, cs);
    }
    Carver cv{(char*)workspace};
    gdn::ChunkBufs cb;
    gdn::BwdBufs bb;
    carve_bwd(d, cv, &cb, &bb, saved == nullptr);
    const float* states = saved ? (const float*)saved : bb.states;
    cudaError_t e = timed(gdn::KID_PREP_BWD, cs, [&] {
        return gdn::launch_prep(d, ty, k, q, v, alpha, beta, cb, true, cs);
    });
    if (e != cudaSuccess) return cuda_fail(e, "chunk kernel");
    if (!saved) {
        e = timed(gdn::KID_STATE_RECOMPUTE, cs, [&] {
            return gdn::launch_scan_fwd(d, ty, q, k, cb, initial_state, nullptr, nullptr,
                                        bb.states, false, cs);
        });
        if (e != cudaSuccess) return cuda_fail(e, "state recompute kernel");
    }
    e = timed(gdn::KID_SCAN_BWD, cs, [&] {
        return gdn::launch_scan_bwd(d, ty, q, k, d_o, cb, states, d_final_state, bb,
                                    d_initial_state, cs);
    });
    if (e != cudaSuccess) return cuda_fail(e, "reverse scan kernel");
    e = timed(gdn::KID_GRAD, cs, [&] {
        return gdn::launch_grad(d, ty, q, k, v, alpha, beta, d_o, cb, states, bb, dq, dk, dv,
                                dalpha, dbeta, cs);
    });
    if (e != cudaSuccess) return cuda_fail(e, "chunk gradient kernel");
    return GDN_OK;
}

// ------------------------------------------------ the recurrence with its prologue

}  // extern "C"

namespace {

// The normalised rows and reciprocal norms of the raw path on the tensor-core
// kernels (q, k bf16 [B,T,H,K]; 1/|q_raw|, 1/|k_raw| fp32 [B,T,H]).
size_t carve_raw(const gdn::Dims& d, Carver& cv, gdn::RawPrologue* rp) {
    const size_t BTH = (size_t)d.B * d.T * d.H;
    rp->on = 1;
    rp->qn = cv.take<__nv_bfloat16>(BTH * d.K);
    rp->kn = cv.take<__nv_bfloat16>(BTH * d.K);
    rp->rq = cv.take<float>(BTH);
    rp->rk = cv.take<float>(BTH);
    return cv.off;
}
// The backward's per-token kdot, in the workspace (after the raw buffers).
float* carve_kdot(const gdn::Dims& d, Carver& cv) { return cv.take<float>((size_t)d.NS() * d.NC * d.C); }

// The composed raw path (shapes outside the tensor-core kernels): the prologue's
// outputs and, for the backward, the gradients of the recurrence's inputs, all
// in the run dtype.
struct ComposedBufs {
    void *qn, *kn, *al, *be, *dqn, *dkn, *dal, *dbe;
};
size_t carve_composed(const gdn::Dims& d, size_t es, Carver& cv, ComposedBufs* c, bool bwd) {
    const size_t BTH = (size_t)d.B * d.T * d.H;
    *c = ComposedBufs{};
    c->qn = cv.take<char>(BTH * d.K * es);
    c->kn = cv.take<char>(BTH * d.K * es);
    c->al = cv.take<char>(BTH * es);
    c->be = cv.take<char>(BTH * es);
    if (bwd) {
        c->dqn = cv.take<char>(BTH * d.K * es);
        c->dkn = cv.take<char>(BTH * d.K * es);
        c->dal = cv.take<char>(BTH * es);
        c->dbe = cv.take<char>(BTH * es);
    }
    return cv.off;
}

// Bytes in front of the ordinary workspace in a raw call's workspace.
size_t raw_prefix(const gdn_problem* p, const gdn::Dims& d, bool bwd) {
    Carver cv{nullptr};
    if (gdn::tc_fwd_supported(d, in_type(p))) {
        gdn::RawPrologue rp;
        carve_raw(d, cv, &rp);
        if (bwd) carve_kdot(d, cv);
        return cv.off;
    }
    ComposedBufs c;
    return carve_composed(d, p->dtype == GDN_BF16 ? 2 : 4, cv, &c, bwd);
}

}  // namespace

extern "C" {

size_t gdn_raw_saved_bytes(const gdn_problem* p) {
    gdn::Dims d{};
    if (check_problem(p, &d) != GDN_OK) return 0;
    if (!gdn::tc_fwd_supported(d, in_type(p))) return gdn_saved_bytes(p);
    Carver cv{nullptr};
    gdn::RawPrologue rp;
    carve_raw(d, cv, &rp);
    return cv.off + gdn_saved_bytes(p);
}

size_t gdn_raw_fwd_workspace_bytes(const gdn_problem* p) {
    gdn::Dims d{};
    if (check_problem(p, &d) != GDN_OK || d.NS() * d.NC == 0) return 0;
    return raw_prefix(p, d, false) + gdn_fwd_workspace_bytes(p);
}

size_t gdn_raw_bwd_workspace_bytes(const gdn_problem* p) {
    gdn::Dims d{};
    if (check_problem(p, &d) != GDN_OK || d.NS() * d.NC == 0) return 0;
    return raw_prefix(p, d, true) + gdn_bwd_workspace_bytes(p);
}

gdn_status gdn_fwd_raw(const gdn_problem* p, const void* q_raw, const void* k_raw, const void* v,
                       const void* a_logit, const void* b_logit, const float* initial_state, void* o,
                       float* final_state, void* saved, void* workspace, size_t workspace_bytes, void* stream) {
    g_err[0] = 0;
    gdn::Dims d{};
    gdn_status st = check_problem(p, &d);
    if (st != GDN_OK) return st;
    if (d.NS() * d.NC == 0)  // nothing to normalise: the state passes through
        return gdn_fwd(p, q_raw, k_raw, v, a_logit, b_logit, initial_state, o, final_state, nullptr, nullptr, 0,
                       stream);
    const size_t es = p->dtype == GDN_BF16 ? 2 : 4;
    const size_t BTH = (size_t)d.B * d.T * d.H;
    const size_t nstate = (size_t)d.NS() * d.V * d.K * sizeof(float);
    const size_t need = gdn_raw_fwd_workspace_bytes(p);
    const Span ins[] = {{q_raw, BTH * d.K * es, "q_raw"},     {k_raw, BTH * d.K * es, "k_raw"},
                        {v, BTH * d.V * es, "v"},             {a_logit, BTH * es, "a_logit"},
                        {b_logit, BTH * es, "b_logit"},       {initial_state, nstate, "initial_state"}};
    const Span outs[] = {{o, BTH * d.V * es, "o"},
                         {final_state, nstate, "final_state"},
                         {saved, gdn_raw_saved_bytes(p), "saved"},
                         {workspace, need, "workspace"}};
    for (int i = 0; i < 6; ++i)
        if ((st = check_ptr(ins[i], i != 5)) != GDN_OK) return st;
    for (int i = 0; i < 4; ++i)
        if ((st = check_ptr(outs[i], i == 0 || i == 3)) != GDN_OK) return st;
    if (workspace_bytes < need)
        return fail(GDN_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
    if ((st = check_overlaps(ins, 6, outs, 4, final_state, initial_state)) != GDN_OK) return st;
    cudaStream_t cs = (cudaStream_t)stream;
    const gdn::InType ty = in_type(p);
    const size_t pre = raw_prefix(p, d, false);
    char* ws = (char*)workspace + pre;
    if (gdn::tc_fwd_supported(d, ty)) {
        gdn::RawPrologue rp;
        Carver cv{(char*)(saved ? saved : workspace)};
        carve_raw(d, cv, &rp);
        void* tc_saved = saved ? (char*)saved + cv.off : nullptr;
        gdn::Dims fd;
        const SplitCfg sp = dense_split(d, &fd);
        return run_fwd_tc(fd, q_raw, k_raw, v, a_logit, b_logit, initial_state, o, final_state, tc_saved, ws,
                          nullptr, &sp, cs, &rp);
    }
    // other shapes: the prologue kernel, then the recurrence on its outputs
    ComposedBufs c;
    Carver cv{(char*)workspace};
    carve_composed(d, es, cv, &c, false);
    cudaError_t e = timed(gdn::KID_PROLOGUE_FWD, cs, [&] {
        return gdn::launch_prologue_fwd(d, ty, q_raw, k_raw, a_logit, b_logit, c.qn, c.kn, c.al, c.be, cs);
    });
    if (e != cudaSuccess) return cuda_fail(e, "prologue kernel");
    return gdn_fwd(p, c.qn, c.kn, v, c.al, c.be, initial_state, o, final_state, saved, ws, workspace_bytes - pre,
                   stream);
}

gdn_status gdn_bwd_raw(const gdn_problem* p, const void* q_raw, const void* k_raw, const void* v,
                       const void* a_logit, const void* b_logit, const float* initial_state, const void* saved,
                       const void* d_o, const float* d_final_state, void* dq_raw, void* dk_raw, void* dv,
                       void* da_logit, void* db_logit, float* d_initial_state, void* workspace,
                       size_t workspace_bytes, void* stream) {
    g_err[0] = 0;
    gdn::Dims d{};
    gdn_status st = check_problem(p, &d);
    if (st != GDN_OK) return st;
    if (d.NS() * d.NC == 0)  // no tokens: d(initial state) = d(final state)
        return gdn_bwd(p, q_raw, k_raw, v, a_logit, b_logit, initial_state, nullptr, d_o, d_final_state, dq_raw,
                       dk_raw, dv, da_logit, db_logit, d_initial_state, nullptr, 0, stream);
    const size_t es = p->dtype == GDN_BF16 ? 2 : 4;
    const size_t BTH = (size_t)d.B * d.T * d.H;
    const size_t nstate = (size_t)d.NS() * d.V * d.K * sizeof(float);
    const size_t need = gdn_raw_bwd_workspace_bytes(p);
    const Span ins[] = {{q_raw, BTH * d.K * es, "q_raw"},
                        {k_raw, BTH * d.K * es, "k_raw"},
                        {v, BTH * d.V * es, "v"},
                        {a_logit, BTH * es, "a_logit"},
                        {b_logit, BTH * es, "b_logit"},
                        {initial_state, nstate, "initial_state"},
                        {saved, gdn_raw_saved_bytes(p), "saved"},
                        {d_o, BTH * d.V * es, "d_o"},
                        {d_final_state, nstate, "d_final_state"}};
    const Span outs[] = {{dq_raw, BTH * d.K * es, "dq_raw"},
                         {dk_raw, BTH * d.K * es, "dk_raw"},
                         {dv, BTH * d.V * es, "dv"},
                         {da_logit, BTH * es, "da_logit"},
                         {db_logit, BTH * es, "db_logit"},
                         {d_initial_state, nstate, "d_initial_state"},
                         {workspace, need, "workspace"}};
    for (int i = 0; i < 9; ++i)
        if ((st = check_ptr(ins[i], !(i == 5 || i == 6 || i == 8))) != GDN_OK) return st;
    for (int i = 0; i < 7; ++i)
        if ((st = check_ptr(outs[i], i != 5)) != GDN_OK) return st;
    if (workspace_bytes < need)
        return fail(GDN_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
    if ((st = check_overlaps(ins, 9, outs, 7, d_initial_state, d_final_state)) != GDN_OK) return st;
    cudaStream_t cs = (cudaStream_t)stream;
    const gdn::InType ty = in_type(p);
    const size_t pre = raw_prefix(p, d, true);
    char* ws = (char*)workspace + pre;
    if (gdn::tc_fwd_supported(d, ty)) {
        gdn::RawPrologue rp;
        Carver cv{(char*)(saved ? const_cast<void*>(saved) : workspace)};
        carve_raw(d, cv, &rp);
        const void* tc_saved = saved ? (const char*)saved + cv.off : nullptr;
        Carver kv{(char*)workspace};  // kdot after the workspace's own raw buffers
        gdn::RawPrologue unused;
        carve_raw(d, kv, &unused);
        rp.kdot = carve_kdot(d, kv);
        gdn::Dims fd;
        const SplitCfg sp = dense_split(d, &fd);
        return run_bwd_tc(fd, q_raw, k_raw, v, a_logit, b_logit, initial_state, tc_saved, d_o, d_final_state,
                          dq_raw, dk_raw, dv, da_logit, db_logit, d_initial_state, ws, nullptr, &sp, cs, &rp);
    }
    // other shapes: the prologue again, the recurrence's backward, then the prologue's
    ComposedBufs c;
    Carver cv{(char*)workspace};
    carve_composed(d, es, cv, &c, true);
    cudaError_t e = timed(gdn::KID_PROLOGUE_FWD, cs, [&] {
        return gdn::launch_prologue_fwd(d, ty, q_raw, k_raw, a_logit, b_logit, c.qn, c.kn, c.al, c.be, cs);
    });
    if (e != cudaSuccess) return cuda_fail(e, "prologue kernel");
    st = gdn_bwd(p, c.qn, c.kn, v, c.al, c.be, initial_state, saved, d_o, d_final_state, c.dqn, c.dkn, dv, c.dal,
                 c.dbe, d_initial_state, ws, workspace_bytes - pre, stream);
    if (st != GDN_OK) return st;
    e = timed(gdn::KID_PROLOGUE_BWD, cs, [&] {
        return gdn::launch_prologue_bwd(d, ty, q_raw, k_raw, a_logit, b_logit, c.dqn, c.dkn, c.dal, c.dbe, dq_raw,
                                        dk_raw, da_logit, db_logit, cs);
    });
    if (e != cudaSuccess) return cuda_fail(e, "prologue backward kernel");
    return GDN_OK;
}

// ------------------------------------------------------------------ reset masks

}  // extern "C"

namespace {

// The reset calls run gdn_varlen_* on the dense tensors (a packed batch of S_max
// sequences over the B*T tokens); their own buffers follow the varlen workspace,
// so the varlen error word stays the first int of the caller's workspace.
struct ResetBufs {
    int32_t *cu, *in_map, *fin_map, *last, *first_carry;
    int* err;
    float *s_in, *s_out;  // per-segment initial / final states or state gradients
};
size_t carve_reset(const gdn::Dims& d, int64_t S_max, Carver& cv, ResetBufs* r) {
    r->cu = cv.take<int32_t>((size_t)S_max + 1);
    r->in_map = cv.take<int32_t>((size_t)S_max);
    r->fin_map = cv.take<int32_t>((size_t)S_max);
    r->last = cv.take<int32_t>((size_t)d.B);
    r->first_carry = cv.take<int32_t>((size_t)d.B);
    r->err = cv.take<int>(1);
    const size_t st = (size_t)S_max * d.H * d.V * d.K;
    r->s_in = cv.take<float>(st);
    r->s_out = cv.take<float>(st);
    return cv.off;
}

// The packed problem the reset calls run: S_max sequences of at most T tokens.
gdn_status reset_problem(const gdn_problem* p, int64_t S_max, gdn_problem* pv, gdn::Dims* d) {
    gdn_status st = check_problem(p, d);
    if (st != GDN_OK) return st;
    if (d->B > 0 && d->T > 0 && (S_max < d->B || S_max > (int64_t)d->B * d->T))
        return fail(GDN_ERR_INVALID_ARG, "max_segments=%lld must be in [B, B*T] = [%d, %lld]", (long long)S_max,
                    d->B, (long long)d->B * d->T);
    if (S_max > 65535) return fail(GDN_ERR_UNSUPPORTED, "max_segments=%lld exceeds 65535", (long long)S_max);
    *pv = *p;
    pv->B = S_max;
    return GDN_OK;
}

}  // namespace

extern "C" {

size_t gdn_reset_saved_bytes(const gdn_problem* p, int64_t max_segments) {
    gdn_problem pv;
    gdn::Dims d{};
    if (reset_problem(p, max_segments, &pv, &d) != GDN_OK) return 0;
    return gdn_varlen_saved_bytes(&pv, (int64_t)d.B * d.T);
}

static size_t reset_ws_bytes(const gdn_problem* p, int64_t max_segments, bool bwd) {
    gdn_problem pv;
    gdn::Dims d{};
    if (reset_problem(p, max_segments, &pv, &d) != GDN_OK || d.NS() * d.NC == 0) return 0;
    const int64_t total = (int64_t)d.B * d.T;
    const size_t inner =
        round_up(bwd ? gdn_varlen_bwd_workspace_bytes(&pv, total) : gdn_varlen_fwd_workspace_bytes(&pv, total));
    Carver cv{nullptr};
    ResetBufs r;
    return inner + carve_reset(d, max_segments, cv, &r);
}

size_t gdn_reset_fwd_workspace_bytes(const gdn_problem* p, int64_t max_segments) {
    return reset_ws_bytes(p, max_segments, false);
}

size_t gdn_reset_bwd_workspace_bytes(const gdn_problem* p, int64_t max_segments) {
    return reset_ws_bytes(p, max_segments, true);
}

gdn_status gdn_reset_fwd(const gdn_problem* p, int64_t max_segments, const uint8_t* reset, const void* q,
                         const void* k, const void* v, const void* alpha, const void* beta,
                         const float* initial_state, void* o, float* final_state, void* saved, void* workspace,
                         size_t workspace_bytes, void* stream) {
    g_err[0] = 0;
    gdn_problem pv;
    gdn::Dims d{};
    gdn_status st = reset_problem(p, max_segments, &pv, &d);
    if (st != GDN_OK) return st;
    if (d.NS() * d.NC == 0)  // no tokens: the state passes through, the mask is not read
        return gdn_fwd(p, q, k, v, alpha, beta, initial_state, o, final_state, nullptr, nullptr, 0, stream);
    const int64_t total = (int64_t)d.B * d.T;
    const size_t es = p->dtype == GDN_BF16 ? 2 : 4;
    const size_t BTH = (size_t)total * d.H;
    const size_t nstate = (size_t)d.NS() * d.V * d.K * sizeof(float);
    const size_t need = gdn_reset_fwd_workspace_bytes(p, max_segments);
    // every argument is checked here, before the first launch (the packed call checks again)
    const Span ins[] = {{q, BTH * d.K * es, "q"},       {k, BTH * d.K * es, "k"},
                        {v, BTH * d.V * es, "v"},       {alpha, BTH * es, "alpha"},
                        {beta, BTH * es, "beta"},       {initial_state, nstate, "initial_state"},
                        {reset, (size_t)total, "reset"}};
    const Span outs[] = {{o, BTH * d.V * es, "o"},
                         {final_state, nstate, "final_state"},
                         {saved, gdn_reset_saved_bytes(p, max_segments), "saved"},
                         {workspace, need, "workspace"}};
    if (!reset) return fail(GDN_ERR_INVALID_ARG, "reset is NULL");
    for (int i = 0; i < 6; ++i)
        if ((st = check_ptr(ins[i], i != 5)) != GDN_OK) return st;
    for (int i = 0; i < 4; ++i)
        if ((st = check_ptr(outs[i], i == 0 || i == 3)) != GDN_OK) return st;
    if (workspace_bytes < need)
        return fail(GDN_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
    if ((st = check_overlaps(ins, 7, outs, 4, final_state, initial_state)) != GDN_OK) return st;
    cudaStream_t cs = (cudaStream_t)stream;
    const size_t inner = round_up(gdn_varlen_fwd_workspace_bytes(&pv, total));
    Carver cv{(char*)workspace + inner};
    ResetBufs r;
    carve_reset(d, max_segments, cv, &r);
    const int64_t row = (int64_t)d.H * d.V * d.K;
    cudaError_t e = gdn::launch_reset_segments(d.B, d.T, reset, (int)max_segments, r.cu, r.in_map, r.fin_map, r.last,
                                               r.first_carry, r.err, cs);
    if (e == cudaSuccess)  // each row's initial state into its first segment (unless reset at t = 0)
        e = gdn::launch_route_states((int)max_segments, row, r.in_map, initial_state, r.s_in, nullptr, nullptr, cs);
    if (e != cudaSuccess) return cuda_fail(e, "reset segments");
    st = gdn_varlen_fwd(&pv, total, r.cu, q, k, v, alpha, beta, r.s_in, o, r.s_out, saved, workspace, inner,
                        stream);
    if (st != GDN_OK) return st;
    // each row's final state from its last segment; the segment error joins the varlen word
    e = gdn::launch_route_states(final_state ? d.B : 0, row, r.last, r.s_out, final_state, r.err, (int*)workspace,
                                 cs);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "reset state routing");
}

gdn_status gdn_reset_bwd(const gdn_problem* p, int64_t max_segments, const uint8_t* reset, const void* q,
                         const void* k, const void* v, const void* alpha, const void* beta,
                         const float* initial_state, const void* saved, const void* d_o, const float* d_final_state,
                         void* dq, void* dk, void* dv, void* dalpha, void* dbeta, float* d_initial_state,
                         void* workspace, size_t workspace_bytes, void* stream) {
    g_err[0] = 0;
    gdn_problem pv;
    gdn::Dims d{};
    gdn_status st = reset_problem(p, max_segments, &pv, &d);
    if (st != GDN_OK) return st;
    if (d.NS() * d.NC == 0)
        return gdn_bwd(p, q, k, v, alpha, beta, initial_state, nullptr, d_o, d_final_state, dq, dk, dv, dalpha,
                       dbeta, d_initial_state, nullptr, 0, stream);
    const int64_t total = (int64_t)d.B * d.T;
    const size_t es = p->dtype == GDN_BF16 ? 2 : 4;
    const size_t BTH = (size_t)total * d.H;
    const size_t nstate = (size_t)d.NS() * d.V * d.K * sizeof(float);
    const size_t need = gdn_reset_bwd_workspace_bytes(p, max_segments);
    // every argument is checked here, before the first launch (the packed call checks again)
    const Span ins[] = {{q, BTH * d.K * es, "q"},
                        {k, BTH * d.K * es, "k"},
                        {v, BTH * d.V * es, "v"},
                        {alpha, BTH * es, "alpha"},
                        {beta, BTH * es, "beta"},
                        {initial_state, nstate, "initial_state"},
                        {saved, gdn_reset_saved_bytes(p, max_segments), "saved"},
                        {d_o, BTH * d.V * es, "d_o"},
                        {d_final_state, nstate, "d_final_state"},
                        {reset, (size_t)total, "reset"}};
    const Span outs[] = {{dq, BTH * d.K * es, "dq"},
                         {dk, BTH * d.K * es, "dk"},
                         {dv, BTH * d.V * es, "dv"},
                         {dalpha, BTH * es, "dalpha"},
                         {dbeta, BTH * es, "dbeta"},
                         {d_initial_state, nstate, "d_initial_state"},
                         {workspace, need, "workspace"}};
    if (!reset) return fail(GDN_ERR_INVALID_ARG, "reset is NULL");
    for (int i = 0; i < 9; ++i)
        if ((st = check_ptr(ins[i], !(i == 5 || i == 6 || i == 8))) != GDN_OK) return st;
    for (int i = 0; i < 7; ++i)
        if ((st = check_ptr(outs[i], i != 5)) != GDN_OK) return st;
    if (workspace_bytes < need)
        return fail(GDN_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
    if ((st = check_overlaps(ins, 10, outs, 7, d_initial_state, d_final_state)) != GDN_OK) return st;
    cudaStream_t cs = (cudaStream_t)stream;
    const size_t inner = round_up(gdn_varlen_bwd_workspace_bytes(&pv, total));
    Carver cv{(char*)workspace + inner};
    ResetBufs r;
    carve_reset(d, max_segments, cv, &r);
    const int64_t row = (int64_t)d.H * d.V * d.K;
    float* s_init = r.s_in;    // the segments' initial states
    float* g_fin = r.s_out;    // the segments' final-state gradients, then their initial-state gradients
    cudaError_t e = gdn::launch_reset_segments(d.B, d.T, reset, (int)max_segments, r.cu, r.in_map, r.fin_map, r.last,
                                               r.first_carry, r.err, cs);
    if (e == cudaSuccess)
        e = gdn::launch_route_states((int)max_segments, row, r.in_map, initial_state, s_init, nullptr, nullptr, cs);
    if (e == cudaSuccess)  // each row's final-state gradient into its last segment
        e = gdn::launch_route_states((int)max_segments, row, r.fin_map, d_final_state, g_fin, nullptr, nullptr, cs);
    if (e != cudaSuccess) return cuda_fail(e, "reset segments");
    // in place: d(initial state) of every segment over its d(final state)
    st = gdn_varlen_bwd(&pv, total, r.cu, q, k, v, alpha, beta, s_init, saved, d_o, g_fin, dq, dk, dv, dalpha,
                        dbeta, g_fin, workspace, inner, stream);
    if (st != GDN_OK) return st;
    // a row's d(initial state) from its first segment; zero if the row resets at t = 0
    e = gdn::launch_route_states(d_initial_state ? d.B : 0, row, r.first_carry, g_fin, d_initial_state, r.err,
                                 (int*)workspace, cs);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "reset state routing");
}

gdn_status gdn_set_sequence_split(int pieces) {
    if (pieces < 0 || pieces > 1024) return fail(GDN_ERR_INVALID_ARG, "pieces=%d must be in [0, 1024]", pieces);
    g_split = pieces;
    return GDN_OK;
}

int gdn_get_sequence_split(void) { return g_split; }

int gdn_num_kernels(void) { return gdn::KID_COUNT; }

const char* gdn_kernel_name(int id) {
    return (id >= 0 && id < gdn::KID_COUNT) ? kKernelNames[id] : "";
}

gdn_status gdn_profiler_start(int capacity) {
    if (capacity < 0) return fail(GDN_ERR_INVALID_ARG, "negative profiler capacity");
    if ((int)g_prof.kid.size() < capacity) {
        const size_t have = g_prof.ev.size();
        g_prof.ev.resize(2 * (size_t)capacity);
        for (size_t i = have; i < g_prof.ev.size(); ++i) {
            cudaError_t e = cudaEventCreate(&g_prof.ev[i]);
            if (e != cudaSuccess) {
                g_prof.ev.resize(i);
                g_prof.kid.resize(i / 2);
                return cuda_fail(e, "cudaEventCreate");
            }
        }
        g_prof.kid.resize(capacity);
    }
    g_prof.n = 0;
    g_prof.on = true;
    return GDN_OK;
}

gdn_status gdn_profiler_stop(void) {
    g_prof.on = false;
    return GDN_OK;
}

gdn_status gdn_profiler_summary(int id, int* launches, double* total_ms) {
    if (!launches || !total_ms) return fail(GDN_ERR_INVALID_ARG, "NULL output pointer");
    *launches = 0;
    *total_ms = 0.0;
    for (int i = 0; i < g_prof.n; ++i) {
        if (g_prof.kid[i] != id) continue;
        cudaError_t e = cudaEventSynchronize(g_prof.ev[2 * i + 1]);
        float ms = 0.f;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]);
        if (e != cudaSuccess) return cuda_fail(e, "profiler event");
        *launches += 1;
        *total_ms += ms;
    }
    return GDN_OK;
}

void gdn_profiler_release(void) {
    for (cudaEvent_t e : g_prof.ev) cudaEventDestroy(e);
    g_prof = Profiler();
}

}  // extern "C"
