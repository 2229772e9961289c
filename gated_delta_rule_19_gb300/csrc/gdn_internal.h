// gdn_internal.h -- shapes, workspace layout and kernel launchers shared by the
// translation units of libgdn.so (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdn {

// Problem dimensions as the kernels see them.  NC = ceil(T / C) chunks per
// (b, h) stream; NS = B * H streams.  All index arithmetic that can exceed 2^31
// is done in int64.
struct Dims {
    int B, T, H, K, V, C, NC;
    // A packed batch read in place (B = 1, T = the packed token count, one row of
    // chunks per head): chunk c of the row starts at packed token tok[c] and has
    // len[c] <= C tokens of its sequence (device arrays of NC ints).  NULL for
    // dense tensors, where chunk c starts at c * C.
    const int* tok = nullptr;
    const int* len = nullptr;
    // Limit of the tensor-core kernels' bounded waits in nanoseconds (0: the default
    // of 2 s); set by the test hook gdn_test_set_wait_limit.
    uint32_t wait_ns = 0;
    __host__ __device__ int64_t NS() const { return (int64_t)B * H; }
    // The chunk (index (b * H + h) * NC + c) that work item wi of a chunk-parallel
    // kernel takes: every stream's chunk c before any chunk c + 1, c ascending or
    // descending, so that the next kernel meets first the chunks written last
    // (still in L2).  NS() * NC for wi past the end.
    __host__ __device__ int64_t chunk_of(int64_t wi, bool descending) const {
        const int64_t n = NS() * NC;
        if (wi >= n) return n;
        int64_t c = wi / NS();
        if (descending) c = NC - 1 - c;
        return (wi % NS()) * NC + c;
    }
};

// First token of chunk c within its batch row, and its number of tokens, for
// kernels compiled for dense tensors (kPacked false: tok, len unused) or for a
// packed batch read in place (kPacked true).
template <bool kPacked>
__device__ __forceinline__ int chunk_tok(const Dims& d, int c) {
    if constexpr (kPacked) return d.tok[c];
    else return c * d.C;
}
template <bool kPacked>
__device__ __forceinline__ int chunk_valid(const Dims& d, int c) {
    if constexpr (kPacked) return d.len[c];
    else return d.T - c * d.C < d.C ? d.T - c * d.C : d.C;
}

// Per-chunk results of the chunk-parallel step (Phase 1 + solve + recompute),
// float32, indexed [stream][chunk][...]:
//   G   [C]     within-chunk cumulative log alpha
//   W   [C,K]   T diag(beta*gamma) K
//   Ut  [C,V]   T diag(beta) V
//   Mqk [C,C]   lower(Gamma .* Q K^T)
//   Tm  [C,C]   (I + A)^-1   (backward only)
struct ChunkBufs {
    float* G;
    float* W;
    float* Ut;
    float* Mqk;
    float* Tm;
};

// Backward-only buffers, float32:
//   states [NS,NC,V,K] chunk-start states (when the caller passed no `saved`)
//   U, dU  [NS,NC,C,V] corrected writes and their gradient
//   dS1    [NS,NC,V,K] gradient of each chunk's end state
//   dW, dQ1, dKh [NS,NC,C,K] chunk-local gradient scratch
struct BwdBufs {
    float* states;
    float* U;
    float* dU;
    float* dS1;
    float* dW;
    float* dQ1;
    float* dKh;
};

enum class InType { F32 = 0, BF16 = 1 };

// Chunk results of the tensor-core forward (bf16 inputs, chunk 64, K and V of 16
// to 128), rows indexed chunk * 64 + r with chunk = stream * NC + c:
//   W [rows, 128], Ut [rows, 128], Mqk [rows, 64] (bf16; columns past K or V hold
//   zeros); G [rows] (fp32).
// err: an int the kernels set (bitwise) when a bounded wait gives up.
//   T [rows, 64] (bf16, (I + A)^-1; written only when non-null, for the backward).
struct TcBufs {
    __nv_bfloat16* W;
    __nv_bfloat16* Ut;
    __nv_bfloat16* Mqk;
    float* G;
    __nv_bfloat16* T;
    int* err;
};

// Backward buffers of the tensor-core path:
//   dU   [rows, V] bf16            gradient of the corrected writes U
//   dS1  [chunks * K, V] bf16      gradient of each chunk's end state, transposed
//   dKp  [chunks * K, 64] bf16     dK^T from the Mqk and state-update terms
//   dWt  [chunks * K, 64] bf16     dW^T
//   dGp  [rows] fp32               dG from the output, Mqk and state-update terms
//   states [chunks * K, V] bf16    chunk-start states when no saved buffer is given
struct TcBwdBufs {
    __nv_bfloat16* dU;
    __nv_bfloat16* dS1;
    __nv_bfloat16* dKp;
    __nv_bfloat16* dWt;
    float* dGp;
    __nv_bfloat16* states;
};

// Kernel identities for the optional launch timer (gdn_profiler_*).  The names
// are the CUDA kernel names, so they match the entries of an ncu launch list.
enum KernelId {
    KID_PREP_FWD = 0,    // prep_kernel, forward
    KID_SCAN_FWD,        // scan_fwd_kernel
    KID_PREP_BWD,        // prep_kernel, backward (also writes T)
    KID_STATE_RECOMPUTE, // scan_fwd_kernel in state-only mode (backward without saved)
    KID_SCAN_BWD,        // scan_bwd_kernel
    KID_GRAD,            // grad_kernel
    KID_PREP_TC,         // prep_fwd_tc
    KID_SCAN_FWD_TC,     // scan_fwd_tc
    KID_PREP_TC_BWD,     // prep_fwd_tc, backward recompute (also writes T)
    KID_STATE_TC,        // scan_fwd_tc in state-only mode
    KID_SCAN_BWD_TC,     // scan_bwd_tc
    KID_GRAD_QK_TC,      // grad_qk_tc
    KID_GRAD_WY_TC,      // grad_wy_tc
    KID_DECODE,          // decode_kernel
    KID_PROLOGUE_FWD,    // prologue_fwd_kernel
    KID_PROLOGUE_BWD,    // prologue_bwd_kernel
    KID_VARLEN_OFFSETS,  // offsets_kernel, chunk_tokens_kernel (chunk offsets and token map)
    KID_VARLEN_GATHER,   // rows16_kernel / elems_kernel, packed -> padded layout
    KID_VARLEN_SCATTER,  // the same, padded layout -> packed
    KID_SPLIT_FWD_P1,    // scan_fwd_tc, split pass 1 (zero-start states and transitions of the pieces)
    KID_SPLIT_BWD_P1,    // scan_bwd_tc, split pass 1 (zero-start state gradients of the pieces)
    KID_SPLIT_TRANS,     // scan_fwd_tc, transitions only (backward with saved)
    KID_SPLIT_COMBINE,   // pieces_kernel, combine_fwd_kernel, combine_bwd_kernel
    KID_COUNT_NONFINITE, // count_nonfinite_kernel
    KID_COUNT
};

// Sets the message gdn_last_error() returns on the calling thread.
void set_last_error(const char* msg);

// Launchers of the SIMT (CUDA-core, float32) kernels.  Each returns the
// cudaError_t of its launch.
cudaError_t launch_prep(const Dims& d, InType ty, const void* k, const void* q,
                        const void* v, const void* alpha, const void* beta,
                        const ChunkBufs& cb, bool write_T, cudaStream_t st);
cudaError_t launch_scan_fwd(const Dims& d, InType ty, const void* q, const void* k,
                            const ChunkBufs& cb, const float* s0, void* o, float* sT,
                            float* states, bool write_o, cudaStream_t st);
cudaError_t launch_scan_bwd(const Dims& d, InType ty, const void* q, const void* k,
                            const void* d_o, const ChunkBufs& cb, const float* states,
                            const float* dsT, const BwdBufs& bb, float* ds0,
                            cudaStream_t st);
cudaError_t launch_grad(const Dims& d, InType ty, const void* q, const void* k,
                        const void* v, const void* alpha, const void* beta,
                        const void* d_o, const ChunkBufs& cb, const float* states,
                        const BwdBufs& bb, void* dq, void* dk, void* dv, void* dalpha,
                        void* dbeta, cudaStream_t st);

// Host helpers of the tensor-core path (tmap.cu).
// [B, T, H, D] bf16 -> 4D TMA map (D, H, T, B), box 64 x 1 x 64 x 1, 128B swizzle.
bool tmap_bthd(CUtensorMap* m, const void* ptr, int B, int T, int H, int D);
// [rows, cols] bf16 row-major -> 2D TMA map, box 64 x 64, 128B swizzle.
bool tmap_rows(CUtensorMap* m, const void* ptr, int64_t rows, int cols);
// [rows, cols] bf16 as 3D (8, rows, cols/8); box (8, box_rows, box_groups), no swizzle:
// lands as the MN-major no-swizzle operand layout [group][row][8].
bool tmap_core8_rows(CUtensorMap* m, const void* ptr, int64_t rows, int cols, int box_rows,
                     int box_groups);
// [B, T, H, D] bf16 as 5D (8, T, D/8, H, B); box (8, 64, box_groups, 1, 1), no swizzle.
bool tmap_core8_bthd(CUtensorMap* m, const void* ptr, int B, int T, int H, int D, int box_groups);
bool tma_available();
int sm_count();

// Tensor-core forward (tc_fwd.cu).  tc_fwd_supported: shape/dtype test only.
bool tc_fwd_supported(const Dims& d, InType ty);
// Packed sequences on the flat chunk layout (B = 1; every sequence starts a new
// chunk): sequence s owns chunks chunk_off[s] .. chunk_off[s+1]-1 of each head's
// row of chunks and state slot s*H + h.  The scans take it to run one stream per
// (sequence, head); the chunk-parallel kernels need nothing (their work is local
// to a chunk).
// The forward scan can also run the transition of a run of chunks: from S0 = I
// with U~ read as 0 its final state is the product of the chunks' maps (the
// within-call sequence split).  mode 0: the sequences only; 1: the sequences
// (CTAs z < nseq) and their transitions (z >= nseq, final states to `trans`);
// 2: the transitions only.
// tok / len of Dims for the flat layout of a packed batch (one block per chunk
// row entry; entries past the sequences get len 0).
cudaError_t launch_varlen_chunk_tokens(int S, int64_t total, int C, int nc_max, const int32_t* cu,
                                       const int* chunk_off, int* tok, int* len, cudaStream_t st);

struct SeqMap {
    const int* chunk_off;  // device, int32 [nseq + 1]
    int nseq;
    int mode = 0;
    float* trans = nullptr;  // [nseq * H, K, K] fp32, slot s*H + h
    // device int32 [nseq], or NULL: the sequence that grid row z runs (longest
    // first, so that the longest chains start in the first wave); mode 0 only
    const int* order = nullptr;
    // chunks of the longest sequence, or 0 if not known (mode 0 only)
    int max_nc = 0;
};
int tc_scan_vt(int64_t streams);
// The slice width for a scan over dims d with sequence map sq (or NULL) and
// `streams` CTA rows of one slice each.
int tc_scan_vt_for(const Dims& d, const SeqMap* sq, int64_t streams);

// Within-call sequence split (split.cu): piece offsets, and the chains of the
// pieces' affine maps forward (states) and backward (state gradients).
cudaError_t launch_split_pieces(int S, int P, int nc, const int* chunk_off, int* piece_off, cudaStream_t st);
cudaError_t launch_combine_fwd(int S, int P, int H, const float* s0, const float* R, const float* trans, float* s_in,
                               float* sT, cudaStream_t st);
cudaError_t launch_combine_bwd(int S, int P, int H, const float* dsT, const float* D, const float* trans,
                               float* ds_out, float* ds0, cudaStream_t st);
// Packed variable-length batches (varlen.cu): rows of packed [total, H, width]
// tensors to and from the padded [S, T, H, width] layout.  `merge` (optional) is
// ORed into `err` once.
constexpr int kVarlenBadOffsets = 1 << 30;  // error-word bit: invalid cu_seqlens
constexpr int kResetTooManySegments = 1 << 29;  // error-word bit: more segments than max_segments
// Reset masks (reset.cu): the segments of a dense [B, T] batch whose streams
// restart at every set mask entry, and the routing of states between rows and
// segments (see gdn_reset_fwd in include/gdn.h).
cudaError_t launch_reset_segments(int B, int T, const uint8_t* reset, int S_max, int32_t* cu, int32_t* in_map,
                                  int32_t* fin_map, int32_t* last, int32_t* first_carry, int* err,
                                  cudaStream_t st);
// out[r] = src[map[r]] for nrows rows of `row` floats (zeros where map < 0 or src
// is NULL); ORs *merge_from into *merge_to first when both are given.
cudaError_t launch_route_states(int nrows, int64_t row, const int32_t* map, const float* src, float* out,
                                const int* merge_from, int* merge_to, cudaStream_t st);
// Work counters of the persistent kernels, in the error-flag area of the workspace
// (64 ints, the first 32 reset at the start of every call): chunks handed out
// beyond each CTA's first one.
constexpr int kSchedQk = 17, kSchedWy = 18, kErrWords = 32;
cudaError_t launch_varlen_rows(const Dims& d, int64_t total, const int32_t* cu, int width_bytes, const void* src,
                               void* dst, uint32_t fill, bool scatter, int* err, const int* merge, cudaStream_t st);
cudaError_t launch_varlen_elems(const Dims& d, int64_t total, const int32_t* cu, int elem_bytes, const void* src,
                                void* dst, uint32_t fill, bool scatter, int* err, cudaStream_t st);
// The flat chunk layout (SeqMap): chunk_off from cu (one block; lengths above
// max_len or invalid pairs count as empty and set the error bit; the offsets
// never pass nc_max) and, when `order` is not NULL, the sequences by chunk count,
// longest first (0 .. S-1 above 1024 sequences).
cudaError_t launch_varlen_offsets(int S, int64_t total, int max_len, int C, int nc_max, const int32_t* cu,
                                  int* chunk_off, int* order, int* err, cudaStream_t st);

// q/k L2 normalisation and gate activations, and their backward (prologue.cu).
cudaError_t launch_prologue_fwd(const Dims& d, InType ty, const void* qr, const void* kr, const void* a,
                                const void* b, void* q, void* k, void* alpha, void* beta, cudaStream_t st);
cudaError_t launch_prologue_bwd(const Dims& d, InType ty, const void* qr, const void* kr, const void* a,
                                const void* b, const void* dq, const void* dk, const void* dalpha, const void* dbeta,
                                void* dqr, void* dkr, void* da, void* db, cudaStream_t st);

// Recurrent step over the call's tokens, state [B,H,V,K] fp32 updated in place
// (decode.cu).
// Adds to *count (device) the number of NaN / inf elements of x[0 .. n-1] (check.cu).
cudaError_t launch_count_nonfinite(const void* x, int64_t n, InType ty, int64_t* count, cudaStream_t st);
cudaError_t launch_decode(const Dims& d, InType ty, const void* q, const void* k, const void* v,
                          const void* alpha, const void* beta, float* state, void* o, cudaStream_t st);

// The prologue in front of the recurrence, folded into the tensor-core kernels
// (gdn_fwd_raw / gdn_bwd_raw): with `on`, q and k are the raw rows and alpha,
// beta the gate logits a, b.  prep_fwd_tc normalises the q, k rows as they land
// (x / sqrt(sum x^2 + 1e-6)), writes them to qn, kn ([B,T,H,K] bf16) and the
// reciprocal norms to rq, rk ([B,T,H] fp32), and takes log alpha = -softplus(a),
// beta = sigmoid(b); the backward turns the gradients of the normalised rows and
// gates into those of the raw inputs.
//   kdot [rows] fp32: per token, k . (the dK part grad_qk_tc hands to grad_wy_tc),
//        which grad_wy_tc needs for the chain rule through the k normalisation.
struct RawPrologue {
    int on = 0;
    __nv_bfloat16* qn = nullptr;
    __nv_bfloat16* kn = nullptr;
    float* rq = nullptr;
    float* rk = nullptr;
    float* kdot = nullptr;
};

cudaError_t launch_prep_tc(const Dims& d, const void* q, const void* k, const void* v,
                           const void* alpha, const void* beta, const TcBufs& tb,
                           cudaStream_t st, const RawPrologue* raw = nullptr);
cudaError_t launch_scan_fwd_tc(const Dims& d, const void* q, const void* k, const TcBufs& tb,
                               const float* s0, void* o, float* sT, __nv_bfloat16* states,
                               cudaStream_t st, const SeqMap* sq = nullptr);
// Tensor-core backward (tc_bwd.cu).
cudaError_t launch_scan_bwd_tc(const Dims& d, const void* q, const void* k, const void* d_o,
                               const TcBufs& tb, const float* dsT, const TcBwdBufs& bb,
                               float* ds0, cudaStream_t st, const SeqMap* sq = nullptr);
cudaError_t launch_grad_qk_tc(const Dims& d, const void* q, const void* k, const void* d_o,
                              const TcBufs& tb, const __nv_bfloat16* states,
                              const TcBwdBufs& bb, void* dq, cudaStream_t st,
                              const RawPrologue* raw = nullptr);
cudaError_t launch_grad_wy_tc(const Dims& d, const void* k, const void* v, const void* alpha,
                              const void* beta, const TcBufs& tb, const TcBwdBufs& bb,
                              void* dk, void* dv, void* dalpha, void* dbeta, cudaStream_t st,
                              const RawPrologue* raw = nullptr);

}  // namespace gdn
