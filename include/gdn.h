/*
 * gdn.h -- C ABI of the GB300 chunkwise gated delta rule library (libgdn.so).
 *
 * The operation ("Sparse Delta Memory: layer and kernels", "What the layer
 * computes" and its dense-limit paragraph; "OpenGDN", "Core operator reference"):
 *
 *     S_t = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t = S_t q_t                      (read after the write, no scale on q)
 *
 * per (batch b, head h) stream, computed chunkwise with the extended-WY
 * decomposition: per chunk of `chunk` tokens the decay-weighted Gram matrices,
 * the solve T = (I + strict_lower(diag(beta) (Gamma .* K K^T)))^-1, the
 * recompute W = T diag(beta gamma) K and U~ = T diag(beta) V, then a sequential
 * scan over chunks that keeps the state on chip ("Sparse Delta Memory", "What
 * the layer computes": Phase 1, Solve, Phase 2; "OpenGDN", "Core operator
 * reference": the 64-token extended-WY chunk form with FP32 state).
 *
 * Layouts (all dense, row-major, no strides):
 *   q, k            [B, T, H, K]   dtype
 *   v, o            [B, T, H, V]   dtype
 *   alpha, beta     [B, T, H]      dtype   (linear gates; precondition 0 < alpha <= 1)
 *   states          [B, H, V, K]   float32 (initial/final state and their gradients)
 *   gradients       same shape and dtype as the input they belong to
 * dtype is GDN_F32 or GDN_BF16 (bf16 results are rounded to nearest even); every
 * accumulation, the gates, the solve and the state are float32 in both cases.
 *
 * Ownership and execution: the caller owns every buffer (device memory).  The
 * library allocates nothing, never synchronises, and enqueues all work on
 * `stream` (a cudaStream_t passed as void*; NULL is the legacy default stream).
 * Results are ready when the stream reaches that point.
 *
 * Errors: every argument check happens on the host before any launch and returns
 * a status (nothing is enqueued then); gdn_last_error() gives a message for the
 * last failure on the calling thread.  GDN_ERR_CUDA reports a failed launch.
 *
 * Requirements: B, H >= 0, T >= 0; K, V in {16, 32, 64, 128}; chunk in
 * {16, 32, 64}; every pointer 16-byte aligned; outputs must not overlap inputs
 * or each other.  Size limits (GDN_ERR_UNSUPPORTED beyond them): B, H <= 65535,
 * T <= 2^30, and for bf16 at chunk 64, which runs on the tensor-core kernels
 * whose TMA row coordinates are 32-bit, B * H * (ceil(T/64) + 1) * 128 < 2^31.  T need not be a multiple of chunk (the tail chunk is padded
 * inside the kernels with alpha = 1, beta = 0, which leaves the state unchanged).
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1, /* null/misaligned/overlapping pointer, bad size   */
    GDN_ERR_UNSUPPORTED = 2, /* K, V, chunk, dtype or a size outside the limits */
    GDN_ERR_WORKSPACE = 3,   /* workspace smaller than the *_workspace_bytes()  */
    GDN_ERR_CUDA = 4         /* a kernel launch failed (cudaGetLastError)        */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

/* Problem description.  `dtype` holds a gdn_dtype value. */
typedef struct {
    int64_t B, T, H, K, V;
    int32_t chunk;
    int32_t dtype;
} gdn_problem;

/* Library version (major * 10000 + minor * 100 + patch). */
int gdn_version(void);

/* Message for a status code (static storage). */
const char* gdn_status_string(gdn_status s);

/* Message describing the last failed call on the calling thread ("" if none). */
const char* gdn_last_error(void);

/* Bytes of device workspace gdn_fwd needs (the per-chunk Phase-1/solve results
 * handed to the scan).  Returns 0 for an invalid problem. */
size_t gdn_fwd_workspace_bytes(const gdn_problem* p);

/* Bytes of the `saved` buffer: the state at the start of every chunk, NC =
 * ceil(T / chunk) per stream ("OpenGDN", "Core operator reference": the reverse
 * keeps chunk boundaries instead of a token history).  Its contents are private
 * to gdn_fwd/gdn_bwd: float32 [B, H, NC, V, K] in general; on the tensor-core
 * path (bf16 inputs, chunk 64) bf16 [B, H, NC, 128, 128] states (they only
 * feed bf16 tensor-core products) followed by the forward's per-chunk solve
 * results, which gdn_bwd then reuses instead of recomputing ("atomic_ops",
 * "Features": the backward reuses forward residuals). */
size_t gdn_saved_bytes(const gdn_problem* p);

/* Bytes of device workspace gdn_bwd needs. */
size_t gdn_bwd_workspace_bytes(const gdn_problem* p);

/*
 * Forward.
 *   q, k, v, alpha, beta : inputs (device, dtype), layouts above.
 *   initial_state        : float32 [B,H,V,K] or NULL (= zeros).
 *   o                    : output [B,T,H,V] (device, dtype).
 *   final_state          : float32 [B,H,V,K] or NULL (= not written).  Passing it as
 *                          the next call's initial_state continues the stream exactly.
 *   saved                : NULL, or gdn_saved_bytes(p) bytes that receive the chunk
 *                          boundary states for gdn_bwd.
 *   workspace            : gdn_fwd_workspace_bytes(p) bytes (contents are scratch).
 * May be called with initial_state == final_state (in-place stream update).
 */
gdn_status gdn_fwd(const gdn_problem* p, const void* q, const void* k, const void* v,
                   const void* alpha, const void* beta, const float* initial_state,
                   void* o, float* final_state, void* saved, void* workspace,
                   size_t workspace_bytes, void* stream);

/*
 * Backward: gradients of L = sum(d_o * o) + sum(d_final_state * final_state)
 * with respect to q, k, v, alpha, beta and initial_state.
 *   saved          : the buffer a gdn_fwd call with the same inputs filled, or NULL
 *                    (the boundary states are then recomputed into the workspace).
 *   d_o            : [B,T,H,V] dtype.
 *   d_final_state  : float32 [B,H,V,K] or NULL (= zeros).
 *   dq, dk, dv, dalpha, dbeta : outputs in dtype, shapes of their inputs.
 *   d_initial_state: float32 [B,H,V,K] or NULL (= not written).
 *   workspace      : gdn_bwd_workspace_bytes(p) bytes.
 */
gdn_status gdn_bwd(const gdn_problem* p, const void* q, const void* k, const void* v,
                   const void* alpha, const void* beta, const float* initial_state,
                   const void* saved, const void* d_o, const float* d_final_state,
                   void* dq, void* dk, void* dv, void* dalpha, void* dbeta,
                   float* d_initial_state, void* workspace, size_t workspace_bytes,
                   void* stream);

/*
 * Forward for callers that cannot allocate device memory.  The pages have no
 * counterpart to this entry point; it is a convenience of this library.
 *
 * gdn_fwd needs a caller-owned workspace.  Some callers cannot provide one: code
 * running inside a host framework that owns all device memory (a plugin, or an
 * inference runtime whose memory pool is fixed and fully committed, where a
 * cudaMalloc fails or is not allowed), and code on a latency-critical path where
 * cudaMalloc/cudaFree would synchronise the device and stall concurrent work.
 * gdn_fwd_noalloc computes exactly what gdn_fwd computes (same kernels, no
 * `saved` output) with its scratch in a fixed array inside the library's device
 * memory: GDN_FWD_NOALLOC_SCRATCH_BYTES on every device that loads the library,
 * held until the process exits.  It calls no allocating routine.
 *   - Problems whose gdn_fwd_workspace_bytes(p) exceeds that size are rejected
 *     with GDN_ERR_UNSUPPORTED before anything is enqueued (e.g. bf16 with
 *     chunk 64 needs 40.25 KiB per (b, h, chunk), so
 *     B*H*ceil(T/64) <= 814, less when the within-call sequence split runs: it
 *     adds 192 KiB per (sequence, piece, head)).
 *   - The array used is the current device's: make the device that holds the
 *     tensors and runs `stream` current before the call.  A q on another
 *     device is rejected with GDN_ERR_INVALID_ARG.
 *   - The first call on a device looks up the array's address there
 *     (cudaGetSymbolAddress, with that device current): make that first call
 *     outside any stream capture.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind; calls that overlap on the GPU (e.g. on two streams) race and
 *     corrupt each other's results, so order them on one stream.  The only
 *     scratch words a call reads before writing them (the tensor-core path's
 *     error word and work counters) are cleared by a cudaMemsetAsync at the
 *     start of each call; everything else is written before it is read.
 * Arguments are those of gdn_fwd without saved/workspace; `o` is required.
 */
#define GDN_FWD_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
gdn_status gdn_fwd_noalloc(const gdn_problem* p, const void* q, const void* k, const void* v,
                           const void* alpha, const void* beta, const float* initial_state,
                           void* o, float* final_state, void* stream);

/*
 * gdn_prologue_fwd / gdn_prologue_bwd -- the step in front of the recurrence in
 * every mixer the pages show ("OpenGDN", Mixer: L2-normalized Q/K and per-head
 * alpha/beta gates), fused into one pass each way.  Per row (b, t, h):
 *     q = q_raw / sqrt(sum_K q_raw^2 + 1e-6)      (the same for k)
 *     alpha = exp(-softplus(a_logit)) = 1 / (1 + e^a_logit)
 *     beta  = sigmoid(b_logit)
 * (a mixer whose gate is alpha = sigmoid(x) passes a_logit = -x).  The backward
 * takes dL/dq, dL/dk, dL/dalpha, dL/dbeta (e.g. from gdn_bwd) and returns the
 * gradients with respect to q_raw, k_raw, a_logit, b_logit, recomputing the
 * norms and gates from the raw inputs (nothing is saved between the two calls).
 *   q_raw, k_raw, q, k, dq, dk, dq_raw, dk_raw  [B,T,H,K] in p->dtype;
 *   a_logit, b_logit, alpha, beta, dalpha, dbeta, da_logit, db_logit  [B,T,H].
 *   p->V and p->chunk are not used (V must still be a supported size).
 * All pointers 16-byte aligned and required; no output may overlap an input or
 * another output.  Errors are returned before any launch.  Allocates nothing;
 * asynchronous on `stream`.  Arithmetic in fp32.
 */
gdn_status gdn_prologue_fwd(const gdn_problem* p, const void* q_raw, const void* k_raw, const void* a_logit,
                            const void* b_logit, void* q, void* k, void* alpha, void* beta, void* stream);
gdn_status gdn_prologue_bwd(const gdn_problem* p, const void* q_raw, const void* k_raw, const void* a_logit,
                            const void* b_logit, const void* dq, const void* dk, const void* dalpha,
                            const void* dbeta, void* dq_raw, void* dk_raw, void* da_logit, void* db_logit,
                            void* stream);

/*
 * The recurrence with its prologue folded in: gdn_fwd / gdn_bwd on raw rows and
 * gate logits ("OpenGDN", Mixer: the mixer normalises q and k to unit L2 length
 * and computes the per-head gates in front of the operator).  Per row (b, t, h),
 * exactly as gdn_prologue_fwd:
 *     q = q_raw / sqrt(sum_K q_raw^2 + 1e-6)   (the same for k)
 *     alpha = exp(-softplus(a_logit)),  beta = sigmoid(b_logit)
 * then gdn_fwd on (q, k, v, alpha, beta); gdn_bwd_raw returns the gradients with
 * respect to q_raw, k_raw, v, a_logit, b_logit and the initial state of
 *     L = sum dO . o + sum d_final_state . final_state.
 * On the tensor-core kernels (bf16, chunk 64, K and V of 16 to 128) the prologue
 * runs inside them: the chunk kernel normalises the rows as they arrive and takes
 * log alpha = -softplus(a) directly in fp32, and the gradient kernels return the
 * raw inputs' gradients, so neither direction makes a separate pass over q and k.
 * Other shapes run the prologue kernel, then gdn_fwd / gdn_bwd, inside the call.
 *
 *   q_raw, k_raw, dq_raw, dk_raw  [B,T,H,K] p->dtype;  v, o, d_o, dv  [B,T,H,V];
 *   a_logit, b_logit, da_logit, db_logit  [B,T,H];  states as for gdn_fwd.
 *   saved      : NULL, or gdn_raw_saved_bytes(p) bytes (opaque): the normalised
 *                rows, their reciprocal norms and the forward's chunk results,
 *                for gdn_bwd_raw on the same inputs.
 *   workspace  : gdn_raw_fwd_workspace_bytes(p) / gdn_raw_bwd_workspace_bytes(p)
 *                bytes; scratch, contents undefined after the call.
 * Pointer, aliasing and error rules are those of gdn_fwd / gdn_bwd (checked before
 * any launch).  Allocates nothing, never synchronises; asynchronous on `stream`.
 */
size_t gdn_raw_saved_bytes(const gdn_problem* p);
size_t gdn_raw_fwd_workspace_bytes(const gdn_problem* p);
size_t gdn_raw_bwd_workspace_bytes(const gdn_problem* p);
gdn_status gdn_fwd_raw(const gdn_problem* p, const void* q_raw, const void* k_raw, const void* v,
                       const void* a_logit, const void* b_logit, const float* initial_state, void* o,
                       float* final_state, void* saved, void* workspace, size_t workspace_bytes, void* stream);
gdn_status gdn_bwd_raw(const gdn_problem* p, const void* q_raw, const void* k_raw, const void* v,
                       const void* a_logit, const void* b_logit, const float* initial_state, const void* saved,
                       const void* d_o, const float* d_final_state, void* dq_raw, void* dk_raw, void* dv,
                       void* da_logit, void* db_logit, float* d_initial_state, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * Packed variable-length batches.  "OpenGDN", Scope, lists ragged batches as not
 * supported; "Sparse Delta Memory: layer and kernels", What the layer computes,
 * masks the tokens past the end of a stream.  These calls run S = p->B
 * independent sequences of different lengths stored back to back: sequence s
 * is rows cu_seqlens[s] .. cu_seqlens[s+1]-1 of the packed tensors, and each
 * sequence has its own initial and final state.  The result for each sequence
 * equals gdn_fwd / gdn_bwd on that sequence alone (B = 1, T = its length).
 *
 *   p            : B = number of sequences S, T = an upper bound on every
 *                  sequence length, H, K, V, chunk, dtype as for gdn_fwd.
 *   total        : packed rows, 0 <= total <= B*T.
 *   cu_seqlens   : int32 [S+1] on the device, cu[0] = 0, non-decreasing,
 *                  cu[S] = total, every length <= T.  It is read by the kernels,
 *                  not on the host: a violation makes the offending sequences
 *                  empty (their outputs are not written) and sets bit 30 of the
 *                  int32 at the start of the workspace; the kernels never touch
 *                  memory outside the buffers.  That word also carries the
 *                  tensor-core kernels' bounded-wait bits (1..64); it is 0 when
 *                  the call succeeded.
 *   q, k         : packed [total, H, K] dtype;  v, o: [total, H, V];
 *   alpha, beta  : packed [total, H];  d_o and the gradients: packed, shapes of
 *                  their inputs.
 *   initial_state, final_state, d_final_state, d_initial_state : float32
 *                  [S, H, V, K] or NULL, as for gdn_fwd / gdn_bwd.
 *   saved        : NULL or gdn_varlen_saved_bytes(p, total) bytes, filled by
 *                  gdn_varlen_fwd and read by gdn_varlen_bwd with the same
 *                  inputs and cu_seqlens.  On the tensor-core path it also keeps
 *                  the chunk offsets and each chunk's first token and length, so
 *                  the backward does not recompute (or re-check) them.
 *   workspace    : gdn_varlen_fwd_workspace_bytes(p, total) /
 *                  gdn_varlen_bwd_workspace_bytes(p, total) bytes.
 * Method, tensor-core path (bf16, chunk 64, K and V of 16 to 128): the kernels
 * read and write the packed tensors in place.  Each sequence starts a new
 * chunk of one row of chunks per head; a device table gives every chunk its
 * first packed row and its number of rows (at most chunk - 1 padded rows per
 * sequence).  Rows of a ragged last chunk past the sequence's end are read
 * (they belong to the next sequence) but count as alpha = 1, beta = 0 and
 * d_o = 0, which leaves the results unchanged, and are never written.  The
 * scans run one stream per (sequence, head) over that sequence's chunks.
 * Other shapes: the sequences are copied into [S, T] streams inside the
 * workspace (padded rows q = k = v = 0, alpha = 1, beta = 0), gdn_fwd /
 * gdn_bwd run on them, and the results are copied back.  Host-side checks as
 * for gdn_fwd; every pointer 16-byte aligned except cu_seqlens (4 bytes);
 * S <= 65535.
 */
size_t gdn_varlen_fwd_workspace_bytes(const gdn_problem* p, int64_t total);
size_t gdn_varlen_bwd_workspace_bytes(const gdn_problem* p, int64_t total);
size_t gdn_varlen_saved_bytes(const gdn_problem* p, int64_t total);
gdn_status gdn_varlen_fwd(const gdn_problem* p, int64_t total, const int32_t* cu_seqlens, const void* q,
                          const void* k, const void* v, const void* alpha, const void* beta,
                          const float* initial_state, void* o, float* final_state, void* saved, void* workspace,
                          size_t workspace_bytes, void* stream);
gdn_status gdn_varlen_bwd(const gdn_problem* p, int64_t total, const int32_t* cu_seqlens, const void* q,
                          const void* k, const void* v, const void* alpha, const void* beta,
                          const float* initial_state, const void* saved, const void* d_o,
                          const float* d_final_state, void* dq, void* dk, void* dv, void* dalpha, void* dbeta,
                          float* d_initial_state, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Dense batches with reset masks.  "OpenGDN", Scope, lists reset masks among the
 * features it does not support, and no page gives a formula; this library reads
 * a reset at (b, t) as clearing the state just before token t, so that the row's
 * stream continues from the zero state at t (the recurrence with alpha_t = 0).
 * Each row is then a run of segments starting at t = 0 or at a reset, and the
 * calls run them as a packed batch (gdn_varlen_fwd / gdn_varlen_bwd) over the
 * B*T tokens of the dense tensors as they lie in memory.  The segmentation and
 * the routing of states between rows and segments are built on the device from
 * the mask: nothing is read back to the host.
 *
 *   p             : B, T, H, K, V, chunk, dtype as for gdn_fwd; q, k, v, alpha,
 *                   beta, o, d_o and the gradients [B,T,H,...] as there.
 *   max_segments  : an upper bound on the number of segments (B plus the number
 *                   of resets at t >= 1), in [B, B*T] and at most 65535.
 *                   Buffers and launches are sized by it.  More segments than the
 *                   bound set bit 29 of the int32 at the start of the workspace,
 *                   and the results are then not valid.
 *   reset         : uint8 [B, T] on the device, nonzero where the stream restarts
 *                   before that token.  A reset at t = 0 discards the row's
 *                   initial state (and its d_initial_state is 0).
 *   initial_state, final_state, d_final_state, d_initial_state : float32
 *                   [B,H,V,K] or NULL, per row, as for gdn_fwd / gdn_bwd.
 *   saved         : NULL or gdn_reset_saved_bytes(p, max_segments) bytes, from
 *                   gdn_reset_fwd for gdn_reset_bwd with the same inputs and mask.
 *   workspace     : gdn_reset_fwd_workspace_bytes / gdn_reset_bwd_workspace_bytes;
 *                   its first int32 is the error word of the packed calls (bit 30:
 *                   invalid offsets, bits 1..64: a bounded wait gave up) with
 *                   bit 29 added; it is 0 after a successful call.
 * Errors are returned before any launch (a NULL mask, a bound outside its range,
 * a workspace too small, overlaps).  Allocates nothing, never synchronises;
 * asynchronous on `stream`.
 */
size_t gdn_reset_saved_bytes(const gdn_problem* p, int64_t max_segments);
size_t gdn_reset_fwd_workspace_bytes(const gdn_problem* p, int64_t max_segments);
size_t gdn_reset_bwd_workspace_bytes(const gdn_problem* p, int64_t max_segments);
gdn_status gdn_reset_fwd(const gdn_problem* p, int64_t max_segments, const uint8_t* reset, const void* q,
                         const void* k, const void* v, const void* alpha, const void* beta,
                         const float* initial_state, void* o, float* final_state, void* saved, void* workspace,
                         size_t workspace_bytes, void* stream);
gdn_status gdn_reset_bwd(const gdn_problem* p, int64_t max_segments, const uint8_t* reset, const void* q,
                         const void* k, const void* v, const void* alpha, const void* beta,
                         const float* initial_state, const void* saved, const void* d_o, const float* d_final_state,
                         void* dq, void* dk, void* dv, void* dalpha, void* dbeta, float* d_initial_state,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * Within-call sequence split (two-level scan) of the tensor-core path.  The
 * chunk scans are sequential over a stream's chunks; with few streams most SMs
 * would idle, so each stream's chunks are cut into pieces that run side by side:
 * over a run of chunks the state map is affine, S_out = S_in P^T + R ("Sparse
 * Delta Memory: layer and kernels", What the layer computes: Phase 2 applies the
 * corrected writes to the chunk-start state), so a first pass computes every
 * piece's R (zero start) and P (its chunks' transition), a short chain links the
 * pieces, and a second pass runs every piece from its true start state.  The
 * backward does the same with the transposed maps.  The results equal the
 * unsplit scan's up to float32 rounding of the chain.
 *
 * gdn_set_sequence_split sets the policy for the calls that follow (process-wide):
 *   0 (default): automatic for gdn_fwd / gdn_bwd on the tensor-core path when
 *      the streams (B*H) would leave most SMs idle and the batch rows are whole
 *      chunks apart (B = 1 or T a multiple of the chunk); none for varlen calls;
 *   1: never;
 *   n >= 2: n pieces per sequence wherever the layout allows it (dense calls as
 *      above, and every varlen call on the tensor-core path).
 * The workspace sizes depend on it: query them under the policy of the calls,
 * and run a backward under the policy of its forward (their `saved` layouts
 * differ).  Returns GDN_ERR_INVALID_ARG outside [0, 1024].
 */
gdn_status gdn_set_sequence_split(int pieces);
int gdn_get_sequence_split(void);

/*
 * gdn_decode -- the recurrent step, for decoding: advances `state` through the
 * call's T tokens (usually 1) and writes their outputs.  It computes exactly the
 * token recurrence of section 1 ("OpenGDN", Core operator reference: a stream
 * continued through state=; "Sparse Delta Memory: layer and kernels",
 * Execution: the single-token call), in fp32, token by token:
 *     S <- alpha S (I - beta k k^T) + beta v k^T,   o = S q.
 * It reads and writes the state once per call, so it is bound by that traffic;
 * for long T, gdn_fwd's chunked kernels are faster.
 *   q, k   [B,T,H,K] and v, o [B,T,H,V] in p->dtype; alpha, beta [B,T,H].
 *   state  [B,H,V,K] fp32, required: read at entry, overwritten with the state
 *          after the last token.  Calls on one stream continue the stream
 *          exactly: T calls of one token equal one call of T tokens bit for bit.
 *   p->chunk is not used (any value is accepted); K, V in {16, 32, 64, 128}.
 * All pointers 16-byte aligned and required; o and state must not overlap each
 * other or any input.  Errors are returned before any launch.  Allocates
 * nothing; asynchronous on `stream`.
 */
gdn_status gdn_decode(const gdn_problem* p, const void* q, const void* k, const void* v,
                      const void* alpha, const void* beta, float* state, void* o, void* stream);

/*
 * gdn_count_nonfinite -- adds to *count the number of elements of x[0 .. n-1]
 * that are NaN or +-inf: a device-side check of inputs or results (for example,
 * the outputs of gdn_fwd after suspect inputs).  It does not synchronise: the
 * caller reads *count after synchronising `stream`.
 *   x      device tensor of n elements in `dtype` (GDN_F32 or GDN_BF16),
 *          16-byte aligned; may be NULL when n = 0.
 *   count  device int64, 8-byte aligned, required, owned by the caller (who
 *          zeroes it before the first call; calls accumulate).
 * Errors (negative n, unsupported dtype, NULL or misaligned pointers) are
 * returned before any launch.  Allocates nothing; asynchronous on `stream`.
 */
gdn_status gdn_count_nonfinite(const void* x, int64_t n, gdn_dtype dtype, int64_t* count, void* stream);

/*
 * gdn_test_set_wait_limit -- test hook for the error path of the tensor-core
 * kernels.  Every wait of those kernels on an mbarrier (a TMA copy or a
 * tensor-core operation completing) gives up after a limit, 2 s by default: the
 * kernel then sets a bit in the workspace's error word (its first int; the
 * kernel-specific code is the bit), stops issuing work, waits with the default
 * limit for the copies and tensor-core operations it already issued, frees its
 * tensor memory and exits, so the CUDA context stays usable.  This call sets the
 * limit, in nanoseconds, for the calls made after it (0 restores the default), of
 * every such wait except those of the q-side gradient kernel for its tensor-core
 * operations (that kernel takes it for its loads only).  With a limit of a few
 * nanoseconds the first wait that does not succeed at once gives up: the call
 * still returns GDN_OK, its error word is nonzero and its outputs are not valid.  Process-wide (it takes effect when a call's arguments
 * are checked); not for production use.
 */
gdn_status gdn_test_set_wait_limit(uint32_t ns);

/*
 * Optional launch timer, for benchmarks.  While started, every kernel launch of
 * gdn_fwd/gdn_bwd is bracketed by two CUDA events recorded on the call's stream
 * (up to `capacity` launches; later launches are not timed).  The events are
 * host-side driver objects created once by gdn_profiler_start; no device memory
 * is allocated.  Kernel ids run from 0 to gdn_num_kernels()-1; gdn_kernel_name
 * gives the CUDA kernel's name (as an ncu launch list shows it).
 * gdn_profiler_summary waits for the recorded events of kernel `id` and returns
 * their count and summed duration in milliseconds.  Not thread-safe.
 */
int gdn_num_kernels(void);
const char* gdn_kernel_name(int id);
gdn_status gdn_profiler_start(int capacity);
gdn_status gdn_profiler_stop(void);
gdn_status gdn_profiler_summary(int id, int* launches, double* total_ms);
void gdn_profiler_release(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
