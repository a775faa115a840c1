/*
 * kda.h -- C ABI of libkda, a GB300 (sm_103a) forward pass of Kimi Delta
 * Attention (KDA), the chunkwise gated delta rule with per-channel decay.
 *
 * What is computed ("You Could Have Come Up with Kimi Delta Attention",
 * sec. 4, the boxed KDA update; gates and norms as in "FlashKDA Delta
 * Attention Algorithm", Core Architecture).  Per sequence n and head h, with
 * state S (V x K, maps keys to values) starting at initial_state[n][h] or 0,
 * for each token t of the sequence in order:
 *
 *     q^ = q_t / sqrt(|q_t|^2 + 1e-6),  k^ = k_t / sqrt(|k_t|^2 + 1e-6)
 *     alpha[d] = exp(lower_bound * sigmoid(g_raw_t[d])),  beta = sigmoid(beta_raw_t)
 *     S~ = S Diag(alpha)                         (forget, per key channel)
 *     e  = beta (v_t - S~ k^)                    (predict and correct)
 *     S  = S~ + e k^T                            (write)
 *     o_t = S (scale q^)                         (read, after the write)
 *
 * and final_state[n][h] = S.  The GPU evaluates the same recurrence in
 * 16-token chunks (sec. 6 of the same page): a token-parallel chunk kernel and
 * a head-parallel recurrence kernel.
 *
 * Tensor conventions (all device pointers, caller-owned, contiguous, row-major,
 * 16-byte aligned):
 *   q, k, v, g_raw   bf16 [T_total, H, D]   (tokens of all sequences packed)
 *   beta_raw         bf16 [T_total, H]
 *   out              bf16 [T_total, H, D]
 *   initial_state    fp32 [N, H, V, K] or NULL (= zeros), V = K = D
 *   final_state      fp32 [N, H, V, K] or NULL (= not written); it may be the
 *                    initial_state buffer (updated in place) on every
 *                    schedule
 *   cu_seqlens       int32 [N + 1] on the device, or NULL.  With it, sequence
 *                    n is tokens [cu_seqlens[n], cu_seqlens[n+1]); it must
 *                    start at 0, be non-decreasing and end at T_total (not
 *                    checked by the forward calls, since the values live on
 *                    the device: kda_validate_cu_seqlens checks them).  Without it
 *                    there are N sequences of T_total / N tokens each.
 *   D must be 128 (the head size the kernels are built for), and T_total
 *   below 2^31 (the token coordinate of the kernels' tensor-map copies).
 *
 * Sequences of length 0 are allowed (their final state is the initial one).
 * Calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy default
 * stream); nothing synchronises inside.  Argument errors are reported before
 * anything is launched; errors found on the device (a bounded wait that ran
 * out) are latched in a device error word that kda_device_status() returns.
 * libkda keeps two things between calls: that error word, and the fixed
 * scratch array of kda_fwd_noalloc, which holds the last kda_fwd_noalloc
 * call's chunk records (see the race note of kda_fwd_noalloc below).  The
 * other entry points keep nothing.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kda_status {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1, /* null, misaligned or inconsistent argument        */
  KDA_ERR_UNSUPPORTED = 2, /* D != 128 or lower_bound outside [-5, 0]          */
  KDA_ERR_WORKSPACE = 3,   /* workspace too small, or its allocation failed     */
  KDA_ERR_LAUNCH = 4,      /* a CUDA call or kernel launch failed               */
  KDA_ERR_TIMEOUT = 5      /* a device-side wait ran out (see kda_device_status) */
} kda_status;

#define KDA_CHUNK 16
#define KDA_HEAD_DIM 128

/* Bytes of device workspace kda_fwd / kda_chunk_prep / kda_chunk_recurrence
 * need for these sizes: one chunk record (26176 bytes) per (chunk slot, head),
 * with T_total / 16 + N + 1 chunk slots, enough for any split of T_total
 * tokens into N sequences.  Returns 0 for invalid sizes. */
size_t kda_workspace_size(int64_t T_total, int32_t H, int32_t N, int32_t D);

/* Whole forward pass: chunk kernel (K1) then recurrence kernel (K2).
 * workspace: device buffer of at least kda_workspace_size(...) bytes, 16-byte
 * aligned, or NULL, in which case libkda allocates it with cudaMallocAsync on
 * `stream` and frees it with cudaFreeAsync after the kernels.
 * scale: the read scale (1 / sqrt(D) in the pages); lower_bound in [-5, 0]:
 * with 16-token chunks this keeps every cumulative decay factor and its
 * inverse inside the normal fp32 range ("FlashKDA v1: A Deep Dive", sec. 1).
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, LAUNCH as listed above. */
kda_status kda_fwd(const void* q, const void* k, const void* v, const void* g_raw,
                   const void* beta_raw, float scale, float lower_bound,
                   const float* initial_state, const int32_t* cu_seqlens, int64_t T_total,
                   int32_t H, int32_t N, int32_t D, void* out, float* final_state,
                   void* workspace, size_t workspace_bytes, void* stream);

/* The same forward pass in one kernel: each (sequence, head) CTA builds the
 * chunk records in shared memory (the K1 arithmetic) and runs the recurrence
 * on them (the K2 arithmetic), so the records never go through HBM and no
 * workspace is needed.  Same arguments, results and errors as kda_fwd minus the
 * workspace; results agree with kda_fwd to rounding (identical arithmetic in a
 * different schedule). */
kda_status kda_fwd_fused(const void* q, const void* k, const void* v, const void* g_raw,
                         const void* beta_raw, float scale, float lower_bound,
                         const float* initial_state, const int32_t* cu_seqlens, int64_t T_total,
                         int32_t H, int32_t N, int32_t D, void* out, float* final_state,
                         void* stream);

/* The same forward pass in the recurrent (decode) schedule: the token-by-token
 * recurrence of "You Could Have Come Up with Kimi Delta Attention" (sec. 4,
 * boxed), run as in its sec. 5 decode regime.  One CTA per (sequence, head, 32
 * value rows) keeps that slice of the fp32 state in registers and walks the
 * sequence's tokens in order.  Meant for short sequences and stateful serving
 * (a few tokens per sequence per call), where moving the state dominates; for
 * long sequences kda_fwd_fused is the faster schedule of the same result.
 * Same arguments, results and errors as kda_fwd_fused.  final_state may be the
 * same buffer as initial_state (updated in place).  Results agree with the
 * chunkwise entry points to rounding. */
kda_status kda_decode(const void* q, const void* k, const void* v, const void* g_raw,
                      const void* beta_raw, float scale, float lower_bound,
                      const float* initial_state, const int32_t* cu_seqlens, int64_t T_total,
                      int32_t H, int32_t N, int32_t D, void* out, float* final_state,
                      void* stream);

/* Options of kda_forward. */
enum { KDA_SCHEDULE_SPLIT = 0, KDA_SCHEDULE_FUSED = 1, KDA_SCHEDULE_DECODE = 2,
       KDA_SCHEDULE_SEGMENTED = 3, KDA_SCHEDULE_AUTO = 4 };
enum { KDA_STATE_F32 = 0, KDA_STATE_BF16 = 1 };
enum { KDA_GATE_PER_CHANNEL = 0, KDA_GATE_PER_HEAD = 1 };
typedef struct {
  int32_t schedule;     /* KDA_SCHEDULE_*: kda_fwd (split), kda_fwd_fused, kda_decode,
                           kda_fwd_segmented (automatic piece count), or AUTO:
                           decode for at most 8 tokens per sequence on average,
                           segmented when kda_segments_auto() > 1 (too few
                           (sequence, head) units for the SMs), fused otherwise */
  int32_t state_dtype;  /* KDA_STATE_*: dtype of initial_state and final_state (both) */
  int32_t gate;         /* KDA_GATE_*: g_raw [T_total, H, D] or [T_total, H] */
} kda_options;

/* The forward pass with options, on any schedule.
 * state_dtype = KDA_STATE_BF16: initial_state and final_state are bf16
 *   [N, H, V, K] (16-byte aligned), converted to and from the fp32 state at
 *   load and store; both have that dtype, as the FlashKDA API requires of a
 *   given pair ("FlashKDA: MoonshotAI's High-Performance Kimi Delta Attention
 *   Kernels", API reference).  The state itself stays fp32 inside the pass.
 * gate = KDA_GATE_PER_HEAD: g_raw is bf16 [T_total, H] (2-byte aligned), one
 *   gate per token and head shared by every key channel, so alpha_t is a scalar
 *   times the identity: the Gated DeltaNet special case of KDA ("You Could
 *   Have Come Up with Kimi Delta Attention", sec. 3), with the same gate map
 *   log alpha = lower_bound * sigmoid(g_raw).
 * workspace / workspace_bytes are used by KDA_SCHEDULE_SPLIT (as in kda_fwd)
 * and KDA_SCHEDULE_SEGMENTED or an AUTO choice of it
 * (kda_segmented_workspace_size with segments = 0; NULL = allocated on the
 * stream); the segmented schedule keeps every piece's
 * states in fp32 and converts only initial_state and final_state.  Everything
 * else is as in kda_fwd; a null `opts` or an unknown option value returns
 * KDA_ERR_INVALID_ARG. */
kda_status kda_forward(const kda_options* opts, const void* q, const void* k, const void* v,
                       const void* g_raw, const void* beta_raw, float scale, float lower_bound,
                       const void* initial_state, const int32_t* cu_seqlens, int64_t T_total,
                       int32_t H, int32_t N, int32_t D, void* out, void* final_state,
                       void* workspace, size_t workspace_bytes, void* stream);

/* The forward pass on HOST buffers: q, k, v, g_raw, beta_raw, initial_state,
 * cu_seqlens, out and final_state are host pointers (pinned memory lets the
 * copies overlap; pageable memory works, with copies that stage through the
 * driver).  Layouts, options and results are those of kda_forward; cu_seqlens
 * is a host int32 [N + 1], checked here (0 first, non-decreasing, T_total
 * last; otherwise KDA_ERR_INVALID_ARG before anything is queued).
 * The call pipelines the host-to-device copies, the passes and the
 * device-to-host copies in `groups` pieces (1 .. 16; 0 = 8):
 *   - G groups of whole sequences, each copied in, run (one kda_forward over
 *     its own sequences) and copied out on streams of its own;
 *   - for N equal sequences without cu_seqlens, fewer than `groups` of them,
 *     and fp32 states: each sequence cut in time into up to G chunk-aligned
 *     slices; slice p of all sequences runs once its rows have arrived,
 *     starting from the fp32 state slice p - 1 left in device memory (exact:
 *     the recurrence is a left-to-right scan).
 * Every copy is one cudaMemcpyAsync (or one cudaMemcpy2DAsync for the rows of
 * all N sequences of a slice) on library-owned copy streams, ordered after
 * the work already queued on `stream`; `stream` waits for the last copy, so
 * the host outputs are complete once `stream` is.  The host inputs must stay
 * unchanged, and the outputs untouched, until then.
 * workspace: device memory of kda_fwd_host_workspace_size() bytes, 256-byte
 * aligned (the inputs, outputs, states and each piece's kda_forward
 * workspace), or NULL (= cudaMallocAsync / cudaFreeAsync on `stream`).
 * Concurrent calls are serialised while they queue their work.
 * Errors: those of kda_forward; KDA_ERR_WORKSPACE for a small or misaligned
 * workspace; KDA_ERR_LAUNCH if a copy or launch fails. */
kda_status kda_fwd_host(const kda_options* opts, const void* q, const void* k, const void* v,
                        const void* g_raw, const void* beta_raw, float scale, float lower_bound,
                        const void* initial_state, const int32_t* cu_seqlens, int64_t T_total,
                        int32_t H, int32_t N, int32_t D, void* out, void* final_state,
                        int32_t groups, void* workspace, size_t workspace_bytes, void* stream);

/* Device workspace bytes of kda_fwd_host for these arguments (cu_seqlens is
 * the host array, or NULL); 0 for invalid arguments. */
size_t kda_fwd_host_workspace_size(const kda_options* opts, int64_t T_total, int32_t H,
                                   int32_t N, int32_t D, const int32_t* cu_seqlens,
                                   int32_t groups);

/* Size of the fixed workspace array used by kda_fwd_noalloc (64 MiB). */
#define KDA_NOALLOC_WORKSPACE_BYTES (64 * 1024 * 1024)

/* kda_fwd without any allocation, for callers that cannot allocate device
 * memory (for example a plugin inside a host engine that owns all device
 * memory and offers no allocator).  The pages have no counterpart to this
 * entry point; it exists for such callers only.
 * Same arguments and results as kda_fwd, minus the workspace: the K1->K2
 * records go to a fixed 64 MiB device array inside libkda.  A GPU holds that
 * array from the first kda_fwd_noalloc call on it (or from library load under
 * eager module loading, CUDA_MODULE_LOADING=EAGER) until the process exits.
 * Limit: kda_workspace_size(T_total, H, N, D) must not exceed
 * KDA_NOALLOC_WORKSPACE_BYTES (e.g. T_total + 16 (N + 1) <= 1280 tokens at
 * H = 32, <= 41,008 at H = 1); larger sizes return KDA_ERR_WORKSPACE before
 * anything is launched.
 * The first call on a device looks up the array's device address with
 * cudaGetSymbolAddress (once per device, with that device current), so make
 * that first call before any stream capture.  All calls share the one array:
 * calls whose kernels overlap on the GPU (different streams, no ordering)
 * race on it and their results are undefined; calls ordered on one stream are
 * fine.  The array keeps the previous call's contents; nothing in it needs to
 * start at zero.  No cudaMalloc, cudaFree or other allocating routine is
 * called. */
kda_status kda_fwd_noalloc(const void* q, const void* k, const void* v, const void* g_raw,
                           const void* beta_raw, float scale, float lower_bound,
                           const float* initial_state, const int32_t* cu_seqlens,
                           int64_t T_total, int32_t H, int32_t N, int32_t D, void* out,
                           float* final_state, void* stream);

/* K1 alone: the token-parallel chunk kernel.  Writes one record per (chunk,
 * head) into `workspace` (same size rule as kda_fwd; must not be NULL).  For
 * chunk c (0-based) of sequence n and head h the record starts at byte
 *   ((floor(bos_n / 16) + n + c) * H + h) * 26176
 * with bos_n the first token of sequence n, and holds, for the chunk's tokens
 * i < 16 (rows past the sequence end are zero), in this order:
 *   [Qdec' ; W'] bf16 32 x 128, 128-byte-swizzled K-major tiles;
 *   [Kend' ; Aqk'] fp32 144 x 16 (Kend'^T rows 0-127, Aqk' rows 128-143), two
 *   32-byte-swizzled K=8 tiles;  U'^T fp32 [128][16];  dlast fp32 [128];
 *   rq fp32 [16];
 * where (sec. 6.1-6.6 of "You Could Have Come Up with Kimi Delta Attention")
 *   Qdec_i = scale q^_i D_{0:i},  Kend_i = k^_i D_{i+1:last},
 *   Akk = (I + R)^-1 with R_ij = beta_i <k^_j|D_{j+1:i}|k^_i> (j < i),
 *   W = Akk diag(beta) [k^_i D_{0:i}],  U = Akk diag(beta) V,
 *   Aqk_ij = scale <k^_j|D_{j+1:i}|q^_i> (j <= i),  dlast = diag(D_{0:last}),
 * stored with the per-token norms rk_j = 1 / |k_j| and rq_i = scale / |q_i|
 * moved between factors (the products the recurrence forms are unchanged):
 * W'_i = rk_i W_i,  U'_i = rk_i U_i,  Kend'_j = Kend_j / rk_j,
 * Qdec'_i = Qdec_i / rq_i,  Aqk'_ij = Aqk_ij / (rq_i rk_j), and rq itself, by
 * which the recurrence scales each output row.
 * The byte layout of each tile is given in chunked_gated_delta_11_gb300/csrc/
 * kda_common.cuh. */
kda_status kda_chunk_prep(const void* q, const void* k, const void* v, const void* g_raw,
                          const void* beta_raw, float scale, float lower_bound,
                          const int32_t* cu_seqlens, int64_t T_total, int32_t H, int32_t N,
                          int32_t D, void* workspace, size_t workspace_bytes, void* stream);

/* K2 alone: the head-parallel recurrence over records written by
 * kda_chunk_prep with the same sizes and cu_seqlens.  One CTA per (sequence,
 * head) keeps the fp32 state in tensor memory and walks its chunks. */
kda_status kda_chunk_recurrence(const void* workspace, size_t workspace_bytes,
                                const float* initial_state, const int32_t* cu_seqlens,
                                int64_t T_total, int32_t H, int32_t N, int32_t D, void* out,
                                float* final_state, void* stream);

/* The forward pass for few long sequences: every sequence is cut into
 * `segments` pieces that run at the same time and are joined by a scan of
 * their state maps.  Each token step of the recurrence is an affine map of
 * the state, S -> S A_t + beta_t v_t k^_t^T with A_t = Diag(alpha_t)
 * (I - beta_t k^_t k^_t^T) ("You Could Have Come Up with Kimi Delta
 * Attention", sec. 4.1), so a piece maps its starting state S_0 to S_0 M + X:
 *   - M = A_1 ... A_n comes from running the piece with v = 0 from the
 *     identity; that run's outputs are y_t = M_t (scale q^_t);
 *   - X comes from running the piece from zero, with outputs o^X_t;
 *   - a scan over the pieces of each (sequence, head), S_0 <- S_0 M + X in
 *     fp32, gives every piece its S_0 and the final state;
 *   - o_t = o^X_t + S_0 y_t, added on the tensor cores (bf16 S_0 and y, fp32
 *     sums, rounded to bf16 once more).
 * Pieces are whole 16-token chunks: piece j of a sequence with c chunks holds
 * chunks [floor(c j / P), floor(c (j + 1) / P)), so pieces may be empty when
 * c < P.  Results equal kda_fwd_fused's up to rounding.
 * Arguments are those of kda_fwd_fused (states fp32), plus:
 *   segments   pieces per sequence P, 1..64; 0 = kda_segments_auto().  P = 1
 *              is kda_fwd_fused itself (no workspace).
 *   gate       KDA_GATE_PER_CHANNEL or KDA_GATE_PER_HEAD (as in kda_forward).
 *   workspace  device memory of kda_segmented_workspace_size() bytes (16-byte
 *              aligned), or NULL (= cudaMallocAsync / cudaFreeAsync on the
 *              stream).  It holds the piece boundaries, the X and M states of
 *              every piece (2 N P H 64 KiB), a bf16 copy of the pieces'
 *              starting states (N P H 32 KiB) and y (T_total H 256 bytes).
 * T_total must be below 2^31 (piece boundaries are int32).  The runtime is set
 * by the longest piece: the pieces' units take N H (2 P - 1) CTAs of the fused
 * kernel, two per SM. */
kda_status kda_fwd_segmented(const void* q, const void* k, const void* v, const void* g_raw,
                             const void* beta_raw, float scale, float lower_bound,
                             const float* initial_state, const int32_t* cu_seqlens,
                             int64_t T_total, int32_t H, int32_t N, int32_t D, void* out,
                             float* final_state, int32_t segments, int32_t gate,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes kda_fwd_segmented needs for these sizes and `segments`
 * (0 = the automatic count); 0 when it needs none or the sizes are invalid. */
size_t kda_segmented_workspace_size(int64_t T_total, int32_t H, int32_t N, int32_t D,
                                    int32_t segments);

/* The automatic piece count on the current device: the largest P with
 * N H (2 P - 1) <= 2 x (SM count), at most 64, and at least 24 chunks per
 * piece on average; 1 means no split. */
int32_t kda_segments_auto(int64_t T_total, int32_t H, int32_t N);

/* Synchronises `stream`, then returns and clears the device error word of the
 * current device: KDA_OK; KDA_ERR_TIMEOUT if a kernel's bounded wait ran out
 * since the last call (its outputs are then invalid); KDA_ERR_INVALID_ARG if
 * kda_validate_cu_seqlens found a bad cu_seqlens; or KDA_ERR_LAUNCH if the
 * synchronisation itself failed. */
kda_status kda_device_status(void* stream);

/* Checks on the device, asynchronously on `stream`, what the forward entry
 * points assume of a device cu_seqlens [N + 1]: it starts at 0, never
 * decreases and ends at T_total.  A violation latches KDA_ERR_INVALID_ARG in
 * the device error word (read it with kda_device_status); nothing traps.
 * The forward calls themselves do not check (the values live on the device);
 * run this first on untrusted input.  Returns KDA_ERR_INVALID_ARG for a null
 * or misaligned pointer, N <= 0, or T_total outside [0, 2^31), and
 * KDA_ERR_LAUNCH if the launch fails. */
kda_status kda_validate_cu_seqlens(const int32_t* cu_seqlens, int32_t N, int64_t T_total,
                                   void* stream);

/* Static description of a status code (never NULL). */
const char* kda_status_string(kda_status status);

/* Diagnostic: one-CTA check of the tensor-core operand conventions used by
 * the recurrence kernel (bf16 MMA with A in tensor memory and the record's
 * 128-byte-swizzled [Qdec ; W] tile; tf32 MMA with N = 144, A in tensor memory
 * and the record's 32-byte-swizzled [Kend ; Aqk] tiles, accumulating into a
 * preset D).  Writes out1 fp32 [128][32] and out2 fp32 [128][144] (device),
 * and 5 to *status
 * (device int) if its wait ran out.  Returns 0, 1 for bad arguments, 4 on a
 * launch error.  The expected values are closed-form small dyadic numbers
 * (see the kernel source), exact in fp32. */
int kda_selftest_tcgen05(float* out1, float* out2, int* status, void* stream);

/* Diagnostic of the device-side timeout path (the failure detection of the
 * bounded waits): one CTA holds tensor memory and waits on an mbarrier that
 * nothing arrives at, with the forward kernels' wait routine but a limit of
 * `limit_cycles` SM cycles (1 .. 2^31; the forward kernels use 2^31, about a
 * second).  When the wait runs out the CTA latches KDA_ERR_TIMEOUT in the
 * device error word, frees its tensor memory and exits, exactly as a forward
 * kernel does; kda_device_status() then returns KDA_ERR_TIMEOUT once and clears
 * it.  Asynchronous on `stream`.  Returns KDA_ERR_INVALID_ARG for a limit
 * outside that range and KDA_ERR_LAUNCH if the launch fails. */
kda_status kda_selftest_timeout(int64_t limit_cycles, void* stream);

/* Context parallelism: the pieces of one long sequence on different ranks.
 * Each token step of the recurrence is an affine map of the state,
 * S -> S A_t + beta_t v_t k^_t^T with A_t = Diag(alpha_t)(I - beta_t k^_t k^_t^T)
 * ("You Could Have Come Up with Kimi Delta Attention", sec. 4.1), so the piece
 * of rank r (tokens in order, all heads) maps its starting state S_0 to
 * S_0 M_r + X_r, and inside it o_t = o^X_t + S_0 y_t, y_t = M_t (scale q^_t).
 * A rank runs kda_piece_forward on its piece, the ranks exchange the (M_r, X_r)
 * pairs (the only exchange step: 2 x H x 64 KiB per rank, gathered in rank
 * order by the caller's collective library), each rank runs kda_pieces_scan
 * over the gathered pairs and kda_piece_fixup on its own outputs.  Results
 * agree with one pass over the whole sequence up to rounding (the fix-up adds
 * S_0 y in bf16 with fp32 sums, as kda_fwd_segmented does).  All pointers are
 * device pointers of the calling rank's GPU; states fp32 [H, V, K] per piece.
 *
 * kda_piece_forward: m_state == NULL: the first piece, a plain fused pass from
 *   initial_state (NULL = zeros) writing `out` and its final state x_state.
 *   m_state != NULL: a later piece (initial_state must be NULL): out = o^X
 *   (from zero), x_state = X_r, m_state = M_r and y (bf16 [T_local, H, V]) =
 *   the identity-start, v = 0 run's outputs (may be NULL for an empty
 *   piece, T_local = 0, whose maps are X = 0 and M = I).  gate: KDA_GATE_*.  workspace:
 *   kda_piece_workspace_size() bytes (needed with m_state).
 * kda_pieces_scan: xs, ms fp32 [P, H, V, K] of the P pieces in order (ms[0] is
 *   not read); replaces xs[j] (j >= 1) by piece j's starting state S_0 and
 *   writes the state after the last piece to final_state (or NULL).
 * kda_piece_fixup: out (bf16 [T_local, H, V]) += s0 (fp32 [H, V, K]) y; needs a
 *   256-byte workspace. */
size_t kda_piece_workspace_size(int64_t T_local, int32_t H);
kda_status kda_piece_forward(const void* q, const void* k, const void* v, const void* g_raw,
                             const void* beta_raw, float scale, float lower_bound,
                             const float* initial_state, int64_t T_local, int32_t H, int32_t D,
                             void* out, float* x_state, float* m_state, void* y, int32_t gate,
                             void* workspace, size_t workspace_bytes, void* stream);
kda_status kda_pieces_scan(float* xs, const float* ms, int32_t P, int32_t H, int32_t D,
                           float* final_state, void* stream);
kda_status kda_piece_fixup(void* out, const void* y, const float* s0, int64_t T_local, int32_t H,
                           int32_t D, void* workspace, size_t workspace_bytes, void* stream);

/* Diagnostic: where the serial chain of the recurrence spends its time.
 * Runs one forward pass over N equal sequences (no cu_seqlens, zero initial
 * state, fp32 final state) with kernel 0 = the chunk kernel then a timed copy
 * of the recurrence kernel (workspace as for kda_fwd, required), or kernel 1 =
 * a timed copy of the fused kernel (workspace unused).  Thread 0 of the first
 * (sequence, head) CTA writes the SM clock (clock64) at the phase boundaries
 * of each of its first max_chunks chunks c to stamps[8 c + k] (device int64,
 * 8-byte aligned, 8 max_chunks entries; entry 7 unused):
 *   k = 0 first MMA issued, 1 first MMA complete, 2 corrected errors written
 *   (second MMA issued), 3 second MMA complete, 4 next record available,
 *   5 snapshot and decay of the state done, 6 outputs stored.
 * The results (out, final_state) are those of kda_fwd.  The timed copies are
 * separate instantiations; the other entry points do not record anything.
 * There is no counterpart on the pages; it backs the per-phase analysis of the
 * chain.  Errors as kda_fwd. */
kda_status kda_profile_phases(int32_t kernel, const void* q, const void* k, const void* v,
                              const void* g_raw, const void* beta_raw, float scale,
                              float lower_bound, int64_t T_total, int32_t H, int32_t N,
                              int32_t D, void* out, float* final_state, void* workspace,
                              size_t workspace_bytes, long long* stamps, int32_t max_chunks,
                              void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
