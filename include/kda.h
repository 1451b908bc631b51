/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention forward library.
 *
 * The operation is the forward pass of KDA, a per-head gated delta rule, as the
 * FlashKDA pages state it: the guancyxx.cn FlashKDA article, section 一
 * ("什么是 Delta Attention": a recurrent state S of shape [K, V] with a learned
 * decay) and section 2.2 (a token-parallel intra-chunk stage and a head-parallel
 * chunk-wise delta-rule recurrence), and the FlashKDA README mirror
 * (ai-feeds.com), section "内核 API" (argument table of flash_kda.fwd) and section
 * "将 FlashKDA 用作 FLA 后端" (L2 norm of q/k, beta sigmoid and gate inside the
 * kernel, transposed [V, K] state layout).
 *
 * Per sequence n and head h, with K = V = 128 and token t of the sequence:
 *   q^ = q_t / sqrt(|q_t|^2 + 1e-6),  k^ = k_t / sqrt(|k_t|^2 + 1e-6)
 *   b  = sigmoid(beta_t)
 *   a_c = lower_bound * sigmoid(exp(A_log[h]) * (g_t[c] + dt_bias[h][c]))   c = 0..127
 *   S' = Diag(exp(a)) S_{t-1};  S_t = S' + k^ (b (v_t - S'^T k^))^T;  o_t = scale * S_t^T q^
 * The pages name g, A_log, dt_bias and lower_bound but print no formula for the
 * gate; the form above is the one this library implements (bounded in
 * (lower_bound, 0)).  The 1e-6 inside the norm is likewise this library's choice.
 *
 * Layouts (row-major, element strides implied, all device pointers unless noted):
 *   q, k, v, g, out : bf16 [B, T, H, 128]          (B = N without cu_seqlens, B = 1 with it)
 *   beta            : bf16 [B, T, H]               (logits; the sigmoid is applied inside)
 *   A_log           : fp32 [H];  dt_bias : fp32 [H, 128]
 *   initial_state, final_state : [N, H, 128 (V), 128 (K)], element [n][h][v][k] = S[k][v],
 *                     bf16 or fp32 as state_dtype says
 *   cu_seqlens      : int64 [N + 1], cumulative sequence lengths (varlen mode)
 *
 * Ownership: the caller allocates and owns every buffer, including out and
 * final_state.  kda_fwd takes its scratch workspace (the per-chunk operands passed from
 * the prep kernel to the recurrence kernel, kda_fwd_workspace_size bytes) from a
 * stream-ordered memory pool that the library owns, one per device, and returns it on
 * the same stream; the pool keeps the memory for later calls until kda_workspace_trim.
 * kda_fwd_ws takes a caller-owned workspace instead.  Calls are asynchronous on
 * `stream`; results are valid once the stream has been synchronised.  initial_state may
 * equal final_state (in-place update).  Calls on different streams may run
 * concurrently if their output buffers (and kda_fwd_ws workspaces) do not overlap.
 *
 * Numerics: the chunked form of the recurrence (64-token chunks, 16-token decay
 * sub-blocks).  A prep kernel computes, for every chunk in parallel, the gate, the L2
 * norms, the decay factors, the strictly-lower beta K K^T and causal Q K^T matrices
 * (tf32 tensor-core products of factors in fp32 range), the (I + A)^-1 inverse (fp32)
 * and the WY products, and stores the recurrence operands in fp16 (each bounded by 1 in
 * magnitude except T' V and T' (K^ . Gamma), which are delta-rule residuals of the
 * inputs).  A recurrence kernel then runs the chunk-to-chunk state update on the tensor
 * cores with fp16 operands and fp32 accumulation; the state itself stays fp32 for the
 * whole call.  The fp16 operands (the state's copy, T' V and the corrected values U) bound
 * the magnitudes: states and values must stay well below the fp16 limit of 6.5e4.  Tested
 * with v scaled by 256 (|v| up to ~1.3e3) and fp32 initial states ~N(0, 300); past the limit
 * the state turns inf / NaN and kda_device_status reports KDA_ERR_NONFINITE.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *kda_stream_t; /* same type as cudaStream_t; NULL = legacy default stream */

typedef enum {
    KDA_DTYPE_NONE = 0, /* no state tensors */
    KDA_DTYPE_BF16 = 1,
    KDA_DTYPE_FP32 = 2
} kda_dtype_t;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARGUMENT = 1, /* NULL required pointer, bad size, misaligned pointer, bad dtype/state combination */
    KDA_ERR_UNSUPPORTED = 2,      /* lower_bound outside [-5, 0], scale not finite, or a size limit of the entry point */
    KDA_ERR_CUDA = 3,             /* a CUDA runtime call or the kernel launch failed */
    KDA_ERR_TIMEOUT = 4,          /* a bounded device wait expired (reported by kda_device_status) */
    KDA_ERR_NONFINITE = 5         /* a final state came out inf / NaN (reported by kda_device_status) */
} kda_status_t;

/*
 * kda_fwd -- the KDA chunked forward pass (the call that flash_kda.fwd makes in
 * the README mirror's "内核 API" section, in C form).
 *
 *   q, k, v, g     bf16 [B, T, H, 128], device, 16-byte aligned.
 *   beta           bf16 [B, T, H], device, 2-byte aligned.
 *   scale          output scale (finite).
 *   out            bf16 [B, T, H, 128], device, 16-byte aligned; written for every token.
 *   A_log          fp32 [H], device.   dt_bias  fp32 [H, 128], device, 16-byte aligned.
 *   lower_bound    gate lower bound, must lie in [-5, 0].
 *   initial_state  [N, H, 128, 128] of state_dtype, device, or NULL (zero initial state).
 *   final_state    [N, H, 128, 128] of state_dtype, device, or NULL (not returned).
 *   state_dtype    dtype of whichever state pointers are non-NULL (both share it); ignored
 *                  when both are NULL.  States must be 16-byte aligned.
 *   cu_seqlens     int64 [N + 1], device, or NULL.  With it, B = 1, T is the total token
 *                  count and sequence n covers tokens [cu[n], cu[n+1]).  The contents must
 *                  satisfy cu[0] = 0, cu[i] <= cu[i+1], cu[N] = T; they are device-resident
 *                  and not checked (see kda_check_cu_seqlens).  Zero-length sequences are
 *                  allowed: their final state equals the initial one.
 *   N              number of sequences (>= 1): B without cu_seqlens.
 *   T              tokens per sequence (without cu_seqlens) or in total (with it), >= 0.
 *   H              number of heads, >= 1.
 *   stream         CUDA stream to run on.
 *
 * When T == 0 (no tokens at all) q, k, v, g, beta and out may be NULL.
 *
 * Fixed-length problems of 1 to 16 tokens per sequence (decode steps, short speculative runs)
 * are evaluated token by token, as kda_fwd_recurrent does (same kernels, same bits, no
 * workspace), where that is faster than the chunked form; everything else takes the chunked
 * form.
 *
 * Fixed-length problems with N x H <= 16 pairs and at least 32 chunks per sequence replace the
 * serial chain of the recurrence by a scan along T when its cost model says it is faster
 * (kda_fwd_scan_groups): the chunks of each pair are cut into G groups; the transition of every
 * group (the affine map S -> M S + B its chunks apply to the state) is formed in parallel, the
 * groups' start states follow serially in fp32 (G - 1 steps of S <- M S + B), and the groups then
 * run in parallel from them.  The results are not the same bits as the serial chain (a different
 * order of operations) but within the same tolerances.
 *
 * Otherwise, fixed-length problems with N x H <= 64 (sequence, head) pairs and at least 32 chunks of 64
 * tokens per sequence run in pieces of whole chunks along T where the overlap pays for a piece's
 * cost (kda_fwd_pieces: up to 8, more for longer sequences and fewer pairs; at least 16 chunks
 * each), all on `stream`: the prep kernel
 * of the next piece is launched as a programmatic dependent of the recurrence over the current
 * one (it reads nothing that recurrence writes), so the two run side by side on different SMs;
 * the prep kernel completes only after that recurrence has.  The state passes between pieces in
 * fp32 (through the workspace), as it does between chunks, so the results are the same bits as
 * without pieces.
 *
 * Returns KDA_OK once the work is enqueued.  Argument errors are reported
 * synchronously before anything is launched; the kernel itself never traps.
 */
kda_status_t kda_fwd(const void *q, const void *k, const void *v, const void *g, const void *beta,
                     float scale, void *out, const float *A_log, const float *dt_bias,
                     float lower_bound, const void *initial_state, void *final_state,
                     kda_dtype_t state_dtype, const int64_t *cu_seqlens, int N, int64_t T, int H,
                     kda_stream_t stream);

/*
 * Bytes of workspace kda_fwd_ws needs for this problem size (an upper bound that depends
 * only on N, T, H and whether cu_seqlens is given: varlen != 0).  0 for invalid sizes and for
 * the fixed-length problems of 1 to 16 tokens per sequence, which need none.
 */
size_t kda_fwd_workspace_size(int N, int64_t T, int H, int varlen);

/*
 * Number of pieces along T in which kda_fwd, kda_fwd_ws and kda_fwd_noalloc run a problem of this
 * size on the current device (see kda_fwd): 1 when the call runs without pieces (every varlen
 * problem, the fixed-length problems outside the piece rule, and those whose overlap would not pay
 * for a second piece), 2 to 8 otherwise.  0 for invalid
 * sizes, or when the device's SM count cannot be read.  Launches nothing.
 */
int kda_fwd_pieces(int N, int64_t T, int H, int varlen);

/*
 * Number of groups G of the chunk-transition scan along T in which kda_fwd, kda_fwd_ws and
 * kda_fwd_noalloc run a problem of this size (see kda_fwd): 1 when the recurrence runs as one serial
 * chain per (sequence, head) pair, 2 to 32 otherwise.  Depends on N, T, H and varlen only (the
 * workspace holds the scan's matrices: (1 + 3 (G - 1)) x N x H x 64 KiB ahead of the operand slots).
 * 0 for invalid sizes.  Launches nothing.
 */
int kda_fwd_scan_groups(int N, int64_t T, int H, int varlen);

/*
 * kda_fwd_ws -- kda_fwd with a caller-owned device workspace of at least
 * kda_fwd_workspace_size(N, T, H, cu_seqlens != NULL) bytes, 256-byte aligned (it may be
 * NULL when that size is 0).  The workspace must not be used by anything else until the
 * call has completed on `stream`.  Same arguments, results and errors as kda_fwd, plus
 * KDA_ERR_INVALID_ARGUMENT for a missing, misaligned or too small workspace.
 *
 * CUDA graphs: a kda_fwd_ws call (like a kda_fwd_recurrent call) can be captured from `stream`
 * into a CUDA graph once a call of any size has run on the device outside a capture (the first
 * call on a device sets the kernels' attributes and caches device properties).  The graph holds
 * the call's launches and copies for whichever schedule the size selects (one launch of each
 * kernel, pieces with programmatic dependent launches, the scan along T, varlen, the
 * token-recurrent kernels) and its replays give the bits of direct calls on the data then in the
 * captured buffers (tests/test_gpu_graph.py).
 */
kda_status_t kda_fwd_ws(const void *q, const void *k, const void *v, const void *g, const void *beta,
                        float scale, void *out, const float *A_log, const float *dt_bias,
                        float lower_bound, const void *initial_state, void *final_state,
                        kda_dtype_t state_dtype, const int64_t *cu_seqlens, int N, int64_t T, int H,
                        void *workspace, size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_fwd_ws_profiled -- kda_fwd_ws that also records CUDA events on `stream` at the stage
 * boundaries, for timing the two kernels separately: stage_events[0] right before the prep
 * kernel (after the varlen plan), [1] between the prep and recurrence kernels, [2] after the
 * recurrence kernel.  stage_events points to 3 cudaEvent_t handles (any may be NULL).  The
 * prep kernel always runs over every chunk before the recurrence starts, all on `stream`, and the
 * recurrence runs as one serial chain per pair, also for the problems that kda_fwd_ws runs in pieces
 * (same results, bit for bit) or with the scan along T (results within the same tolerances).
 */
kda_status_t kda_fwd_ws_profiled(const void *q, const void *k, const void *v, const void *g, const void *beta,
                                 float scale, void *out, const float *A_log, const float *dt_bias,
                                 float lower_bound, const void *initial_state, void *final_state,
                                 kda_dtype_t state_dtype, const int64_t *cu_seqlens, int N, int64_t T, int H,
                                 void *workspace, size_t workspace_bytes, void *const *stage_events,
                                 kda_stream_t stream);

/* Bits of kda_fwd_ws_variant: the FlashKDA pages' own precision choices for the chunked path. */
#define KDA_VARIANT_BF16_STATE 1u       /* the state kept in bf16 between 64-token chunks (rounded to nearest) */
#define KDA_VARIANT_NEUMANN_INVERSE 2u  /* (I + A)^-1 as the fp16 Neumann-series product */

/*
 * kda_fwd_ws_variant -- kda_fwd_ws with measurement variants that follow the guancyxx.cn FlashKDA
 * article, section 2.3 ("bf16 循环状态 + fp16 矩阵求逆"): a state stored in bf16 between chunks instead
 * of the library's fp32 state, and an fp16 Neumann-series product (I - A)(I + A^2)(I + A^4) ...
 * (I + A^32) for the chunk inverse instead of the library's blocked fp32 substitution.  variant is
 * an OR of KDA_VARIANT_* bits (0 gives exactly kda_fwd_ws).  They exist to measure those choices on
 * this hardware: the bf16 state is less precise (its rounding accumulates over the chunks) and the
 * Neumann product costs more tensor-core steps; neither is faster here.  Same arguments, layouts and
 * errors as kda_fwd_ws, plus KDA_ERR_INVALID_ARGUMENT for unknown variant bits.  Fixed-length
 * problems of 1 to 16 tokens per sequence take the token-recurrent kernels whatever the variant.
 */
kda_status_t kda_fwd_ws_variant(const void *q, const void *k, const void *v, const void *g, const void *beta,
                                float scale, void *out, const float *A_log, const float *dt_bias,
                                float lower_bound, const void *initial_state, void *final_state,
                                kda_dtype_t state_dtype, const int64_t *cu_seqlens, int N, int64_t T, int H,
                                void *workspace, size_t workspace_bytes, unsigned variant, kda_stream_t stream);

/* Capacity of the static workspace of kda_fwd_noalloc (256 MiB per device). */
#define KDA_NOALLOC_SCRATCH_BYTES 268435456

/*
 * kda_fwd_noalloc -- kda_fwd that allocates no memory: its workspace is a fixed array of
 * KDA_NOALLOC_SCRATCH_BYTES in the library's device code (a file-scope __device__ array).  The
 * FlashKDA pages have no counterpart of this entry point.  It is meant for callers that cannot
 * allocate device memory while they run the forward pass: a runtime that reserves its whole
 * memory budget up front and forbids allocator calls afterwards, or code whose latency-critical
 * path must not enter the CUDA allocator (cudaMalloc, stream-ordered pools) at all.
 *
 *   - Every device that loads the library holds its own copy of the array from then until the
 *     process exits (256 MiB of device memory each, whether or not this entry point is called).
 *   - The first call on a device that needs a workspace looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; later calls reuse it.  Make
 *     that first call on each device before capturing any stream.
 *   - All calls on one device share the array and it keeps the contents of the last call: calls
 *     whose kernels may overlap on the GPU (different streams without an ordering between them)
 *     race and give undefined results.  The forward pass writes every part of the array it reads
 *     before reading it, so nothing has to be cleared between calls.
 *   - Problems whose workspace (kda_fwd_workspace_size(N, T, H, cu_seqlens != NULL)) exceeds
 *     KDA_NOALLOC_SCRATCH_BYTES (a single 8192-token sequence with 96 heads does) are rejected
 *     with KDA_ERR_UNSUPPORTED before any CUDA call.  Fixed-length problems of 1 to 16 tokens per
 *     sequence need no workspace and make no lookup.
 *
 * Same arguments, results and other errors as kda_fwd; KDA_ERR_CUDA if the address lookup fails.
 */
kda_status_t kda_fwd_noalloc(const void *q, const void *k, const void *v, const void *g, const void *beta,
                             float scale, void *out, const float *A_log, const float *dt_bias,
                             float lower_bound, const void *initial_state, void *final_state,
                             kda_dtype_t state_dtype, const int64_t *cu_seqlens, int N, int64_t T, int H,
                             kda_stream_t stream);

/*
 * kda_fwd_recurrent -- the same operation as kda_fwd, evaluated token by token: the
 * per-token update of the guancyxx.cn FlashKDA article, section 一 (the recurrent form
 * that the chunked form of section 2.2 reorganises).  A persistent grid walks the
 * (sequence, head, half of the values) items; each CTA holds an item's 64 state columns
 * in fp32 registers while the next items' states and tokens stream in (fixed-length
 * problems of 1 to 4 tokens per sequence mostly take a decode kernel whose warps work
 * without CTA barriers, longer or varlen problems 8-token stages; both give the same
 * bits).  Meant for decode
 * steps (one or a few tokens per sequence) and short prefills, where it moves only the
 * state and the tokens (no per-chunk operands, no workspace, no allocation); its cost
 * grows linearly with the longest sequence, so long sequences belong to kda_fwd.  Same
 * arguments, layouts, ownership (including in-place initial_state == final_state) and
 * errors as kda_fwd, plus KDA_ERR_UNSUPPORTED when T >= 2^31 or 2 N H >= 2^31.  Results agree with
 * kda_fwd's within the parity tolerances, not bit for bit: this path keeps every operand
 * in fp32.
 */
kda_status_t kda_fwd_recurrent(const void *q, const void *k, const void *v, const void *g, const void *beta,
                               float scale, void *out, const float *A_log, const float *dt_bias,
                               float lower_bound, const void *initial_state, void *final_state,
                               kda_dtype_t state_dtype, const int64_t *cu_seqlens, int N, int64_t T, int H,
                               kda_stream_t stream);

/*
 * kda_fwd_host -- kda_fwd on HOST buffers: q, k, v, g, beta, out, A_log, dt_bias,
 * initial_state, final_state and cu_seqlens are host pointers with kda_fwd's layouts and
 * alignments.  The library copies the inputs to the current device, runs the forward pass there
 * and copies out (and final_state) back, and returns when the results are in host memory.  The
 * FlashKDA pages have no counterpart: it is this library's end-to-end entry point.  Fixed-length
 * problems are cut into pieces of whole 64-token chunks, varlen problems into pieces of whole
 * sequences (the longest, from 4 chunks on, last and in pieces of whole chunks), and the copies of
 * neighbouring pieces overlap the kernels on three streams of the library's own; the state passes
 * between pieces of one sequence in fp32 (pieces of whole sequences share none),
 * so the results are bit-identical to kda_fwd on the same data -- except where kda_fwd, or a
 * piece, runs the scan along T (kda_fwd_scan_groups > 1: at most 16 (sequence, head) pairs with
 * long sequences), whose grouping of the chunks differs: there the two agree within the parity
 * tolerances of the oracle (and bit for bit when the decay is strong enough that a chunk forgets
 * its start state, as with lower_bound = -5).  The fixed-length pieces are up to 8 big pieces of
 * about T / 8 tokens, then a tail that halves down to 128 tokens.  Page-locked (pinned) host
 * memory lets the copies run asynchronously; pageable memory works but the copies do not overlap.
 * Device memory comes from the library's pool (see kda_workspace_trim).  Calls are serialised per
 * device.  Errors: those of kda_fwd (cu_seqlens is also checked, on the host, as
 * kda_check_cu_seqlens does), KDA_ERR_CUDA for a failed copy, allocation or launch.
 */
kda_status_t kda_fwd_host(const void *q, const void *k, const void *v, const void *g, const void *beta,
                          float scale, void *out, const float *A_log, const float *dt_bias,
                          float lower_bound, const void *initial_state, void *final_state,
                          kda_dtype_t state_dtype, const int64_t *cu_seqlens, int N, int64_t T, int H);

/*
 * kda_fwd_host_plan -- the pieces kda_fwd_host cuts a problem of N sequences and T tokens into, in
 * the order it copies them in (a host-side query: it touches no device).  cu_seqlens is a HOST
 * pointer (varlen) or NULL (fixed length, T tokens per batch row).  Piece i covers token rows
 * [first_token[i], first_token[i] + tokens[i]) (of every batch row, fixed length) and sequences
 * [first_seq[i], first_seq[i] + seqs[i]) (fixed length: 0 and N); a piece of the longest varlen
 * sequence covers one sequence (seqs = 1) in part, starting at a multiple of 64 tokens from the
 * sequence's start.  Writes at most max_pieces entries (the four arrays may be NULL when it is 0)
 * and returns the number of pieces, or -1 for N < 1, T outside [0, 2^40], or a cu_seqlens that
 * kda_check_cu_seqlens rejects.  The plan depends on N, T and cu_seqlens only.
 */
int kda_fwd_host_plan(int N, int64_t T, const int64_t *cu_seqlens, int64_t *first_token, int64_t *tokens,
                      int *first_seq, int *seqs, int max_pieces);

/*
 * Returns the workspace memory kda_fwd's pools hold but no call is using to the driver.
 * KDA_ERR_CUDA if a pool could not be trimmed.
 */
kda_status_t kda_workspace_trim(void);

/*
 * Host-side check of a cu_seqlens array (host pointer, N + 1 entries) against the
 * contract above.  Returns KDA_OK or KDA_ERR_INVALID_ARGUMENT.  No CUDA calls.
 */
kda_status_t kda_check_cu_seqlens(const int64_t *host_cu_seqlens, int N, int64_t T);

/* Static English description of a status code (never NULL). */
const char *kda_status_string(kda_status_t status);

/*
 * Waits for `stream`, then reports what the kernels of this library on this device (kda_fwd and
 * its variants, kda_fwd_recurrent) recorded since the last call, and clears it:
 *   KDA_ERR_TIMEOUT           a kernel gave up a bounded wait on the tensor cores or a bulk copy;
 *                             the outputs of that call are not valid;
 *   KDA_ERR_INVALID_ARGUMENT  a device-resident cu_seqlens broke its contract (cu[0] != 0,
 *                             cu[N] != T or a decreasing entry); the kernels clamped every
 *                             sequence into [0, T] and the chunk table into the workspace, so no
 *                             access left the buffers, but the outputs are not valid;
 *   KDA_ERR_NONFINITE         the chunked path ended a (sequence, head) with a non-finite state:
 *                             an inf / NaN input, or a value beyond the fp16 range of its
 *                             tensor-core operands (see Numerics above);
 * in that order of precedence, else KDA_OK.  KDA_ERR_CUDA if the stream or the query failed.
 * The kernels never spin without a limit and never trap.
 */
kda_status_t kda_device_status(kda_stream_t stream);

/* Default of kda_set_wait_limit: mbarrier polls before a wait of the chunked kernels gives up. */
#define KDA_DEFAULT_WAIT_POLLS 16777216u

/*
 * Sets how many times a wait of the chunked kernels (kda_fwd and its variants, on the tensor cores
 * and on bulk copies) polls before it gives up, for the kernels launched after the call, process-wide
 * (default KDA_DEFAULT_WAIT_POLLS, which is far beyond any wait of a working kernel).  A wait that
 * gives up makes its CTA wait for its own work in flight (with the default limit), free its tensor
 * memory and leave; kda_device_status then reports KDA_ERR_TIMEOUT and the call's outputs are not
 * valid.  polls = 0 makes every such wait give up at once: a way to exercise that error path without
 * a hang.  The token-recurrent kernels (kda_fwd_recurrent, decode-sized kda_fwd calls) always use
 * the default.  Thread-safe; not a diagnostic of anything on its own.
 */
void kda_set_wait_limit(uint32_t polls);

/* Largest dynamic shared memory one CTA of the forward kernels uses (for diagnostics). */
size_t kda_fwd_smem_bytes(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
