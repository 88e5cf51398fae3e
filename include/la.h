/*
 * la.h -- C ABI of the GB300 (sm_103a) causal linear-attention library.
 *
 * The library computes the generalised linear-attention recurrence
 *
 *     S_t = S_{t-1} A_t + beta_t v_t k_t^T ,      o_t = S_t q_t
 *
 * ("History Replays Itself: Unleashing Long-Context Capability in Linear
 * Attention" (NoteBank), Sec. 2, Eq. (1)) in two instantiations:
 *
 *   Taylor / BASED   A_t = I, beta_t = 1 on the feature-mapped keys
 *                    phi(x) = [1, x, vec(x x^T)/sqrt(2)], with the
 *                    normaliser  y_i = s_i^T phi(q_i) / (z_i^T phi(q_i) + eps),
 *                    s_i = s_{i-1} + phi(k_i) v_i^T, z_i = z_{i-1} + phi(k_i)
 *                    ("BASED：简单线性注意力如何平衡召回能力与生成吞吐", reading
 *                    notes of "Simple linear attention language models balance
 *                    the recall-throughput tradeoff", Sec. 2.2 = paper
 *                    Eqs. (1)-(3); Sec. 2.3 = paper Eq. (4)).
 *   Gated DeltaNet   A_t = alpha_t (I - beta_t k_t k_t^T), i.e.
 *                    S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T
 *                    (the delta-rule family named in NoteBank Sec. 2; its
 *                    per-token cost J(7 d_k d_v + d_k + 2 d_v) in App. C.6,
 *                    Eq. (11) counts exactly this update).
 *
 *   Scalar gate      A_t = alpha_t I, i.e. S_t = alpha_t S_{t-1} + beta_t v_t k_t^T
 *                    (the "gated" family NoteBank Sec. 2 names next to the
 *                    delta rule; alpha = beta = 1 is standard additive linear
 *                    attention, A_t = I); same arguments as Gated DeltaNet.
 *
 * All run as a chunked prefill that returns the final state (the state is
 * carried across chunk boundaries, NoteBank Sec. 3.2) and as a one-token
 * decode step that updates the state in place.  Outputs are read after the
 * token's own write (o_t = S_t q_t with S_t already holding token t).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library never allocates or frees memory; scratch space comes from the
 *     caller's workspace buffer, sized by the *_workspace_size queries.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL is the legacy default stream).  Argument validation happens on the
 *     host before anything is launched; a rejected call launches nothing.
 *   - Element strides are given per tensor for the batch, head and token
 *     axes; the last (feature) axis must be contiguous.  Base pointers and
 *     token strides must be 16-byte aligned (in bytes), as the tile loaders
 *     move 16-byte vectors and TMA boxes.
 *   - States are fp32, contiguous, and may alias (state_in == state_out is
 *     an in-place update, the copy-and-branch use of NoteBank Alg. 1).
 *   - No exception crosses the ABI; every failure is a la_status.
 */
#ifndef LA_H
#define LA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LA_ABI_VERSION 2

typedef enum la_status {
  LA_OK = 0,
  LA_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad size, stride or alignment */
  LA_ERR_UNSUPPORTED = 2,      /* well-formed but outside the built kernels   */
  LA_ERR_WORKSPACE = 3,        /* workspace missing or too small              */
  LA_ERR_CUDA = 4,             /* a CUDA runtime/driver call failed           */
  LA_ERR_TIMEOUT = 5           /* a bounded device-side wait gave up          */
} la_status;

typedef enum la_dtype { LA_DTYPE_F32 = 0, LA_DTYPE_BF16 = 1 } la_dtype;

typedef enum la_variant { LA_VARIANT_TAYLOR = 0, LA_VARIANT_GDN = 1, LA_VARIANT_GATED = 2 } la_variant;

/* A strided [B, H, N, d] view; strides in ELEMENTS; the d axis is contiguous. */
typedef struct la_tensor {
  void* ptr;
  int64_t stride_b, stride_h, stride_t;
} la_tensor;

/* Taylor (BASED) prefill.
 *   q, k : [B, H, N, d_feat]   in_dtype      (d_feat = d' = 16)
 *   v    : [B, H, N, d_v]      in_dtype      (d_v = 64)
 *   y    : [B, H, N, d_v]      out_dtype     y_i = s_i^T phi(q_i) / (z_i^T phi(q_i) + eps)
 *   s_in : [B, H, D, d_v] fp32 contiguous, D = 1 + d' + d'^2 = 273, rows in
 *          the order [1, x_0..x_{d'-1}, x_a x_b/sqrt2 for a, then b]; NULL = zero.
 *   z_in : [B, H, D] fp32 contiguous; NULL = zero.
 *   s_out, z_out : final state after token N-1 (required; may alias s_in/z_in).
 *   eps  : added to the denominator (0 reproduces the pages' definition).
 *   decay: NULL, or [H] fp32 on the device: a fixed retention lambda_h per
 *          head, s_i = lambda_h s_{i-1} + phi(k_i) v_i^T and z_i likewise
 *          (BASED notes, the paragraph on decay after Table 7: the 10B-token
 *          runs use a fixed per-head decay rate).  For lambda_h in [0, 1]
 *          every intermediate stays in range; values are not checked. */
typedef struct la_based_prefill_args {
  int64_t B, H, N, d_feat, d_v;
  la_dtype in_dtype, out_dtype;
  la_tensor q, k, v, y;
  const float* s_in;
  const float* z_in;
  float* s_out;
  float* z_out;
  float eps;
  const float* decay;
} la_based_prefill_args;

/* Gated DeltaNet prefill.
 *   q, k : [B, H, N, d_k]  in_dtype;  v, o : [B, H, N, d_v] in/out_dtype
 *          (d_k = d_v = 128)
 *   alpha, beta : [B, H, N] fp32 strided views (their feature axis is absent;
 *          stride_t must be 1)
 *   q_scale : multiplies q (1 = the pages' parametrisation: input scaling is
 *          absorbed into q, NoteBank Sec. 2)
 *   S_in : [B, H, d_v, d_k] fp32 contiguous (row i = value index); NULL = zero
 *   S_out: final state (required; may alias S_in). */
typedef struct la_gdn_prefill_args {
  int64_t B, H, N, d_k, d_v;
  la_dtype in_dtype, out_dtype;
  la_tensor q, k, v, o;
  la_tensor alpha, beta;
  float q_scale;
  const float* S_in;
  float* S_out;
} la_gdn_prefill_args;

/* One decode step for S sequences x H heads, state updated in place.
 *   variant : LA_VARIANT_TAYLOR, LA_VARIANT_GDN or LA_VARIANT_GATED (the
 *          scalar gate; layouts as GDN)
 *   q, k : [S, H, d_k] contiguous in_dtype (Taylor: d_k means d' = 16)
 *   v    : [S, H, d_v] contiguous in_dtype
 *   alpha, beta : [S, H] fp32 contiguous (GDN and scalar gate; ignored for Taylor)
 *   out  : [S, H, d_v] contiguous out_dtype
 *   state: GDN / scalar gate [S, H, d_v, d_k] fp32; Taylor [S, H, D, d_v] fp32 (s)
 *   z    : Taylor [S, H, D] fp32 (ignored otherwise)
 *   eps  : Taylor denominator term; q_scale: GDN / scalar-gate query scale.
 *   decay: Taylor only: NULL or [H] fp32 per-head retention lambda_h, as in
 *          la_based_prefill_args (ignored otherwise). */
typedef struct la_decode_args {
  la_variant variant;
  int64_t S, H, d_k, d_v;
  la_dtype in_dtype, out_dtype;
  const void* q;
  const void* k;
  const void* v;
  const float* alpha;
  const float* beta;
  void* out;
  float* state;
  float* z;
  float eps;
  float q_scale;
  const float* decay;
} la_decode_args;

/* Bytes of device workspace the matching prefill call needs for `args`
 * (0 = none; a NULL workspace is then accepted).  Pure host functions of the
 * sizes and dtypes in `args` (no pointer is read), so they can be asked
 * before any buffer is allocated.  The workspace must be 16-byte aligned;
 * its contents need no initialisation and are dead when the call's work on
 * the stream has finished.
 *
 * Gated-delta-rule prefill (bf16 inputs) has two schedules:
 *   - records (the fastest): one record of 16,384 bytes per 64-token chunk
 *     of every (b,h) (the bf16 images of T diag(beta), T = (I + L)^{-1}, and
 *     of the chunk's causal queries against its keys), read once by a
 *     warp-specialized scan per (b,h) that also reads q, k, v once and forms
 *     everything else.  When the (b,h) pairs leave at least 16 SMs free and
 *     sequences are not split, the records are formed in the scan's own
 *     launch (a cooperative launch over every SM) by CTAs beside the scan
 *     and handed over through one 4-byte flag per record; otherwise a
 *     chunk-parallel kernel forms them first.  la_gdn_prefill_workspace_size
 *     returns what it needs: the records, the flags (rounded up to 256
 *     bytes), 4,352 bytes of launch scratch, plus the segment scratch below
 *     when long sequences are split;
 *   - one kernel that walks the chunks of each (b,h) itself; it needs scratch
 *     only when it splits long sequences of few (b,h) pairs into segments
 *     (one 64 KiB fp32 map pair per segment but the last, one 64 KiB entry
 *     state per segment); la_gdn_prefill_workspace_size_min returns that
 *     (often 0).
 * la_gdn_prefill runs the records schedule when the workspace holds at
 * least la_gdn_prefill_workspace_size bytes, else the one-kernel schedule
 * when it holds at least la_gdn_prefill_workspace_size_min bytes, else fails
 * with LA_ERR_WORKSPACE.  Both compute the same result up to rounding. */
size_t la_based_prefill_workspace_size(const la_based_prefill_args* args);
size_t la_gdn_prefill_workspace_size(const la_gdn_prefill_args* args);
size_t la_gdn_prefill_workspace_size_min(const la_gdn_prefill_args* args);

/* Chunked Taylor prefill (BASED notes Sec. 2.2 and Sec. 2.5: the block
 * decomposition U_b = (M_b . Phi_Qb Phi_Kb^T) V_b + Phi_Qb S_{<b}). */
la_status la_based_prefill(const la_based_prefill_args* args, void* workspace,
                           size_t workspace_bytes, void* stream);

/* Chunked gated-delta-rule prefill (NoteBank Sec. 2 Eq. (1); chunks carry
 * the state across boundaries as in NoteBank Sec. 3.2).  When the records
 * schedule forms its records inside the scan's launch (see the workspace
 * notes above), that launch is cooperative and places one CTA on every SM of
 * the device: it starts once all SMs are free and holds them until it ends,
 * so it does not overlap with the caller's kernels on other streams.  Its
 * CTAs wait on one another only through bounded waits (LA_ERR_TIMEOUT). */
la_status la_gdn_prefill(const la_gdn_prefill_args* args, void* workspace,
                         size_t workspace_bytes, void* stream);

/* Chunked scalar-gate prefill, A_t = alpha_t I (NoteBank Sec. 2 Eq. (1) with
 * the gated family's retention): S_t = alpha_t S_{t-1} + beta_t v_t k_t^T,
 * o_t = S_t (q_scale q_t).  Arguments, layouts, workspace (query it with the
 * la_gdn_prefill_workspace_size functions), schedules and errors exactly as
 * la_gdn_prefill; the chunk form is the same with L = 0, so T = I. */
la_status la_gated_prefill(const la_gdn_prefill_args* args, void* workspace,
                           size_t workspace_bytes, void* stream);

/* la_gdn_prefill for callers that cannot allocate device memory (the pages
 * have no counterpart; this is an interface convenience).  Some callers have
 * no workspace to hand over: a plug-in inside a host framework that owns all
 * device memory and forbids its plug-ins to allocate, an engine that reserved
 * its whole memory budget up front, or a latency-critical loop that must not
 * pay the implicit device-wide synchronisation of cudaMalloc/cudaFree.  This
 * entry point computes exactly what la_gdn_prefill computes, but takes its
 * scratch from a fixed 16 MiB array in the library's own device memory, so it
 * calls no cudaMalloc, cudaFree or other allocating routine.
 *   - Limit: problems whose la_gdn_prefill_workspace_size_min exceeds
 *     16 MiB (16777216 bytes) are refused with LA_ERR_WORKSPACE before
 *     anything is launched; problems that need no scratch always run.  The
 *     records schedule runs when its records fit the array, otherwise
 *     the one-kernel schedule.
 *   - Every GPU that loads the library holds the 16 MiB array until the
 *     process exits.
 *   - The first call in each CUDA context looks up the array's device
 *     address (cudaGetSymbolAddress, with that context's device current)
 *     and caches it under the context's id; make that first call before
 *     any stream capture.  A device reset (cudaDeviceReset, or anything
 *     else that destroys and recreates the primary context) invalidates the
 *     cached address: the next call then looks it up again, so the first
 *     call after a reset must also come before any capture.
 *   - All calls share the one array and it keeps the last call's contents
 *     (nothing in it needs to start at zero).  Calls whose GPU work overlaps,
 *     e.g. on two streams at once, race on it: serialise them.
 * Arguments, validation and other errors as for la_gdn_prefill. */
la_status la_gdn_prefill_noalloc(const la_gdn_prefill_args* args, void* stream);

/* One decode step of sliding-window softmax attention, the window layers of
 * BASED (BASED notes Sec. 2.4: standard softmax over the last `window`
 * tokens, whose KV the layer keeps; Sec. 2.5: the step fuses dot products,
 * softmax and weighted sum).  S sequences x H heads, head dim d.
 *   q, k, v : [S, H, d] contiguous in_dtype (any rotary embedding applied)
 *   k_cache, v_cache : [S, H, window, d] contiguous in_dtype ring buffers;
 *          token p lives in slot p % window; the step writes k, v of token
 *          pos into slot pos % window (updated in place)
 *   pos  : [S] int64 device array, tokens already seen per sequence (read
 *          only: the caller advances it); slots 0..min(pos, window-1) must
 *          hold tokens pos - min(pos, window - 1) .. pos - 1
 *   out  : [S, H, d] out_dtype, o = sum_j softmax_j(scale q . k_j) v_j over
 *          tokens max(0, pos - window + 1) .. pos
 *   scale: multiplies q . k (1/sqrt(d) for standard softmax attention)
 * d: a multiple of 8 in [8, 128]; window in [1, 256]; pointers 16-byte
 * aligned.  A negative pos skips that sequence and sets the device status
 * word (la_device_status reports LA_ERR_INVALID_ARGUMENT). */
typedef struct la_swa_decode_args {
  int64_t S, H, d, window;
  la_dtype in_dtype, out_dtype;
  const void* q;
  const void* k;
  const void* v;
  void* k_cache;
  void* v_cache;
  const int64_t* pos;
  void* out;
  float scale;
} la_swa_decode_args;

/* Like la_decode_step, the step's kernel is launched as a programmatic
 * dependent of the kernel before it on the stream: it may be scheduled while
 * that kernel finishes, but touches memory only once it has completed, so the
 * usual stream order holds. */
la_status la_swa_decode_step(const la_swa_decode_args* args, void* stream);

/* One recurrent decode step (NoteBank Eq. (1) for one token; BASED notes
 * Sec. 2.5: the decode step fuses the outer-product write with the query
 * readout and still reads and writes the whole persistent state).  The step's
 * kernel is launched as a programmatic dependent of the kernel before it on
 * the stream: it may be scheduled while that kernel finishes (which hides the
 * launch gap between consecutive steps) but reads and writes memory only once
 * it has completed, so the usual stream order holds. */
la_status la_decode_step(const la_decode_args* args, void* stream);

/* Readout-boundary state rescaling (NoteBank App. D.1: S <- lambda S with
 * lambda in [0, 1]; lambda = 1 keeps the state, lambda = 0 resets it).
 *   states : n_states consecutive fp32 states of elems_per_state elements
 *            each (any state of this library: GDN / scalar-gate S, Taylor s
 *            or z), device memory, 4-byte aligned (16 bytes runs faster)
 *   lambda : device array of n_states factors, or NULL to use lambda_all
 * A factor of 0 writes zeros whatever the state held.  Asynchronous on
 * stream; the states are updated in place. */
la_status la_state_rescale(float* states, int64_t n_states, int64_t elems_per_state,
                           const float* lambda, float lambda_all, void* stream);

/* State copy and branch (NoteBank App. B, Alg. 1: the question is processed
 * on a copy of the state): destination state i becomes a copy of source
 * state index[i], for i < n_dst (one source may feed several destinations).
 *   dst : n_dst states, src : n_src states (fp32, elems_per_state each,
 *         device memory, 4-byte aligned); dst and src must not overlap
 *         (LA_ERR_INVALID_ARGUMENT otherwise, nothing launched)
 *   index : device int64 array of n_dst source indices
 * An index outside [0, n_src) leaves that destination untouched and sets the
 * device status word: la_device_status then reports LA_ERR_INVALID_ARGUMENT. */
la_status la_state_gather(float* dst, const float* src, const int64_t* index, int64_t n_dst,
                          int64_t n_src, int64_t elems_per_state, void* stream);

/* ---- NoteBank write side and routing ("History Replays Itself: Unleashing
 * Long-Context Capability in Linear Attention" (NoteBank), Sec. 2 Eqs. (3)-(5),
 * App. B Eqs. (8)-(9)).  A channel is one (layer, head) of the backbone:
 * the L x H channels of one document are passed as [L, H, N, d] views. */

/* Per-token distinctiveness (Eqs. (3), (8)).  For every chunk of `chunk`
 * tokens ([c*chunk, (c+1)*chunk), the last one possibly short) and channel:
 *   mu = unit(mean of the chunk's unit keys),  d_ch[l,h,t] = 1 - <unit(k_t), mu>;
 * d_mean[t] = mean of d_ch over the channels; w[t] = d_mean[t] + ... +
 * d_mean[t + window - 1] for t <= N - window (the sliding window whose
 * maximum picks a note's first window, App. B.2: window = 48).  A zero key
 * normalises to zero (it scores 1).
 *   k      : [L, H, N, d] in_dtype view (stride_b = layer, stride_h = head,
 *            stride_t = token; the feature axis contiguous), d a multiple of
 *            32 up to 256
 *   chunk  : 1..1024 (the pages' write chunk is 512 for GDN)
 *   window : 1..4096
 *   d_ch   : [L, H, N] fp32, d_mean : [N] fp32, w : [N - window + 1] fp32 or
 *            NULL; device memory, contiguous.
 * fp32 arithmetic; the channel mean and window sums add in a fixed order. */
typedef struct la_notebank_scores_args {
  int64_t L, H, N, d;
  la_dtype in_dtype;
  la_tensor k;
  int64_t chunk, window;
  float* d_ch;
  float* d_mean;
  float* w;
} la_notebank_scores_args;
la_status la_notebank_scores(const la_notebank_scores_args* args, void* stream);

/* Note addresses (Eqs. (4), (9)): for note i with token span
 * [spans[2i], spans[2i] + spans[2i+1]) and channel (l,h),
 *   t_star[i,l,h] = argmax over the span of d_ch[l,h,t] (the earliest token
 *                   on ties),
 *   rho[i,l,h,:]  = q[l,h,t_star, coords[l,h,0..15]] rounded to bf16 (the
 *                   query, not the key, at the chosen position; coords is the
 *                   fixed coordinate selection P^{l,h}).
 *   q      : [L, H, N, d] in_dtype view;  d_ch : [L, H, N] fp32 (la_notebank_scores)
 *   coords : [L, H, 16] int32, each in [0, d);  spans : [n_notes, 2] int64
 *   t_star : [n_notes, L, H] int32;  rho : [n_notes, L, H, 16] bf16
 * All device memory.  A span outside [0, N) or of length < 1, or a coordinate
 * outside [0, d), writes t_star = -1 and a zero address for that (note,
 * channel) and sets the device status word (la_device_status reports
 * LA_ERR_INVALID_ARGUMENT). */
typedef struct la_notebank_address_args {
  int64_t L, H, N, d, n_notes;
  la_dtype in_dtype;
  la_tensor q;
  const float* d_ch;
  const int32_t* coords;
  const int64_t* spans;
  int32_t* t_star;
  void* rho;
} la_notebank_address_args;
la_status la_notebank_address(const la_notebank_address_args* args, void* stream);

/* Routing (Eq. (5)).  For channel j and note i:
 *   s[i,j] = max over question tokens tau of <unit(u[j,tau]), unit(rho[i,j])>
 * in fp32 (bf16 inputs converted, then normalised); winner[j] = the first
 * note with the largest s[., j]; votes[i] = number of channels won; top =
 * the at most R notes with votes >= 1 and the most votes (ties to the
 * earlier-inserted note), sorted by positions[] (text order; insertion order
 * when positions is NULL), padded with -1.  n_notes = 0 gives winner = -1.
 *   rho : [n_notes, J, 16] bf16 (notes in insertion order, 16-byte aligned)
 *   u   : [J, n_q, 16] bf16 question features (16-byte aligned), n_q 1..512
 *   positions : [n_notes] int64 or NULL;  s : [n_notes, J] fp32 or NULL
 *   winner : [J] int32;  votes : [n_notes] int32;  top : [R] int32 (R 1..64)
 * All device memory. */
typedef struct la_notebank_route_args {
  int64_t n_notes, J, n_q, R;
  const void* rho;
  const void* u;
  const int64_t* positions;
  float* s;
  int32_t* winner;
  int32_t* votes;
  int32_t* top;
} la_notebank_route_args;
la_status la_notebank_route(const la_notebank_route_args* args, void* stream);

/* Synchronises `stream`, then reports (and clears when `clear` != 0) the
 * device-side status word: LA_ERR_TIMEOUT when a bounded wait expired,
 * LA_ERR_INVALID_ARGUMENT when la_state_gather skipped an out-of-range
 * index, la_swa_decode_step met a negative position or la_notebank_address
 * a bad span or coordinate, else LA_OK; LA_ERR_CUDA if the synchronisation
 * failed. */
la_status la_device_status(void* stream, int clear);

/* Self-test of the bounded-wait error path (infrastructure; the pages have no
 * counterpart).  Launches one thread on `stream` that waits on a shared-memory
 * barrier with the same bounded wait the tensor-core kernels use.  With
 * arrive == 0 nothing ever arrives, so the wait gives up after limit_ns and
 * sets the device status word (la_device_status then reports
 * LA_ERR_TIMEOUT); with arrive != 0 the thread arrives itself and the wait
 * completes at once.  No fault, trap or unbounded wait is involved, and the
 * context stays usable.  limit_ns must lie in [1e6, 2e9]; otherwise
 * LA_ERR_INVALID_ARGUMENT and nothing is launched. */
la_status la_selftest_bounded_wait(int arrive, int64_t limit_ns, void* stream);

/* Static description of a status code; never NULL. */
const char* la_status_string(la_status status);

/* LA_ABI_VERSION of the built library. */
int la_abi_version(void);

/* The cudaError_t value (as an int) behind the most recent LA_ERR_CUDA that a
 * call of this library returned to the calling thread; 0 if there was none.
 * Thread-local, so calls from other threads do not overwrite it. */
int la_last_cuda_error(void);

/* The CUDA runtime's name of a cudaError_t value (e.g. from
 * la_last_cuda_error), for callers that do not link the CUDA runtime
 * themselves; never NULL. */
const char* la_cuda_error_name(int code);

#ifdef __cplusplus
}
#endif

#endif /* LA_H */
