/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) speculative-decoding verify step.
 *
 * What the call computes.  A target model has scored a block of drafted
 * tokens in one forward pass; this library turns the target logits and the
 * draft logits into the tokens that are kept.  The rules come from the
 * source pages:
 *   - draft -> verify -> accept/reject: accept drafted tokens from the first
 *     one while the check passes, resample one token at the first failure,
 *     drop every later candidate, and emit one extra target token when the
 *     whole block passes ("DeepSeek DSpark speculative decoding" tutorial,
 *     section "推测解码的两步流程"; the DSpine page, section "原理");
 *   - the check is lossless rejection sampling (DFlash/Spec V2 page, A3, and
 *     its citation of Leviathan et al.; DSpark tutorial, FAQ):
 *     accept x_j iff u_j * p_d(x_j) < p_t(x_j); the replacement is drawn from
 *     max(0, p_t - p_d) renormalised; the bonus token from p_t;
 *   - greedy decoding accepts x_j iff it equals the target argmax (DFlash
 *     page, A4: greedy evaluations);
 *   - confidence label c*_j = 1 - 1/2 * ||p_d,j - p_t,j||_1 for every drafted
 *     position (DSpark tutorial, section "置信度预测头");
 *   - ragged per-request verify length l_r (DSpark tutorial, section
 *     "硬件感知前缀调度器"); block 16 = 1 start token + 15 guesses (DSpine
 *     page, section "这份权重是什么");
 *   - temperature, top_k, top_p processing of both models (DSpine page,
 *     section "加速效果": T 1.0, top_p 0.95, top_k 20).
 * Where the pages leave a step open, this library reads it as follows (the
 * CPU oracle reads it the same way): filter order temperature -> top-k ->
 * renormalise -> top-p (the shortest prefix reaching top_p) -> renormalise;
 * ties broken by (value desc, id asc), -0 and +0 being one value; inverse
 * CDF over ascending ids with a strict ">"; one uniform per target row; a
 * residual mass max(0, p_t - p_d) that is zero up to fp32 rounding (at most
 * 2^-21) falls back to p_t.
 *
 * Layout.  B requests; request r owns l_r target rows (1 <= l_r <= max_len):
 * rows row_offsets[r] .. row_offsets[r] + l_r - 1 of target_logits, where
 * target row j < l_r - 1 scores drafted token j and row l_r - 1 is the bonus
 * row.  Request r owns l_r - 1 draft rows starting at row row_offsets[r] - r
 * of draft_logits.  N_t = row_offsets[B] = sum l_r, N_d = N_t - B.  All
 * logits are row-major with row stride V elements.
 *
 * Ownership and memory.  The caller owns every buffer.  The library
 * allocates nothing: scratch lives in the caller's workspace (size from
 * spec_verify_workspace_size), which must be zeroed once before its first
 * use and can then be reused by any number of calls (the cross-CTA exchange
 * tags every word with a per-call tag; zero is never a tag).  Device pointers
 * must be device memory of the current CUDA device.  The logits base
 * pointers must be 16-byte aligned; other device pointers 4-byte aligned;
 * the workspace 256-byte aligned.  The kernels read the 16-byte blocks that
 * cover each logits row, up to 15 bytes past the end of the last row when
 * V * element size is not a multiple of 16.
 *
 * Streams.  Every call only enqueues work on `stream` (a cudaStream_t; NULL
 * is the legacy default stream) and returns without synchronising the host.
 * Host-visible argument errors are returned before anything is enqueued.
 * Data-dependent problems are OR-ed into *dev_error on the device (never a
 * trap); outputs of a request whose data raised a flag are unspecified.
 * The caller zeroes *dev_error before the call if it wants this call's
 * flags only.  Calls that share a workspace must be ordered on the GPU.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* dtype of both logits buffers */
#define SV_BF16 0 /* bfloat16, 2 bytes */
#define SV_FP32 1 /* float32, 4 bytes */

/* verify mode */
#define SV_GREEDY 0
#define SV_SAMPLE 1

/* host status codes (return values) */
#define SV_OK 0
#define SV_ERR_ARG (-1)         /* null/misaligned pointer, bad size or parameter */
#define SV_ERR_DTYPE (-2)       /* dtype is neither SV_BF16 nor SV_FP32 */
#define SV_ERR_CUDA (-3)        /* a CUDA runtime call or a launch failed */
#define SV_ERR_UNSUPPORTED (-4) /* a shape the kernels do not take */
#define SV_ERR_WORKSPACE (-5)   /* workspace missing, misaligned or too small */
#define SV_ERR_TOO_LARGE (-6)   /* spec_verify_static: more than SV_STATIC_MAX_ROWS rows */

/* device error bits OR-ed into *dev_error */
#define SV_DEVERR_NAN 1     /* a row holds NaN or +inf, or is entirely -inf */
#define SV_DEVERR_TOKEN 2   /* a drafted token is outside [0, V) */
#define SV_DEVERR_LEN 4     /* l_r outside [1, max_len] or row_offsets inconsistent */
#define SV_DEVERR_TIMEOUT 8 /* a bounded device wait gave up */

/* limits */
#define SV_MAX_LEN 256       /* largest accepted max_len */
#define SV_MAX_FILTER_K 64   /* largest kept set of the small kept-set path */
#define SV_STATIC_MAX_ROWS 4096 /* largest n_target_rows of spec_verify_static */

/*
 * Bytes of workspace a call with these sizes needs (a multiple of 256).
 * Pure host function; touches no device.
 */
size_t spec_verify_workspace_size(int32_t B, int32_t n_target_rows);

/*
 * The verify step: the work of spec_verify_rows followed by that of
 * spec_verify_finalize on the same stream.  Unfiltered calls take one
 * launch: the CTAs of the rows kernel finish the requests (the phase-2 work)
 * themselves once their own slices are done and the rows of the request are
 * complete everywhere.  Filtered calls take the two kernels.
 *
 *  target_logits  [N_t, V] device, dtype; 16-byte aligned base.
 *  draft_logits   [N_d, V] device, dtype; may be NULL when N_d == 0.
 *  draft_tokens   [N_d] int32 device: drafted token of each draft row.
 *  uniforms       [N_t] float32 device, values in [0, 1): u of target row
 *                 off_r + j tests drafted token j (j < l_r - 1); the one of
 *                 row off_r + l_r - 1 drives the replacement / bonus draw.
 *  verify_lens    [B] int32 device: l_r.
 *  row_offsets    [B+1] int32 device: prefix sums of l_r, row_offsets[0] = 0.
 *  B, V           > 0.
 *  n_target_rows  N_t on the host (must equal row_offsets[B]; checked on
 *                 the device, SV_DEVERR_LEN).
 *  max_len        host upper bound of every l_r, 1..SV_MAX_LEN.
 *  dtype          SV_BF16 or SV_FP32.
 *  temperature    T > 0 (required in sampling mode and whenever out_conf or
 *                 out_row_stats is requested; otherwise ignored).
 *  top_k          <= 0 or >= V: off.  Else keep the top_k tokens.
 *  top_p          in (0, 1]; 1 = off.  Filtered calls whose kept set is at
 *                 most SV_MAX_FILTER_K tokens (top_k <= 64 on) run the small
 *                 kept-set path: one pass per row selects the set exactly,
 *                 then one CTA per request decides on it.  Larger kept
 *                 sets (top_k above 64, or top_p over the whole vocabulary)
 *                 run the general path: per row a search over weight bins
 *                 and key digits with exact fixed-point mass sums finds the
 *                 kept set's threshold, then one CTA per request decides
 *                 and draws.  The general path takes V up to 2^21 (else
 *                 SV_ERR_UNSUPPORTED).
 *  mode           SV_GREEDY or SV_SAMPLE.
 *  out_tokens     [N_t] int32 device: for request r, entries off_r .. off_r
 *                 + a_r - 1 = accepted drafts, entry off_r + a_r = the final
 *                 (replacement, bonus or greedy) token, later entries -1.
 *  out_accept_len [B] int32 device: a_r in [0, l_r - 1].
 *  out_conf       [N_d] float32 device or NULL: c* per draft row.
 *  out_row_stats  [N_t + N_d][3] float32 device or NULL: per row (target
 *                 rows first, then draft rows) m = max logit / T, Z = sum
 *                 over the kept set of exp(logit / T - m), argmax (lowest
 *                 id; the int32 bit pattern stored in the float slot).
 *  dev_error      [1] int32 device or NULL: device error bits (see above).
 *  workspace      device scratch of workspace_bytes >= spec_verify_workspace_size.
 *  stream         cudaStream_t.
 * Returns SV_OK or a negative SV_ERR_* code.
 */
int spec_verify(const void* target_logits, const void* draft_logits,
                const int32_t* draft_tokens, const float* uniforms,
                const int32_t* verify_lens, const int32_t* row_offsets,
                int32_t B, int32_t V, int32_t n_target_rows, int32_t max_len,
                int32_t dtype, float temperature, int32_t top_k, float top_p, int32_t mode,
                int32_t* out_tokens, int32_t* out_accept_len, float* out_conf,
                float* out_row_stats, int32_t* dev_error,
                void* workspace, size_t workspace_bytes, void* stream);

/*
 * Phase 1 of spec_verify (same arguments; out_tokens, out_accept_len and
 * out_conf are not touched).  Unfiltered: one persistent cooperative grid
 * (one CTA per SM) streams every target row and its draft partner from HBM
 * once, slice by slice through shared memory; the CTAs holding the slices of
 * a row exchange partial statistics through the workspace, and the
 * per-row statistics, accept decisions and per-slice label partials go to
 * the workspace (row statistics also to out_row_stats when given).  In
 * unfiltered sampling mode the per-slice sums of min(p_t, p_d) are formed
 * even without out_conf: the final draw picks its slice from them.
 * Filtered: one CTA per row selects the kept set into the workspace.  This
 * is the bandwidth-bound phase.
 */
int spec_verify_rows(const void* target_logits, const void* draft_logits,
                     const int32_t* draft_tokens, const float* uniforms,
                     const int32_t* verify_lens, const int32_t* row_offsets,
                     int32_t B, int32_t V, int32_t n_target_rows, int32_t max_len,
                     int32_t dtype, float temperature, int32_t top_k, float top_p, int32_t mode,
                     int32_t* out_tokens, int32_t* out_accept_len, float* out_conf,
                     float* out_row_stats, int32_t* dev_error,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * Phase 2 of spec_verify (same arguments).  Per request: the first-rejection
 * scan over the accept decisions left in the workspace by phase 1, the c*
 * labels (sums of the per-slice partials, or over the kept sets), then the
 * final token -- in unfiltered sampling mode an inverse-CDF draw that picks
 * the vocabulary slice from the per-slice masses phase 1 left in the
 * workspace and re-reads only that slice of the rejected row pair (or of the
 * bonus row) from HBM -- and the outputs.  Must run after spec_verify_rows
 * with identical arguments and workspace; kernels launched between the two
 * on the stream must not write the workspace.  (spec_verify launches this
 * phase so that it overlaps the end of phase 1.)
 */
int spec_verify_finalize(const void* target_logits, const void* draft_logits,
                         const int32_t* draft_tokens, const float* uniforms,
                         const int32_t* verify_lens, const int32_t* row_offsets,
                         int32_t B, int32_t V, int32_t n_target_rows, int32_t max_len,
                         int32_t dtype, float temperature, int32_t top_k, float top_p,
                         int32_t mode, int32_t* out_tokens, int32_t* out_accept_len,
                         float* out_conf, float* out_row_stats, int32_t* dev_error,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * spec_verify without a workspace argument, for callers that cannot allocate
 * device memory when they verify (a plain-C host loop without a caching
 * allocator, where cudaMalloc / cudaFree would synchronise the device every
 * step; a process whose memory is committed up front to other pools).  The
 * source pages have no counterpart of this call: it is an interface
 * convenience, and computes exactly what spec_verify computes.
 *
 * Scratch is a file-scope device array of this library sized for
 * SV_STATIC_MAX_ROWS target rows (about 21.9 MB of device memory, reserved
 * when the library's module is loaded on a device).  Nothing is allocated by
 * the call.  n_target_rows > SV_STATIC_MAX_ROWS returns SV_ERR_TOO_LARGE
 * before anything is enqueued.
 *
 * The first call on a device (with that device current) looks up the
 * array's address and enqueues a clear of it on `stream`; make that first
 * call before capturing any stream into a CUDA graph.  The array is shared by
 * every call on the device: calls whose GPU work can overlap (different
 * streams without ordering, concurrent host threads) race on it and must be
 * serialised by the caller.  All other arguments, outputs and errors are as
 * for spec_verify.
 */
int spec_verify_static(const void* target_logits, const void* draft_logits,
                       const int32_t* draft_tokens, const float* uniforms,
                       const int32_t* verify_lens, const int32_t* row_offsets,
                       int32_t B, int32_t V, int32_t n_target_rows, int32_t max_len,
                       int32_t dtype, float temperature, int32_t top_k, float top_p,
                       int32_t mode, int32_t* out_tokens, int32_t* out_accept_len,
                       float* out_conf, float* out_row_stats, int32_t* dev_error,
                       void* stream);

/*
 * DSpark hardware-aware prefix scheduler ("DeepSeek DSpark speculative
 * decoding" tutorial, section "硬件感知前缀调度器"): the verify lengths l_r
 * of a pool of B requests for the next step.  Drafted position k of request
 * r carries a conditional survival probability c_{r,k} (section "置信度预测头";
 * the verify step's own labels c* serve where no confidence head exists);
 * its prefix survival is S_{r,k} = prod_{i<=k} c_{r,i}.  Every request starts
 * at l_r = 1; candidates are added best S first (equal S: lower r, then
 * lower k) while Theta = tau * SPS(B) strictly rises, with tau =
 * sum_r (1 + sum_{k < l_r - 1} S_{r,k}) the expected tokens of the step and
 * B = sum_r l_r; the scan also stops when the table has no SPS(B + 1).  One
 * CTA, float64 throughout.
 *
 *  conf       [B][K] float32 device, row-major: c_{r,k} for k = 0..K-1 (the
 *             first drafted position first); clamped to [0, 1], NaN as 0.
 *             May be NULL when K == 0.
 *  B, K       1 <= B, 0 <= K, B * K <= SV_SCHEDULE_MAX_CANDIDATES
 *             (else SV_ERR_UNSUPPORTED).
 *  sps        [n_sps] float64 device: SPS(b) for batch b = 0..n_sps-1 (the
 *             target's steps per second at b verified tokens); n_sps > B.
 *  out_lens   [B] int32 device: l_r in [1, K + 1].
 *  out_theta  [2] float64 device or NULL: Theta of the schedule and the
 *             number of candidates added.
 *  stream     cudaStream_t; stream-ordered, no host synchronisation.
 * Returns SV_OK, SV_ERR_ARG (null, misaligned or inconsistent arguments),
 * SV_ERR_UNSUPPORTED or SV_ERR_CUDA.
 */
#define SV_SCHEDULE_MAX_CANDIDATES 8192
int spec_verify_schedule(const float* conf, int32_t B, int32_t K, const double* sps,
                         int32_t n_sps, int32_t* out_lens, double* out_theta, void* stream);

/*
 * Tuning and testing hook (the pages have no counterpart): sets one
 * process-wide knob of the rows kernel for every later call; value < 0
 * restores its default.  The defaults are the shipped configuration; the
 * library reads no environment variable.
 *   SV_TUNE_SLICE        target slice length in elements (0 or default: 22000
 *                        bytes' worth), up to 2^24
 *   SV_TUNE_STAGES       most shared-memory stages, 4..6
 *   SV_TUNE_WARPS        consumer warps, 16 or 24
 *   SV_TUNE_PASS1_WARPS  consumer warps on pass 1 when labels are on, 0 .. 23;
 *                        0 or default: half, or 11 of 16 when the exact
 *                        row maximum is tracked (greedy, row statistics)
 *   SV_TUNE_POLL_NS      sleep between polls of another CTA's words, 0..10000
 *                        (default 64 ns)
 *   SV_TUNE_XWAIT_NS     limit of a wait on words that other CTAs of the
 *                        same launch publish, 0..200000000 (default 200 ms);
 *                        a wait that reaches it gives up, the call raises
 *                        SV_DEVERR_TIMEOUT and its outputs are unspecified
 *                        (waits on a CTA's own copies keep their own limit).
 * Host only; takes effect on the next call.  Returns SV_OK or SV_ERR_ARG
 * (unknown knob, value out of range).
 */
#define SV_TUNE_SLICE 0
#define SV_TUNE_STAGES 1
#define SV_TUNE_WARPS 2
#define SV_TUNE_PASS1_WARPS 3
#define SV_TUNE_POLL_NS 4
#define SV_TUNE_XWAIT_NS 5
int spec_verify_set_tuning(int32_t knob, int64_t value);

/* Static text for a status code (host). */
const char* spec_verify_status_string(int status);

/* Number of vocabulary slices (work units, each held by one CTA) into which
 * the rows kernel cuts a row of V logits of this dtype on the current
 * device, or a negative SV_ERR_* code. */
int spec_verify_slices_per_row(int32_t V, int32_t dtype, int32_t top_k, float top_p);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
