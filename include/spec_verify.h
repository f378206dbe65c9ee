/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) verification step of speculative sampling.
 *
 * The operation is the target-side modified rejection sampling of
 * "Accelerating Large Language Model Decoding with Speculative Sampling"
 * (Chen et al., DeepMind), as summarised by the wikillm.com paper card:
 *   - §4.2 "Decoding transforms": the temperature transform softmax(l / T) is
 *     applied to both the target rows q and the draft rows p before anything else;
 *   - §4.2 "Modified rejection sampling" and Algorithm 2 step 3: draft token
 *     x~_t is accepted, left to right, while u_t < min(1, q(x~_t) / p(x~_t));
 *     at the first rejection one token is drawn from the normalised residual
 *     (q - p)_+ = max(0, q - p) / sum max(0, q - p), and the scan stops;
 *   - Algorithm 2 step 4 and the card's Pitfalls ("Bonus-token typo"): if all K
 *     drafts are accepted, one bonus token is drawn from the (K+1)-th target row;
 *   - the card's Pitfalls ("The residual distribution needs care"): a residual
 *     that sums to zero falls back to q itself.
 * Each sequence therefore emits between 1 and K+1 tokens (§4.2).
 *
 * Conventions the pages leave open, fixed here:
 *   - uniforms[b, t], t < K, drives the test of draft t; uniforms[b, K] drives
 *     the residual draw; uniforms[b, K+1] drives the bonus draw;
 *   - the test is strict (u < min(1, q/p)); p(x~) = 0 with q(x~) > 0 accepts,
 *     q(x~) = 0 rejects;
 *   - a draw from weights w with uniform u is the inverse CDF over ascending
 *     token id: the smallest i with w_0 + ... + w_i > u * sum(w); when no
 *     such i exists (u = 1) the largest i with w_i > 0 is taken;
 *   - -inf logits are masked entries (probability 0).
 *
 * All entry points are plain C. Pointers marked "device" must point to memory
 * of the current CUDA device; the library never allocates, frees or keeps
 * pointers between calls. Work is enqueued on `stream` (a cudaStream_t passed
 * as void*; NULL means the legacy default stream) and runs asynchronously.
 *
 * A call enqueues a memset of the workspace's control block and then either
 *   - two kernels: the streaming kernel, then the draw kernel as its
 *     programmatic dependent (launched while the streaming grid drains, and
 *     waiting on the device for it to complete); or, for calls streaming
 *     between 16 MiB and 1 GiB of logits,
 *   - one fused kernel whose CTAs take tickets: streaming work first, then the
 *     draw of each sequence, which waits on the device for that sequence's
 *     plan. The wait is bounded: after 200 ms it sets SV_DEV_TIMEOUT and the
 *     kernel winds down.
 * Make the first call on a device before capturing a stream into a CUDA graph.
 */
#ifndef SPEC_VERIFY_H_
#define SPEC_VERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Logit element types. */
enum {
  SV_BF16 = 0, /* bfloat16 */
  SV_F32 = 1   /* IEEE fp32 */
};

/* Host-side return codes (no work is enqueued when one of these is returned). */
enum {
  SV_OK = 0,
  SV_ERR_NULL = 1,        /* a required pointer is NULL */
  SV_ERR_SHAPE = 2,       /* B < 0, K outside [1, 64], V outside [1, 2^31 - 1], or sizes overflow */
  SV_ERR_TEMPERATURE = 3, /* temperature not finite or not > 0 */
  SV_ERR_DTYPE = 4,       /* dtype is neither SV_BF16 nor SV_F32 */
  SV_ERR_ALIGN = 5,       /* a pointer is not aligned to its element (workspace: 256 bytes) */
  SV_ERR_WORKSPACE = 6,   /* workspace_bytes below sv_workspace_size(), or staging too small */
  SV_ERR_CUDA = 7,        /* a CUDA runtime call failed */
  SV_ERR_SCRATCH_LIMIT = 8 /* spec_verify_static: the problem needs more than its fixed scratch */
};

/* Size of the fixed device scratch array behind spec_verify_static. */
#define SV_STATIC_SCRATCH_BYTES (8u << 20)

/* Device-side status bits, OR-ed into the status word of the workspace. A
 * sequence that raises one of the first four gets out_tokens[b, :] = -1 and
 * n_accepted[b] = -1; other sequences are unaffected. */
enum {
  SV_DEV_TOKEN_RANGE = 16,   /* a draft token outside [0, V) */
  SV_DEV_NONFINITE = 32,     /* a logit row holds NaN or +inf */
  SV_DEV_EMPTY_ROW = 64,     /* a logit row is entirely -inf */
  SV_DEV_UNIFORM_RANGE = 128,/* a uniform is NaN or outside [0, 1] */
  SV_DEV_TIMEOUT = 256       /* a bounded wait in the fused kernel ran out (results invalid) */
};

/* Bytes of device workspace spec_verify needs for this problem size; 0 for an
 * invalid size. The workspace is scratch owned by the caller; it must be
 * 256-byte aligned and must not be shared by calls in flight at the same time.
 * Pure host function: it touches no device. */
size_t sv_workspace_size(int B, int K, int V, int dtype);

/* One verification step for a batch of B independent sequences.
 *
 *   target_logits  device, [B, K+1, V] row-major, dtype; row t of sequence b is
 *                  q(. | prefix, x~_1..x~_t), t = 0..K (the target's K+1 outputs)
 *   draft_logits   device, [B, K, V] row-major, dtype; row t is p(. | prefix, x~_1..x~_t)
 *   draft_tokens   device, [B, K] int32, the drafted tokens x~ (expected in [0, V))
 *   uniforms       device, [B, K+2] fp32, expected in [0, 1)
 *   B, K, V        batch, lookahead (1..64), vocabulary (1..2^31-1)
 *   dtype          SV_BF16 or SV_F32
 *   temperature    T > 0, applied to both p and q (softmax(l / T))
 *   out_tokens     device, [B, K+1] int32 (written): accepted drafts, then the
 *                  drawn token, then -1 padding
 *   n_accepted     device, [B] int32 (written): accepted drafts per sequence, 0..K
 *   workspace      device, sv_workspace_size(B, K, V, dtype) bytes, 256-byte aligned
 *
 * Inputs are read only. Base pointers of the logits need only element
 * alignment; 16-byte aligned bases with V * sizeof(dtype) a multiple of 16
 * take the 16-byte vector-load path. Returns SV_OK once the work is enqueued, or
 * a host-side error code with nothing enqueued. B == 0 returns SV_OK at once.
 * Device-side problems are reported through sv_read_device_status(). */
int spec_verify(const void* target_logits, const void* draft_logits,
                const int32_t* draft_tokens, const float* uniforms, int B, int K, int V,
                int dtype, float temperature, int32_t* out_tokens, int32_t* n_accepted,
                void* workspace, size_t workspace_bytes, void* stream);

/* spec_verify plus intermediate values for inspection (each pointer may be NULL;
 * all are fp64 device arrays, NaN for every entry of a failed sequence):
 *   row_lse      [B, 2K+1]: log sum_i exp(l_i / T) per row, target rows 0..K
 *                first, then draft rows 0..K-1 (from the streaming pass)
 *   thresholds   [B, K]: min(1, q(x~_t)/p(x~_t)) for every t, the acceptance
 *                test's threshold (card, §4.2 "Modified rejection sampling")
 *   sample_prob  [B]: normalised weight of the drawn token in the
 *                distribution it was drawn from (residual, fallback q, or bonus q)
 *   row_max      [B, 2K+1]: max_i l_i / T per row, same row order as row_lse
 *   ratios       [B, K]: the ratio q(x~_t)/p(x~_t) itself, not clamped at 1;
 *                +inf where p(x~_t) = 0 < q(x~_t), 0 where q(x~_t) = 0
 * Every t < K gets a threshold and a ratio, also past the first rejection. */
int spec_verify_debug(const void* target_logits, const void* draft_logits,
                      const int32_t* draft_tokens, const float* uniforms, int B, int K, int V,
                      int dtype, float temperature, int32_t* out_tokens, int32_t* n_accepted,
                      void* workspace, size_t workspace_bytes, void* stream, double* row_lse,
                      double* thresholds, double* sample_prob, double* row_max,
                      double* ratios);

/* spec_verify that also records three caller-owned CUDA events (cudaEvent_t
 * passed as void*, created with timing enabled) on `stream`: `ev_start` before
 * the first kernel, `ev_stats_done` between the streaming row-statistics
 * kernel and the draw kernel (after the fused kernel, when that one runs),
 * `ev_end` after the last kernel. Elapsed times between them time the
 * streaming pass and the draw. With `ev_stats_done` set the draw kernel is an
 * ordinary launch rather than a programmatic dependent, so the pair runs back
 * to back without overlap. Any event may be NULL. */
int spec_verify_profiled(const void* target_logits, const void* draft_logits,
                         const int32_t* draft_tokens, const float* uniforms, int B, int K, int V,
                         int dtype, float temperature, int32_t* out_tokens, int32_t* n_accepted,
                         void* workspace, size_t workspace_bytes, void* stream, void* ev_start,
                         void* ev_stats_done, void* ev_end);

/* Bytes of device staging memory spec_verify_host needs (inputs and outputs). */
size_t sv_staging_size(int B, int K, int V, int dtype);

/* spec_verify on HOST buffers: copies the four inputs host -> device into
 * `staging` (device, sv_staging_size() bytes, 256-byte aligned), runs the step,
 * copies out_tokens / n_accepted back to the host buffers and synchronises
 * `stream`. Pinned host memory gives the fastest copies. Returns a host-side
 * error code, or else the device status bits of this call (0 = all ok). */
int spec_verify_host(const void* h_target_logits, const void* h_draft_logits,
                     const int32_t* h_draft_tokens, const float* h_uniforms, int B, int K,
                     int V, int dtype, float temperature, int32_t* h_out_tokens,
                     int32_t* h_n_accepted, void* staging, size_t staging_bytes,
                     void* workspace, size_t workspace_bytes, void* stream);

/* spec_verify_host without the wait: the copies and the step are enqueued on
 * `stream`, and the call returns SV_OK (or a host-side error code, with
 * nothing enqueued) at once. h_out_tokens / h_n_accepted hold the results
 * once `stream` has reached this point (cudaStreamSynchronize, or an event
 * recorded after the call); the device status bits are read with
 * sv_read_device_status(workspace, stream). The host input buffers must stay
 * unchanged until then, and pinned host memory is needed for the copies to be
 * asynchronous. A serving loop overlaps the copies of one step with the
 * kernels of the previous one by giving consecutive calls different streams,
 * staging buffers and workspaces. */
int spec_verify_host_async(const void* h_target_logits, const void* h_draft_logits,
                           const int32_t* h_draft_tokens, const float* h_uniforms, int B, int K,
                           int V, int dtype, float temperature, int32_t* h_out_tokens,
                           int32_t* h_n_accepted, void* staging, size_t staging_bytes,
                           void* workspace, size_t workspace_bytes, void* stream);

/* spec_verify for callers that cannot allocate device memory (the paper has no
 * counterpart to this; it is a property of this library only). Some callers
 * cannot provide a workspace: code running during stream capture in the global
 * or thread-local mode (where cudaMalloc is not allowed), plugins whose device
 * memory must all come from a host framework's pool, and latency-critical loops
 * where cudaMalloc may stall the device. This entry point allocates nothing and
 * takes no workspace: its scratch is one fixed array of SV_STATIC_SCRATCH_BYTES
 * (8 MiB) of device memory inside the library, which every GPU that loads the
 * library holds until the process exits.
 *
 * Arguments, layouts and results are those of spec_verify. Problems whose
 * sv_workspace_size exceeds SV_STATIC_SCRATCH_BYTES are rejected with
 * SV_ERR_SCRATCH_LIMIT and nothing is enqueued. Every call on a device shares
 * that device's array, which keeps the previous call's contents; each call
 * clears what must start at zero itself. Calls that overlap on the GPU (on
 * different streams, or from different threads) race on the array and must
 * be serialised by the caller. Outside stream capture every call looks up the
 * array's device address in the current context (cudaGetSymbolAddress); a
 * call made while `stream` is being captured reuses the address of the last
 * call on that device, so make one call outside capture first (and again
 * after cudaDeviceReset or a change of context). Device status bits are not
 * readable for these calls (there is no workspace to read them from): a
 * sequence that failed shows -1 in all its outputs and n_accepted = -1, and a
 * draw that did not complete shows -1 at position n_accepted. */
int spec_verify_static(const void* target_logits, const void* draft_logits,
                       const int32_t* draft_tokens, const float* uniforms, int B, int K, int V,
                       int dtype, float temperature, int32_t* out_tokens, int32_t* n_accepted,
                       void* stream);

/* ---------------------------------------------------------------- draft-side sampler
 *
 * Step 1 of the card's Algorithm 2: the draft model's tokens x~_t ~ p(.),
 * drawn from the transformed distribution p = softmax(l / T) ("Accelerating
 * Large Language Model Decoding with Speculative Sampling", wikillm.com paper
 * card, §4.2 "Decoding transforms", and the Pitfalls item on transformed
 * distributions): the draws that feed the verifier use the very distribution
 * the verifier's ratios and residual use. One token per row, by
 * the inverse-CDF convention above with the row's uniform; rows are
 * independent, so a caller samples one draft position for a batch per call
 * (or several positions at once when their logits are already known). */

/* Bytes of device workspace spec_draft_sample needs for N rows of V elements;
 * 0 for invalid sizes. Pure host function. */
size_t sv_sample_workspace_size(int N, int V, int dtype);

/* One token per row:
 *   logits       device, [N, V] row-major, dtype elements (element-aligned;
 *                16-byte aligned with V * sizeof(dtype) a multiple of 16 takes
 *                the 16-byte vector-load path)
 *   uniforms     device, [N] fp32: the uniform of each row's draw
 *   temperature  T > 0, finite (fp32)
 *   out_tokens   device, [N] int32: the drawn token, or -1 for a failed row
 *   sample_prob  device, [N] fp64, may be NULL: probability of the drawn token
 *   workspace    device, sv_sample_workspace_size() bytes, 256-byte aligned,
 *                caller-owned; one call at a time per workspace
 * A row fails (token -1, status bit) if it holds NaN or +inf, is entirely
 * -inf, or its uniform is NaN or outside [0, 1]; other rows are unaffected.
 * Returns SV_OK once the work is enqueued on `stream`, or a host-side error
 * code with nothing enqueued; N == 0 returns SV_OK at once. Device status bits
 * are read with sv_read_device_status(). */
int spec_draft_sample(const void* logits, const float* uniforms, int N, int V, int dtype,
                      float temperature, int32_t* out_tokens, double* sample_prob,
                      void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------- greedy mode
 *
 * Verification at T = 0. The paper reports greedy results but does not state
 * the rule; the card's Pitfalls ("Greedy mode is not specified") infer it by
 * applying the general rule to one-hot distributions: accept while the draft's
 * greedy token equals the target's, otherwise emit the target's greedy token.
 * Here: x~_t is accepted while it equals argmax q_t (ties go to the smallest
 * token id; -inf entries are masked); at the first mismatch j, argmax q_j is
 * emitted; if all K match, argmax q_K (the bonus token). No uniforms, no
 * temperature and no draft logits are read; the target rows are read once. */

/* Bytes of device workspace spec_verify_greedy needs; 0 for invalid sizes. */
size_t sv_greedy_workspace_size(int B, int K, int V, int dtype);

/* Greedy verification: target_logits, draft_tokens, out_tokens, n_accepted,
 * workspace and stream as for spec_verify (out_tokens holds the accepted
 * drafts, then the emitted token, then -1 padding). A sequence fails (all -1,
 * status bit) if a target row holds NaN or +inf or is entirely -inf, or a
 * draft token lies outside [0, V). Returns SV_OK once enqueued, or a host-side
 * error code with nothing enqueued; B == 0 returns SV_OK at once. */
int spec_verify_greedy(const void* target_logits, const int32_t* draft_tokens, int B, int K,
                       int V, int dtype, int32_t* out_tokens, int32_t* n_accepted,
                       void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------- top-k filtered verification
 *
 * The card's §4.2 "Decoding transforms": top-k is applied to both p and q,
 * and the rejection scheme then runs on the filtered distributions (the
 * Pitfalls section: the same transformed distributions are used for the
 * thresholds, the residual and the bonus draw). Each of the 2K+1 rows keeps
 * its top_k largest logits; ties go to the smaller token id and -0.0 equals
 * +0.0; the other entries count as -inf. The kept entries' softmax at
 * temperature T, the thresholds min(1, q/p), the residual max(0, q - p) and
 * the inverse-CDF draws are those of spec_verify, on the filtered rows. */

/* Bytes of device workspace spec_verify_topk needs; 0 for invalid sizes.
 * top_k >= V keeps every entry and needs sv_workspace_size(B, K, V, dtype). */
size_t sv_topk_workspace_size(int B, int K, int V, int dtype, int top_k);

/* Top-k filtered verification. Arguments as for spec_verify, plus
 *   top_k  entries kept per row: 1 <= top_k <= 256, or top_k >= V (every
 *          entry kept: the call is spec_verify's); other values return
 *          SV_ERR_SHAPE
 * Each row is reduced to its top_k entries in one pass over it (one CTA per
 * row: a running threshold and a candidate buffer in shared memory, with an
 * exact radix select over the row for adversarial orders), their softmax is
 * taken in fp64, and the verification runs on the kept (token id,
 * probability) pairs (one CTA per sequence): two kernels per call. Failures and status bits as for
 * spec_verify (a row holding +inf or NaN fails its sequence, a row whose kept
 * entries are all -inf is an empty row). Returns SV_OK once enqueued, or a
 * host-side error code with nothing enqueued; B == 0 returns SV_OK at once. */
int spec_verify_topk(const void* target_logits, const void* draft_logits,
                     const int32_t* draft_tokens, const float* uniforms, int B, int K, int V,
                     int dtype, float temperature, int top_k, int32_t* out_tokens,
                     int32_t* n_accepted, void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------- nucleus (top-p) filtered verification
 *
 * The card's §4.2 "Decoding transforms" with the nucleus rule on both p and
 * q: each of the 2K+1 rows keeps the shortest prefix of its entries, ordered
 * by logit (larger first, ties to the smaller token id, -0.0 equal to +0.0),
 * whose probability softmax(l / T) reaches top_p; the other entries count as
 * -inf. The filtered rows are then verified exactly as by spec_verify. */

/* Bytes of device workspace spec_verify_topp needs (spec_verify's, and one
 * 8-byte cut key per row); 0 for invalid sizes. */
size_t sv_topp_workspace_size(int B, int K, int V, int dtype);

/* Nucleus filtered verification. Arguments as for spec_verify, plus
 *   top_p        probability mass kept per row: top_p > 0; top_p >= 1 keeps
 *                every entry (the call is spec_verify's); NaN or top_p <= 0
 *                returns SV_ERR_SHAPE
 *   kept_counts  device, [B, 2K+1] int32, may be NULL: entries kept per row
 *                (target rows 0..K, then draft rows 0..K-1); V for a row that
 *                fails (NaN, +inf or all -inf), which is left as it is
 * Per row, a cut is found without a sort: mass histograms over the scaled
 * distance (m - l) / T of each entry from the row maximum, at finer and finer
 * widths, locate the cut to a bin of at most 1024 entries, whose keys are then
 * searched exactly with their masses (a bin that never gets that small, from
 * heavy ties, is resolved bit by bit over the key). Rows up to 512 KB are held
 * in the shared memory of a thread-block cluster (up to 8 CTAs per row), so
 * each row is read from memory once; longer rows are re-read per pass. Weights
 * are float-float exponentials. The cut also yields each row's kept mass, so
 * the verification (a scan kernel, then the draw) reads the rows unchanged
 * and applies each row's kept set as it loads them: sv_topp_kernels_per_call
 * kernels per call. Returns SV_OK once enqueued, or a host-side error code
 * with nothing enqueued; B == 0 returns SV_OK at once. */
int spec_verify_topp(const void* target_logits, const void* draft_logits,
                     const int32_t* draft_tokens, const float* uniforms, int B, int K, int V,
                     int dtype, float temperature, float top_p, int32_t* out_tokens,
                     int32_t* n_accepted, int32_t* kept_counts, void* workspace,
                     size_t workspace_bytes, void* stream);

/* Reads the device status word of the last call that used `workspace`: waits
 * for `stream`, then stores the OR of the SV_DEV_* bits in *status. */
int sv_read_device_status(const void* workspace, void* stream, int* status);

/* Static description of a return code or device status bit set. */
const char* sv_status_string(int status);

/* Kernels one spec_verify call over these sizes launches (for launch
 * accounting): 1 (the fused kernel) for calls streaming between 16 MiB and
 * 1 GiB; else 2 for calls whose draw needs few chunks (the streaming kernel and
 * a one-launch draw) or 3 (the streaming kernel, the draw's sum kernel and its
 * finish kernel); 0 for invalid sizes or B == 0. */
int sv_kernels_per_call(int B, int K, int V, int dtype);

/* Kernels one spec_verify_topp call with top_p < 1 over these sizes launches:
 * the cut kernel, the scan kernel and the draw (one kernel when the draw
 * needs few chunks, else two), so 3 or 4; 0 for invalid sizes or B == 0. */
int sv_topp_kernels_per_call(int B, int K, int V, int dtype);

/* Test hook: 0 (the default) chooses the kernels by size, 1 forces the kernel
 * pair, 2 forces the fused kernel. Process-wide; for tests that compare the
 * two paths. */
void sv_force_path(int path);

/* Test hook for failure detection: with `on` nonzero, calls never publish
 * their plans' release flag, so on the fused path every draw CTA's bounded
 * wait runs out (200 ms) and the call ends with SV_DEV_TIMEOUT; no GPU fault,
 * and the context stays usable. Process-wide; 0 restores normal calls. */
void sv_test_withhold_plans(int on);

/* ---------------------------------------------------------------- the scoring step's projection
 *
 * Algorithm 2 step 2 of the card: one target call scores the K+1 prefixes
 * (§4.1 "Why it works (conditional scoring)"); the verification then needs,
 * per scored row, only the statistics of the temperature transform (§4.2
 * "Decoding transforms") and the logit at the drafted token (§4.2 "Modified
 * rejection sampling"). This call fuses the model's final projection with
 * those statistics: the logits l = h W^T are formed on the tensor cores
 * (bf16 operands, fp32 accumulation) and reduced on chip, never stored.
 *
 * Bytes of device workspace sv_lmhead_stats needs; 0 for invalid sizes
 * (N < 0, V < 1, D < 8 or not a multiple of 8). Pure host function. */
size_t sv_lmhead_workspace_size(int N, int D, int V);

/* For every row n of the hidden states:
 *   hidden       device, [N, D] bf16, row-major, 16-byte aligned
 *   weight       device, [V, D] bf16, row-major, 16-byte aligned: the
 *                projection's weight, one row per token (l = h W^T)
 *   tokens       device, [N] int32: a token per row, or -1 for none
 *   temperature  T > 0, finite (fp32)
 *   row_max      device, [N] fp64 (written): max_i l_i / T
 *   lse          device, [N] fp64 (written): log sum_i exp(l_i / T)
 *   at           device, [N] fp32 (written): l at tokens[n], NaN where tokens[n]
 *                is outside [0, V)
 *   workspace    device, sv_lmhead_workspace_size() bytes, 256-byte aligned;
 *                its first 4 bytes are the device status word (read with
 *                sv_read_device_status): 32 = a row with a non-finite logit
 *                (its row_max and lse are NaN), 256 = a bounded wait ran out
 * The logits carry fp32 accumulation error: against exact arithmetic, a
 * logit differs by about 2^-24 sqrt(D) times the magnitude of the partial
 * sums. Returns SV_OK once the two kernels are enqueued on `stream`, or a
 * host-side error code with nothing enqueued; N == 0 returns SV_OK at once. */
int sv_lmhead_stats(const void* hidden, const void* weight, const int32_t* tokens, int N, int D,
                    int V, float temperature, double* row_max, double* lse, float* at,
                    void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H_ */
