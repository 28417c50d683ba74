/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) speculative-sampling
 * verification library.
 *
 * One call verifies a batch of B independent requests.  Request b proposed
 * draft tokens y_0..y_{gamma_b-1}; the target model produced gamma_b + 1 logit
 * rows (positions 0..gamma_b) and, for full-q verification, the draft model
 * produced gamma_b logit rows.  The library decides how many draft tokens are
 * accepted and which token is committed after them.
 *
 * Method (tutorial page "5.1 投机解码核心原理", infra-guide):
 *   section 2.1  p_i, q_i are the distributions used for sampling, temperature
 *                applied: p_i = softmax(target_row_i / T_b), same for q_i;
 *   section 3.1  greedy: accept y_i iff y_i = argmax p_i, else emit argmax, stop;
 *   section 3.2  accept y_i iff u_i < min(1, p_i(y_i) / q_i(y_i)); on reject
 *                draw from [p_i - q_i]_+ / sum [p_i - q_i]_+;
 *   section 3.3  one-hot q (draft gives tokens only): accept iff u_i < p_i(y_i);
 *                on reject draw from p_i with y_i removed, renormalised;
 *   section 5.1  stop at the first reject, later candidates are void;
 *   section 5.2  all gamma accepted: one more token from p_gamma (bonus).
 * Draft signals (SpecKV page, draft signal extraction): per draft row
 *   H_i = -sum_v q_i(v) log2 q_i(v) (bits) and c_i = max_v q_i(v); per request
 *   mean_i H_i, max_i H_i, mean_i c_i, min_i c_i over i < gamma_b.
 *
 * Conventions shared by every call
 *   - Index 0-based: target rows i = 0..gamma_b (row gamma_b is the bonus row),
 *     draft rows and draft tokens i = 0..gamma_b-1.  The pages count from 1.
 *   - Layouts are row-major and contiguous:
 *       target_logits [B, G+1, V], draft_logits [B, G, V]  (dtype below),
 *       draft_tokens [B, G] int32, gamma [B] int32 (NULL: every gamma_b = G),
 *       temperature [B] float32 (> 0), uniforms [B, G+1] float32 in [0, 1):
 *       column i < gamma_b drives the test at position i, column G drives the
 *       final draw;
 *       accept_len [B] int32, tokens [B, G+1] int32 (committed tokens
 *       y_0..y_{k-1}, then the drawn token at index k, then -1),
 *       status [B] int32 bitmask (SPEC_ST_*), signals [B, 4] float32
 *       (mean H, max H, mean c, min c), row_signals [B, G, 2] float32
 *       (H_i, c_i), accept_prob [B, G] float32 (a_i for i <= k, NaN after).
 *   - Every pointer except `workspace` sizes is DEVICE memory owned by the
 *     caller.  The library never allocates, frees or synchronises: each call
 *     only enqueues kernels on `stream` and returns.  Outputs are valid once
 *     the stream reaches them.  `stream` may be NULL (legacy default stream).
 *   - Logit rows may hold -inf (a token of probability 0).  NaN or +inf in a
 *     row the method reads, or a row with no finite maximum, is an error.
 *   - Rows past a request's gamma_b, and rows after its first reject (except
 *     draft rows needed for signals), are never read.  Reading stops early:
 *     rows the method does not need may or may not be read; the results do
 *     not depend on which.
 *   - Host return codes (SPEC_OK / SPEC_ERR_*) cover what the host can check
 *     without touching device memory: null required pointers, sizes, dtype,
 *     workspace size.  Nothing is launched when they are not SPEC_OK.
 *   - Problems found on the device are reported per request in `status`.
 *     A request with an error bit other than SPEC_ST_ZERO_RESIDUAL or
 *     SPEC_ST_GUARDED commits nothing: accept_len = 0, tokens all -1,
 *     accept_prob and signals NaN.  Other requests are unaffected.
 *   - Given identical inputs the outputs are bit-identical from call to call.
 *   - Calls that share a workspace must not overlap on the device (enqueue
 *     them on one stream, or give each its own workspace).
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                       /* the CUDA runtime's cudaStream_t */
typedef struct CUstream_st* spec_stream_t;

/* logit dtypes */
enum { SPEC_F32 = 0, SPEC_BF16 = 1 };

/* host return codes */
enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = 1,   /* null pointer, bad size or dtype        */
    SPEC_ERR_WORKSPACE = 2,     /* workspace NULL or smaller than needed  */
    SPEC_ERR_CUDA = 3,          /* a CUDA call or launch failed           */
    SPEC_ERR_UNSUPPORTED = 4    /* device is not sm_103 / sm_100 family   */
};

/* per-request status bits */
enum {
    SPEC_ST_OK = 0,
    SPEC_ST_NONFINITE = 1,       /* NaN / +inf / no finite max in a read row */
    SPEC_ST_BAD_TOKEN = 2,       /* draft token outside [0, V)              */
    SPEC_ST_BAD_GAMMA = 4,       /* gamma_b outside [0, G]                  */
    SPEC_ST_ZERO_RESIDUAL = 8,   /* residual mass rounded to 0: drew from p */
    SPEC_ST_GUARDED = 16,        /* informational: a near-tie draw was taken
                                    again in extended precision; the outputs
                                    are valid                                */
    SPEC_ST_TIMEOUT = 32,        /* an internal wait hit its time limit     */
    SPEC_ST_BAD_TEMPERATURE = 64,/* temperature <= 0 or not finite          */
    SPEC_ST_BAD_UNIFORM = 128    /* a uniform that was used is not in [0,1) */
};

/* Limits checked by the host: 1 <= B <= 65535, 0 <= G <= 31, 2 <= V < 2^28,
 * and the internal work and queue counts (B (2G+1) ceil(V / 16384) chunks,
 * B (4 ceil(V / 4096) + 2 G ceil(V / 16384) + 2) dynamic-queue entries)
 * below 2^31; no device could hold
 * the logits of sizes past those. */
#define SPEC_MAX_B 65535
#define SPEC_MAX_G 31

/* Bytes of device workspace every call with these sizes needs (0 if the
 * sizes are outside the limits).  Pure host function; the workspace holds
 * per-row partial statistics, counters and the row schedule.  It needs no
 * initialisation and no alignment beyond 256 bytes. */
size_t spec_workspace_bytes(int B, int G, int V);

/* Human-readable name of a host return code (SPEC_OK, SPEC_ERR_*). */
const char* spec_status_string(int code);

/* Human-readable name of one per-request status bit (SPEC_ST_*). */
const char* spec_request_status_string(int bit);

/* Number of kernels this host thread has launched through the library. */
uint64_t spec_launch_count(void);

/* Profiling aid.  The next verification call made by this host thread records
 * `begin_event` on its stream just before its verify kernel (the persistent
 * kernel that streams the logits and settles every request) and `end_event`
 * just after it; the hook then
 * clears itself.  Both are cudaEvent_t handles owned by the caller; NULL
 * clears the hook.  The event records sit between two launches of the call,
 * so that call's start-up overlap with the kernel before is lost. */
int spec_profile_next_call(void* begin_event, void* end_event);

/* Testing aid for the timeout path; the method has no counterpart.  Every
 * wait inside a call (for a staged piece of a row, another CTA's partial
 * statistics, a draw's slice sums) gives up after `cycles` SM clock cycles;
 * the request it served then commits nothing and reports SPEC_ST_TIMEOUT,
 * and every other role of the call gives up as soon as it sees that.  The
 * setting applies to calls enqueued afterwards by any host thread;
 * cycles <= 0 restores the default of 4e9 cycles (about 2 s at 2 GHz), which
 * no healthy call comes near.  A low value (1) makes most requests of a call
 * time out; it is meant only for tests of that path.  The wait for a CTA's
 * own copies in flight before it exits always keeps the default.  Returns
 * SPEC_OK. */
int spec_set_wait_limit(long long cycles);

/* Greedy verification (tutorial page, section 3.1).  For i = 0..gamma_b-1:
 * g_i = argmax target row i (lowest index among equal maxima); stop at the
 * first y_i != g_i with k = i and commit g_i; if none, k = gamma_b and commit
 * the argmax of row gamma_b.  Temperature and uniforms are not used. */
int spec_verify_greedy(const void* target_logits, int dtype, int B, int G, int V,
                       const int32_t* draft_tokens, const int32_t* gamma,
                       int32_t* accept_len, int32_t* tokens, int32_t* status,
                       void* workspace, size_t workspace_bytes, spec_stream_t stream);

/* Stochastic verification with full draft distributions (sections 3.2,
 * 4, 5.1, 5.2).  accept_i  <=>  u_i * q_i(y_i) < p_i(y_i).  The final draw is
 * inverse-CDF in ascending token order: with weights w (the residual
 * [p_k - q_k]_+ after a reject at k, else p_gamma), W = sum w, t = u_G * W,
 * the token is the smallest x with sum_{v<=x} w_v > t.  If the residual mass
 * rounds to zero the draw uses p_k and sets SPEC_ST_ZERO_RESIDUAL.
 * signals (optional, [B,4]): the SpecKV signals of q at the request's
 * temperature over all gamma_b draft rows (NaN when gamma_b = 0); requesting
 * them makes the call read every draft row.  accept_prob optional.
 * draft_logits may be NULL only when G = 0. */
int spec_verify_sample(const void* target_logits, const void* draft_logits, int dtype,
                       int B, int G, int V,
                       const int32_t* draft_tokens, const int32_t* gamma,
                       const float* temperature, const float* uniforms,
                       int32_t* accept_len, int32_t* tokens,
                       float* signals, float* accept_prob, int32_t* status,
                       void* workspace, size_t workspace_bytes, spec_stream_t stream);

/* Stochastic verification with a one-hot q (section 3.3): accept_i <=>
 * u_i < p_i(y_i); after a reject at k the draw uses p_k with y_k removed
 * (W summed over v != y_k); else p_gamma.  accept_prob (optional) = p_i(y_i). */
int spec_verify_onehot(const void* target_logits, int dtype, int B, int G, int V,
                       const int32_t* draft_tokens, const int32_t* gamma,
                       const float* temperature, const float* uniforms,
                       int32_t* accept_len, int32_t* tokens,
                       float* accept_prob, int32_t* status,
                       void* workspace, size_t workspace_bytes, spec_stream_t stream);

/* Draft signals only (SpecKV page): signals [B,4] required, row_signals
 * [B,G,2] optional (NaN for i >= gamma_b), status optional. */
int spec_draft_signals(const void* draft_logits, int dtype, int B, int G, int V,
                       const int32_t* gamma, const float* temperature,
                       float* signals, float* row_signals, int32_t* status,
                       void* workspace, size_t workspace_bytes, spec_stream_t stream);

/* Per-position divergence statistics of a draft chain.  For each request b
 * and position i < gamma_b, with p = softmax(target row i / T_b) and
 * q = softmax(draft row i / T_b), five fp32 values at stats[(b G + i) 5 + k]:
 *   k = 0: A = sum_v min(p(v), q(v)), = 1 - TV(p, q), the expected acceptance
 *          of the position (tutorial page section 4.3);
 *   k = 1: L1 = sum_v |p(v) - q(v)| (the L1 / TV distance of the DLite page's
 *          distillation loss and of the DDTE page's selector inputs);
 *   k = 2: KL(p||q) = sum p log2(p/q)  (forward KL, DLite page), +inf when
 *          some q(v) = 0 < p(v) (a draft logit of -inf);
 *   k = 3: KL(q||p) (with k = 2, the DDTE page's bidirectional KL);
 *   k = 4: H(p) = -sum p log2 p, the target entropy (DDTE page).
 * All in bits, as the draft signals.  Positions i >= gamma_b give NaN.
 *   target_logits  [B, G+1, V] (rows 0..G-1 are read), draft_logits [B, G, V],
 *                  dtype SPEC_F32 or SPEC_BF16, device, caller-owned, read
 *                  only;
 *   gamma          [B] int32 or NULL (= G); temperature [B] fp32 (required);
 *   stats          [B, G, 5] fp32 (required when G > 0), written;
 *   status         [B] int32 or NULL: zeroed, then SPEC_ST_BAD_GAMMA or
 *                  SPEC_ST_BAD_TEMPERATURE (every position of the request is
 *                  NaN) and SPEC_ST_NONFINITE (a position with NaN, +inf or no
 *                  finite maximum in either row is NaN; the others are valid).
 * Every row of positions < gamma_b is read twice (the second read mostly
 * from L2).  No workspace.  Host errors: SPEC_ERR_INVALID_ARG (sizes, dtype,
 * NULL required pointers, misalignment), SPEC_ERR_CUDA, SPEC_ERR_UNSUPPORTED. */
int spec_divergence_stats(const void* target_logits, const void* draft_logits, int dtype,
                          int B, int G, int V, const int32_t* gamma, const float* temperature,
                          float* stats, int32_t* status, spec_stream_t stream);

/* Top-k / top-p filtering of logit rows before verification (tutorial page
 * section 2.1: p and q are the distributions actually sampled from, with
 * temperature, top-k and top-p already applied when used).  Row r of
 * logits [n, V] is filtered in place, by value (ties stay together):
 *   top-k, when 1 <= top_k[r] < V: keep x >= the k-th largest logit;
 *   top-p, when 0 < top_p[r] < 1, on the distribution left by top-k at
 *   temperature[r]: keep x >= t*, the largest value whose upper mass
 *   sum_{x >= t*} softmax(x / T) reaches top_p;
 *   a removed logit becomes -inf.
 *   logits       [n, V], dtype SPEC_F32 or SPEC_BF16, device, caller-owned,
 *                read and written;
 *   top_k        [n] int32 or NULL (no top-k); top_p [n] fp32 or NULL (no
 *                top-p); temperature [n] fp32 or NULL (= 1; used by top-p);
 *   status       [n] int32 or NULL: 0, SPEC_ST_NONFINITE (a NaN or +inf, or
 *                no finite logit: the row is left unchanged) or
 *                SPEC_ST_BAD_TEMPERATURE (top-p with a temperature <= 0 or not
 *                finite: unchanged).
 * The top-p decision compares masses that fp32 weights carry to ~1e-6: a row
 * whose mass at t* lies within that of top_p can keep one value group more or
 * less than an exact computation.  Results are deterministic.  Filtering a
 * target and a draft row with the same settings gives the p and q the
 * verification calls then use.  No workspace.  Host errors:
 * SPEC_ERR_INVALID_ARG (n < 1, V outside [2, 2^28), dtype, NULL logits,
 * misalignment), SPEC_ERR_CUDA, SPEC_ERR_UNSUPPORTED. */
int spec_filter_top_k_top_p(void* logits, int dtype, int n, int V, const int32_t* top_k,
                            const float* top_p, const float* temperature, int32_t* status,
                            spec_stream_t stream);

/* The SpecKV gamma selector (SpecKV page, acceptance prediction and gamma
 * selection).  For each request, with the context
 * x = [mean H, mean c, max H, min c, comp] (the signals of spec_verify_sample
 * or spec_draft_signals, taken in that order, and a compression level), an
 * MLP f(x, gamma) with 16 hidden units predicts the acceptance rate; the
 * expected tokens of a step are f(x, gamma) gamma + 1 and
 * gamma* = argmax over gamma in {2, 4, 6, 8}, ties to the smaller gamma.
 * The MLP takes [x, gamma] standardised as (z - mu) / sd, has one ReLU hidden
 * layer and an identity output.
 *   signals     [B, 4] fp32 (mean H, max H, mean c, min c: the library's
 *               signal layout), device, read only;
 *   comp        [B] fp32 or NULL (= 0): the compression level feature;
 *   model       SPEC_GAMMA_MODEL_FLOATS fp32, device: mu[6], sd[6],
 *               W1[16][6] (row h holds hidden unit h's weights), b1[16],
 *               w2[16], b2;
 *   gamma_star  [B] int32, written: 2, 4, 6 or 8; -1 when a feature is not
 *               finite (a request with gamma_b = 0 or an error);
 *   expected    [B, 4] fp32 or NULL: f gamma + 1 for gamma = 2, 4, 6, 8 (NaN
 *               for a non-finite feature).
 * No workspace.  Host errors: SPEC_ERR_INVALID_ARG (B outside [1, 65535], NULL
 * signals, model or gamma_star, misalignment: signals 16-byte, the others
 * 4-byte), SPEC_ERR_CUDA, SPEC_ERR_UNSUPPORTED. */
#define SPEC_GAMMA_MODEL_FLOATS 141
int spec_gamma_select(const float* signals, const float* comp, const float* model, int B,
                      int32_t* gamma_star, float* expected, spec_stream_t stream);

/* Size of the library-owned scratch used by spec_verify_sample_static: 8 MiB.
 * It holds the workspace of spec_workspace_bytes(B, G, V) <= this value, e.g.
 * B <= 268 at G = 8, V = 151936, or B <= 276 at G = 7, V = 151936. */
#define SPEC_STATIC_WORKSPACE_BYTES (8u << 20)

/* spec_verify_sample without a caller workspace.  The pages have no
 * counterpart: this is a convenience of the library, not part of the method.
 *
 * Arguments, outputs and results are those of spec_verify_sample (same
 * meaning, layout and ownership); the call uses a file-scope device buffer
 * of SPEC_STATIC_WORKSPACE_BYTES inside the library instead.  The call
 * itself allocates nothing: no cudaMalloc, no cudaFree, no other allocating
 * routine.  It is meant for callers that cannot allocate: a C caller with no
 * device allocator of its own; a serving loop whose device memory is all
 * held by a pool allocator, so that no free bytes are left for a workspace;
 * a per-step decode path that must not pay cudaMalloc/cudaFree, which can
 * synchronise the device and stall every other stream.
 *
 * Setup: the first call on each device (with that device current) looks up
 * the buffer's device address once (cudaGetSymbolAddress; a failure returns
 * SPEC_ERR_CUDA and the next call tries again) and configures the kernels,
 * as the first call of any entry point does.  Make that first call before
 * any stream capture begins.
 * Contents: nothing in the buffer has to start at zero; every call's first
 * kernel resets each counter and flag it reads.
 * Sharing: every call of this entry point on one device uses the same
 * buffer.  Two calls whose executions overlap on the device (different
 * streams, or different host threads without ordering between them) race on
 * it and corrupt each other's results.  Calls on one stream run one after
 * the other and are safe.
 * Errors: as spec_verify_sample, and SPEC_ERR_WORKSPACE (before any CUDA
 * call) when spec_workspace_bytes(B, G, V) > SPEC_STATIC_WORKSPACE_BYTES. */
int spec_verify_sample_static(const void* target_logits, const void* draft_logits, int dtype,
                              int B, int G, int V,
                              const int32_t* draft_tokens, const int32_t* gamma,
                              const float* temperature, const float* uniforms,
                              int32_t* accept_len, int32_t* tokens,
                              float* signals, float* accept_prob, int32_t* status,
                              spec_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_VERIFY_H */
