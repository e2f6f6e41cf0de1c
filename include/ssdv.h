/*
 * ssdv.h -- C ABI of libssdv: batched speculative-decoding verification and
 * Saguaro pre-speculation on one GPU (sm_103a).
 *
 * Notation (speculative-decoding blog "投机解码 (Speculative Decoding):
 * 小模型猜、大模型验", section 3): q = target distribution, p = draft
 * distribution, gamma = number of draft tokens per request.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers named *_logits, draft_tokens, out_*, gamma, temperature,
 *    workspace, bonus_topk, saguaro_tokens, stats are DEVICE pointers owned by
 *    the caller.  The library allocates no device memory and keeps no pointer
 *    after a call returns.
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL = the legacy default stream), except where stated otherwise.
 *  - Logit layout: target [B, gamma_max+1, V] and draft [B, gamma_max, V],
 *    row-major, contiguous, row stride V elements.  Row i of the target is the
 *    target distribution for position i (row gamma is the position after the
 *    last draft token); row i of the draft is the draft distribution that
 *    proposed draft token i.  dtype is SSD_BF16 or SSD_F32 for both.
 *  - Rows whose start is 16-byte aligned (base 16-byte aligned and V*size
 *    a multiple of 16) are read with 16-byte vector loads straight into
 *    registers; other rows are copied into shared memory with plain loads.
 *    Both give the same results.
 *  - Every real row must hold at least one finite logit; NaN and +inf logits
 *    are not valid input.  -inf logits are allowed (probability 0).
 *  - Temperature: softmax(x / T) on both target and draft.  T == 0 selects
 *    greedy verification (accept while the draft token equals the target
 *    argmax, lowest index among equal logits; the correction / bonus is the
 *    target argmax).  0 < T < 1e-6, T < 0, NaN and inf are rejected.
 *  - Uniforms: Philox4x32-10 (Salmon et al., SC'11) with key (seed low 32
 *    bits, seed high 32 bits) and counter (request b, position i, 0, 0);
 *    word 0 is the accept draw, word 1 the resample / bonus draw, word 2 the
 *    Saguaro draw; u = (word >> 8) * 2^-24.  The same inputs and seed always
 *    give the same outputs.
 *  - Errors found on the host are returned before anything is launched.
 *    Errors found on the device (a draft token outside [0, V), a per-request
 *    gamma above gamma_max, a bad per-request temperature) make that request's
 *    outputs -1 and set a bit in the workspace status word (see
 *    ssd_read_status); the other requests are unaffected.
 *
 * Tuning overrides (environment variables, read on every call).  They split
 * the work differently.  SSDV_PPW, SSDV_SEGMENT, SSDV_SAG_PPW and
 * SSDV_SAG_SEGMENT leave every sum in the same order and the outputs
 * unchanged; SSDV_CHUNK_BYTES and SSDV_SMALL_V change the order of the row
 * sums, so a draw within rounding of a threshold may come out the other way.
 * ---------------------------------------------------------------------------
 *  - SSDV_CHUNK_BYTES: bytes of a row per streaming CTA (default 24576; a
 *    chunk holds at most 16384 elements and a row at most 32 chunks).
 *  - SSDV_PPW: pieces (128 vectors) of the draw row per warp of the
 *    verification sampling kernel (default 2 for plain calls, 1 when that
 *    grid fits one wave, 4 for pipelined calls).
 *  - SSDV_SEGMENT: requests per launch segment of verification (default and
 *    maximum 65535, the grid's third dimension).
 *  - SSDV_SMALL_V: 0 turns off the one-warp-per-request kernel that
 *    vocabularies up to 256 take (default 1).
 *  - SSDV_SAG_PPW: pieces per warp of the Saguaro residual and mix kernels
 *    (default 16, at least 2).
 *  - SSDV_SAG_SEGMENT: requests per launch segment of the Saguaro calls
 *    (default and maximum 65535).
 */
#ifndef SSDV_H
#define SSDV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SSD_OK = 0,
  SSD_ERR_NULL = 1,        /* a required pointer is NULL                        */
  SSD_ERR_SHAPE = 2,       /* B, gamma, V or k out of range                      */
  SSD_ERR_DTYPE = 3,       /* unknown ssd_dtype                                  */
  SSD_ERR_ALIGN = 4,       /* a pointer is not aligned to its element size       */
  SSD_ERR_TOKEN_RANGE = 5, /* (device) a draft token outside [0, V)              */
  SSD_ERR_TEMPERATURE = 6, /* temperature negative, NaN, inf or in (0, 1e-6)     */
  SSD_ERR_CUDA = 7,        /* a CUDA runtime call failed (see ssd_last_error)     */
  SSD_ERR_UNSUPPORTED = 8, /* no launch configuration fits this device / shape   */
  SSD_ERR_WORKSPACE = 9,   /* workspace missing or smaller than required         */
  SSD_ERR_GAMMA = 10,      /* (device) a per-request gamma above gamma_max       */
  SSD_ERR_DRAW = 11        /* (device) a draw found no token of positive weight  */
} ssd_status;

typedef enum { SSD_BF16 = 0, SSD_F32 = 1 } ssd_dtype;

/* Where Saguaro's predicted bonus tokens come from (SSD notes, section 3.1):
 * the k largest entries of the residual r_j, or the draft's k most likely
 * tokens (its k largest logits of row j; the target's at j = gamma, where
 * there is no draft row). */
typedef enum { SSD_TOPK_RESIDUAL = 0, SSD_TOPK_DRAFT = 1 } ssd_topk_source;

#define SSD_MAX_GAMMA 31   /* largest gamma / gamma_max accepted                 */
#define SSD_MAX_TOPK 8     /* largest k accepted by ssd_saguaro_prespec           */
#define SSD_MAX_V (1 << 19)  /* fp32 units above ~440k need more than 16 CTAs */
#define SSD_NSTAT_VERIFY 10
#define SSD_NSTAT_SAGUARO 10

/* Bytes of device workspace ssd_verify / ssd_verify_pipelined /
 * ssd_verify_ragged / ssd_verify_ragged_pipelined / ssd_debug_rowstats need
 * for a batch of B requests with
 * up to gamma_max draft tokens.  The workspace holds a status word and two
 * halves, used by alternate calls, of arrival counters (cleared by every call),
 * per-chunk row statistics and per-piece residual sums. */
size_t ssd_workspace_bytes(int B, int gamma_max);

/* Zero a workspace (asynchronous memset on `stream`).  Zero a workspace once
 * before its first use so that its status word starts clear; after that it can
 * be reused by later calls of any shape that fits it, on the same stream.  Two
 * calls that may run at the same time on the GPU need two workspaces. */
ssd_status ssd_workspace_init(void* workspace, size_t ws_bytes, void* stream);

/* Batched verification, one gamma and one temperature for the whole batch.
 *
 * Blog section 3: for each request b and draft position i = 0..gamma-1, draw
 * u_i and accept draft token x_i iff u_i < min(1, q_i(x_i) / p_i(x_i)); at the
 * first rejection n, emit one token sampled from (q_n - p_n)+ / sum (q_n - p_n)+
 * (from q_n if that mass is zero) and stop; if all gamma are accepted, emit a
 * bonus token sampled from q_gamma.  Greedy (T == 0): accept while x_i equals
 * argmax of target row i; emit the argmax at the stopping position.
 *
 *   target_logits  [B, gamma+1, V], draft_logits [B, gamma, V] (unused and may
 *                  be NULL when temperature == 0)
 *   draft_tokens   [B, gamma] int32
 *   out_tokens     [B, gamma+1] int32: x_0..x_{n-1}, the correction or bonus
 *                  token at index n, then -1
 *   n_accepted     [B] int32: n in 0..gamma (-1 for a request with an error)
 *   workspace      >= ssd_workspace_bytes(B, gamma) bytes, zeroed once
 *
 * Constraints: 1 <= B, 0 <= gamma <= SSD_MAX_GAMMA, 1 <= V <= SSD_MAX_V. */
ssd_status ssd_verify(const void* target_logits, const void* draft_logits, ssd_dtype dtype,
                      const int32_t* draft_tokens, int B, int gamma, int V, float temperature,
                      uint64_t seed, int32_t* out_tokens, int32_t* n_accepted, void* workspace,
                      size_t ws_bytes, void* stream);

/* Verification with top-p (nucleus) truncation on both sides (the
 * verification blog's closing remark and its section on matching sampling
 * parameters: speculative decoding stacks on temperature and top-p when the
 * target and the draft truncate the same way).  Every target row q_i and
 * draft row p_i keeps the tokens whose logit is at least th, the largest logit
 * value with P{x >= th} >= top_p (the most likely tokens until their mass
 * reaches top_p, plus every token tied with the last one needed), and is
 * renormalised; then ssd_verify's steps run on the truncated distributions: a
 * draft token outside the target's nucleus is rejected, one outside the
 * draft's is accepted, the correction comes from (q'_n - p'_n)+ and the bonus
 * from q'_gamma.  temperature == 0 (greedy) or top_p == 1 is ssd_verify.
 *   0 < top_p <= 1; B <= 65535.
 *   workspace >= ssd_verify_top_p_workspace_bytes(B, gamma) bytes, zeroed once.
 * Kernels: the streaming pass; then per level of the threshold select (3 for
 * bf16, 4 for fp32: one of mass bins, then the logit key's digits inside the
 * chosen bin) a histogram pass over the rows and a select pass; then the
 * sampling kernel. */
ssd_status ssd_verify_top_p(const void* target_logits, const void* draft_logits, ssd_dtype dtype,
                            const int32_t* draft_tokens, int B, int gamma, int V, float temperature,
                            float top_p, uint64_t seed, int32_t* out_tokens, int32_t* n_accepted,
                            void* workspace, size_t ws_bytes, void* stream);

/* Bytes of device workspace ssd_verify_top_p needs (a verification workspace
 * plus the per-row select state and radix histograms). */
size_t ssd_verify_top_p_workspace_bytes(int B, int gamma_max);

/* Pipelined verification: ssd_verify for a chain of calls whose inputs are
 * already complete.  This entry point has no counterpart in the method's
 * description; it serves a caller that keeps several independent batches in
 * flight (a round of batch A verified while batch B's next round drafts).
 *
 * Same arguments, outputs, numerics and random draws as ssd_verify.  The
 * difference is ordering: ssd_verify's kernels wait for the previous kernel on
 * `stream` to complete before they read anything, so a call never overlaps the
 * previous one.  Here the streaming kernel may start reading this call's
 * logits while the previous call's sampling kernel still runs, which hides
 * that kernel's latency.  The caller guarantees that the inputs (logits, draft
 * tokens) were complete before the previous verification call on `stream`
 * completed: produced before it in stream order, or resident all along.
 * Outputs and the workspace are still ordered: every call's outputs are
 * written after the previous call's, and alternate calls use alternate halves
 * of the workspace.  Use ssd_verify when the logits come from the kernel just
 * before the call. */
ssd_status ssd_verify_pipelined(const void* target_logits, const void* draft_logits, ssd_dtype dtype,
                                const int32_t* draft_tokens, int B, int gamma, int V, float temperature,
                                uint64_t seed, int32_t* out_tokens, int32_t* n_accepted, void* workspace,
                                size_t ws_bytes, void* stream);

/* Verification without a caller workspace.  This entry point has no
 * counterpart in the method's description: it is a packaging variant of
 * ssd_verify for callers that cannot hand over device memory -- a plain C
 * caller with no caching allocator (a cudaMalloc/cudaFree per call would
 * synchronise the device and cost more than the verification itself), or an
 * engine that has reserved all free HBM up front for its KV-cache pool, so
 * that one more allocation would fail.
 *
 * Same arguments, outputs, numerics and random draws as ssd_verify (the same
 * kernels run); the scratch is a fixed file-scope device array of
 * SSD_NOALLOC_SCRATCH_BYTES bytes inside the library, and the call allocates
 * no device memory.  The batch must fit it:
 * ssd_workspace_bytes(B, gamma) <= SSD_NOALLOC_SCRATCH_BYTES, which holds
 * whenever B * (gamma + 1) <= 1600 (B = 64 at gamma <= 24, B = 256 at
 * gamma <= 5); a larger batch returns SSD_ERR_WORKSPACE before anything is
 * launched.
 *
 * Every call looks up the current device's copy of the array with
 * cudaGetSymbolAddress (a host-side query that allocates nothing).  The first
 * call that sees a given address -- the first call on each device, and the
 * first after a device reset, which reloads the library's device code and may
 * move the array -- zeroes it with cudaMemsetAsync on `stream`; make that
 * first call before any stream capture begins.  The kernels clear their own arrival counters on every call; the
 * status word is never read back on this path (a request with bad input still
 * gets n_accepted = -1 and out_tokens = -1).
 *
 * One array per device is shared by every caller: calls in sequence on one
 * stream are safe, but calls that may overlap on the GPU (two streams, or two
 * host threads with no ordering between their streams) race on the scratch
 * and give wrong results.  Use ssd_verify with separate workspaces there. */
#define SSD_NOALLOC_SCRATCH_BYTES (16u << 20)
ssd_status ssd_verify_noalloc(const void* target_logits, const void* draft_logits, ssd_dtype dtype,
                              const int32_t* draft_tokens, int B, int gamma, int V, float temperature,
                              uint64_t seed, int32_t* out_tokens, int32_t* n_accepted, void* stream);

/* Ragged verification: request b uses gamma[b] draft tokens (0..gamma_max;
 * a negative gamma[b] marks a padded request whose outputs are all -1) and
 * temperature[b] (0 = greedy).  Layouts are padded to gamma_max: target rows
 * > gamma[b], draft rows >= gamma[b], draft tokens >= gamma[b], and every draft
 * row of a greedy request are never read.  out_tokens [B, gamma_max+1]. */
ssd_status ssd_verify_ragged(const void* target_logits, const void* draft_logits, ssd_dtype dtype,
                             const int32_t* draft_tokens, int B, int gamma_max, int V,
                             const int32_t* gamma, const float* temperature, uint64_t seed,
                             int32_t* out_tokens, int32_t* n_accepted, void* workspace,
                             size_t ws_bytes, void* stream);

/* Pipelined ragged verification: ssd_verify_ragged for a chain of calls whose
 * inputs are already complete.  Like ssd_verify_pipelined, this entry point
 * has no counterpart in the method's description.  Same arguments, outputs,
 * numerics and random draws as ssd_verify_ragged; the difference is the one
 * between ssd_verify_pipelined and ssd_verify.  The streaming kernel may read
 * this call's logits while the previous call's sampling kernel still runs, so
 * the caller guarantees that the inputs (logits, draft tokens, gamma and
 * temperature arrays) were complete before the previous verification call on
 * `stream` completed. */
ssd_status ssd_verify_ragged_pipelined(const void* target_logits, const void* draft_logits, ssd_dtype dtype,
                                       const int32_t* draft_tokens, int B, int gamma_max, int V,
                                       const int32_t* gamma, const float* temperature, uint64_t seed,
                                       int32_t* out_tokens, int32_t* n_accepted, void* workspace,
                                       size_t ws_bytes, void* stream);

/* Saguaro pre-speculation (SSD notes, sections 3.1 and 3.2).  For each request
 * b and each acceptance length j = 0..gamma:
 *   r_j = (q_j - p_j)+ / sum (q_j - p_j)+  for j < gamma (q_j if that mass is
 *         zero), and r_gamma = q_gamma;
 *   bonus_topk[b, j, 0..k-1] = the k largest entries of r_j, descending, the
 *         lower index first among equal values (topk_source ==
 *         SSD_TOPK_RESIDUAL), or the k largest draft logits of row j (target
 *         logits at j = gamma), same order (SSD_TOPK_DRAFT);
 *   saguaro_tokens[b, j] = one sample from p_saguaro proportional to
 *         sqrt(p_D(v) * max(r_j(v), 1e-8)), p_D = p_j (q_gamma at j = gamma).
 *   target_logits [B, gamma+1, V], draft_logits [B, gamma, V];
 *   bonus_topk [B, gamma+1, k] int32, saguaro_tokens [B, gamma+1] int32.
 *   workspace >= ssd_saguaro_workspace_bytes(B, gamma, V) bytes, zeroed once
 *   (ssd_workspace_init), 16-byte aligned; its status word reports device
 *   errors as for verification (ssd_read_status).
 * Constraints: temperature > 0, 1 <= k <= SSD_MAX_TOPK, k <= V. */
ssd_status ssd_saguaro_prespec(const void* target_logits, const void* draft_logits, ssd_dtype dtype,
                               int B, int gamma, int V, int k, ssd_topk_source topk_source,
                               float temperature, uint64_t seed,
                               int32_t* bonus_topk, int32_t* saguaro_tokens, void* workspace,
                               size_t ws_bytes, void* stream);

/* Bytes of device workspace ssd_saguaro_prespec / ssd_debug_saguaro_stats
 * need for B requests, gamma draft tokens and vocabulary V (either dtype): a
 * status word, arrival counters, per-chunk row statistics, per-piece weight
 * sums and every warp's top-8 candidates. */
size_t ssd_saguaro_workspace_bytes(int B, int gamma, int V);

/* Verification and Saguaro pre-speculation of the same round in one call
 * (SSD notes, section 4.1: the target verifies a round while the next one is
 * pre-speculated from the same distributions).  Outputs exactly those of
 * ssd_verify (out_tokens, n_accepted) and of ssd_saguaro_prespec (bonus_topk,
 * saguaro_tokens) on the same arguments, with every logit row read from HBM
 * once for both, plus the cache check of ssd_cache_check (hit, n_hits; either
 * may be NULL).  temperature > 0 (Saguaro has no greedy form).
 *   workspace >= ssd_saguaro_workspace_bytes(B, gamma, V) bytes, zeroed once.
 * Constraints: those of ssd_verify and ssd_saguaro_prespec. */
ssd_status ssd_verify_saguaro(const void* target_logits, const void* draft_logits, ssd_dtype dtype,
                              const int32_t* draft_tokens, int B, int gamma, int V, int k,
                              ssd_topk_source topk_source, float temperature, uint64_t seed,
                              int32_t* out_tokens,
                              int32_t* n_accepted, int32_t* bonus_topk, int32_t* saguaro_tokens,
                              int32_t* hit, int32_t* n_hits, void* workspace, size_t ws_bytes,
                              void* stream);

/* Verification of draft tokens sampled from the Saguaro distribution (SSD
 * notes, sections 3.2 and 5.1: SSD is standard speculative decoding under
 * Saguaro sampling).  Position i's draft token x_i was drawn from
 *   p'_i(v) = sqrt(p_i(v) * max(r_i(v), 1e-8)) / sum_w sqrt(p_i(w) * max(r_i(w), 1e-8)),
 *   r_i = (q_i - p_i)+ / sum (q_i - p_i)+  (q_i when that mass is zero),
 * so p'_i takes p_i's place: accept iff u_i < min(1, q_i(x_i) / p'_i(x_i)),
 * and the correction at the first rejection n comes from
 * (q_n - p'_n)+ / sum (q_n - p'_n)+ (q_n if that mass is zero); the bonus from
 * q_gamma.  Arguments and outputs as ssd_verify; temperature > 0.
 *   workspace >= ssd_saguaro_workspace_bytes(B, gamma, V) bytes, zeroed once.
 * Kernels: the streaming pass, the Saguaro residual and mix passes over the
 * draft positions (no top-k, no draw), then the sampling kernel. */
ssd_status ssd_verify_saguaro_draft(const void* target_logits, const void* draft_logits,
                                    ssd_dtype dtype, const int32_t* draft_tokens, int B, int gamma,
                                    int V, float temperature, uint64_t seed, int32_t* out_tokens,
                                    int32_t* n_accepted, void* workspace, size_t ws_bytes,
                                    void* stream);

/* The Saguaro cache check (SSD notes, sections 3.3 and 4.1): a round hits the
 * pre-speculated cache when its correction / bonus token is among the bonus
 * tokens predicted for its acceptance length.
 *   bonus_topk [B, gamma+1, k] (ssd_saguaro_prespec), out_tokens [B, gamma+1]
 *   and n_accepted [B] (ssd_verify) of the same round;
 *   hit [B] int32 (nullable): the slot s with bonus_topk[b, n_b, s] ==
 *       out_tokens[b, n_b], else -1 (and -1 for a request with n_b = -1);
 *   n_hits [1] int32 (nullable): the number of hits (set, not accumulated).
 * At least one of hit / n_hits must be given.  One small kernel. */
ssd_status ssd_cache_check(const int32_t* bonus_topk, const int32_t* out_tokens,
                           const int32_t* n_accepted, int B, int gamma, int k, int32_t* hit,
                           int32_t* n_hits, void* stream);

/* Debug / parity: ssd_verify (same arguments and outputs) that also returns
 * the per-position quantities it computes, for every position whether or not
 * it is reached (the residual pass then runs at every position).
 * stats [B, gamma+1, 10] float:
 *   0 target row max (raw logit), 1 ln sum exp((x - max)/T) of the target row,
 *   2 draft row max, 3 its log-sum, 4 q_i(x_i), 5 p_i(x_i),
 *   6 residual mass sum (q_i - p_i)+, 7 accept probability min(1, q/p),
 *   8, 9 the distances u - C_{k-1}/S and C_k/S - u of the resample / bonus
 *   uniform u to the normalised CDF boundaries of the token drawn at this
 *   position (the correction after a rejection, or the bonus).
 * Row gamma fills only 0, 1, 8 and 9; entries that do not apply are NaN.
 * Greedy (T == 0) fills only entry 0 (the target row max). */
ssd_status ssd_debug_rowstats(const void* target_logits, const void* draft_logits, ssd_dtype dtype,
                              const int32_t* draft_tokens, int B, int gamma, int V,
                              float temperature, uint64_t seed, int32_t* out_tokens,
                              int32_t* n_accepted, float* stats, void* workspace,
                              size_t ws_bytes, void* stream);

/* Debug / parity: the per-position quantities ssd_saguaro_prespec computes.
 * stats [B, gamma+1, 10] float: 0 target log-sum, 1 draft log-sum (NaN at
 * j = gamma), 2 residual mass S_j (1 at j = gamma), 3 Zs = sum_v sqrt(p_D(v) *
 * max(r_j(v), 1e-8)), 4 p_saguaro(token), 5 r_j of top slot 0, 6 r_j of top
 * slot k-1 (with SSD_TOPK_DRAFT: p_j of those slots, q_gamma at j = gamma),
 * 7 NaN, 8, 9 the distances u - lo, hi - u of the Saguaro uniform to the
 * normalised CDF boundaries of the drawn token.
 * Outputs and workspace as ssd_saguaro_prespec. */
ssd_status ssd_debug_saguaro_stats(const void* target_logits, const void* draft_logits,
                                   ssd_dtype dtype, int B, int gamma, int V, int k,
                                   ssd_topk_source topk_source,
                                   float temperature, uint64_t seed, int32_t* bonus_topk,
                                   int32_t* saguaro_tokens, float* stats, void* workspace,
                                   size_t ws_bytes, void* stream);

/* Debug / parity: the uniforms the kernels draw.  out [B, W, 3] float gets,
 * for request b < B and position i < W, the accept, resample / bonus and
 * Saguaro uniforms (Philox4x32-10 words 0, 1, 2 of counter (b, i, 0, 0)). */
ssd_status ssd_debug_uniforms(uint64_t seed, int B, int W, float* out, void* stream);

/* Read and clear the device status word of a workspace.  Synchronises
 * `stream`.  *status gets SSD_OK or the lowest-numbered device error seen
 * since the last read. */
ssd_status ssd_read_status(void* workspace, size_t ws_bytes, int* status, void* stream);

/* Static text for a status code. */
const char* ssd_status_str(ssd_status status);

/* Detail of the last error returned on the calling thread ("" if none). */
const char* ssd_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SSDV_H */
