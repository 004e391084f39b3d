/*
 * smcsd.h -- C ABI of the GB300 library for the speculative-decoding verify step over
 * vocabulary-wide logits: temperature / power-target logsumexp, SD rejection sampling,
 * SMC-SD importance reweighting, effective sample size, systematic resampling, the paged-KV
 * page-table remap, and the PACER blockwise stop rule with ragged verify.
 *
 * Sources (gist.science summary pages; the pages print no formulas, so where a step is only
 * named the textbook rule is used and stated below):
 *   [SMC]   "Faster LLM Inference via Sequential Monte Carlo": sec. 1 (SD verifies by rejection
 *           sampling, the block is discarded after the first rejection), sec. 2 steps 1-4
 *           (N particles, K drafts each, one target scoring pass, reweighting by the
 *           target/draft probability ratio, resampling when the effective sample size falls
 *           below a threshold, exactly K+1 tokens per particle and step), sec. 3 (page-based
 *           KV: resampling is a metadata update; power sampling and reward-weighted decoding as
 *           modified targets; error bounds in N), sec. 5 (reward optimisation and hard
 *           constraints through the same importance weights).
 *   [PACER] "PACER: Blockwise Pre-verification for Speculative Decoding with Adaptive Length",
 *           Methodik 1-3 (blocks of b drafts whose hidden states, with position embeddings, give
 *           an estimated acceptance; the block mean against a threshold t that is multiplied by
 *           rho after each block that passes).
 *   [UAG]   "Cross-Family Speculative Decoding for Polish Language Models on Apple Silicon",
 *           sec. 1 (the target verifies k candidates in one pass).
 *
 * Conventions for every entry point
 *   - Every pointer argument is a DEVICE pointer owned by the caller, except where noted. The
 *     library allocates nothing and keeps no state between calls outside the caller's buffers;
 *     the one exception is smc_step_static, whose scratch is a device area of the library's own.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream). Every call
 *     only enqueues work on it and returns; results are valid once the stream has reached them.
 *   - Logits are row-major [rows, V] with V contiguous; dtype SMCSD_F32 (float32) or SMCSD_BF16.
 *     -inf marks a masked token. NaN or +inf, or a row with nothing but -inf, is an error
 *     detected on the device (SMCSD_ERR_NONFINITE).
 *   - Uniforms are float32 in [0,1), supplied by the caller (one per random decision), so that a
 *     run is reproducible and its randomness can be shared with a checker.
 *   - `ws` is a scratch buffer of at least smcsd_workspace_size(op, ...) bytes, 256-byte aligned,
 *     which must be zero-filled once before its first use (smcsd_workspace_init). Every call that
 *     returns SMCSD_OK leaves the buffer's counters at zero again, so a buffer can be reused by
 *     calls in stream order without clearing. Calls that may overlap on the GPU need separate
 *     buffers.
 *   - Return value: SMCSD_OK, or a negative status for errors found on the host before anything
 *     is enqueued (bad argument, dtype, workspace size) or at launch (CUDA error). Errors that
 *     depend on device data (non-finite logits, token ids or offsets out of range) are recorded
 *     in `ws` and read with smcsd_check_status(). The kernels never trap and never wait on
 *     another block; the waits inside a block (the copy pipeline of the streaming pass) give
 *     up after about 2 s and record SMCSD_ERR_TIMEOUT. So a bad input cannot fault or hang the
 *     GPU; outputs are unspecified after such an error.
 */
#ifndef SMCSD_H
#define SMCSD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define SMCSD_OK 0
#define SMCSD_ERR_INVALID_ARG (-1) /* null pointer, non-positive size, T <= 0, alpha <= 0, ... */
#define SMCSD_ERR_DTYPE (-2)       /* dtype other than SMCSD_F32 / SMCSD_BF16 */
#define SMCSD_ERR_WORKSPACE (-3)   /* ws_bytes smaller than smcsd_workspace_size() or ws misaligned */
#define SMCSD_ERR_CUDA (-4)        /* a CUDA call or kernel launch failed */
#define SMCSD_ERR_NONFINITE (-5)   /* device: NaN/+inf logit or weight, or an all-masked row */
#define SMCSD_ERR_RANGE (-6)       /* device: token id, offset, ancestor or page id out of range */
#define SMCSD_ERR_TIMEOUT (-7)     /* device: a bounded wait inside a kernel ran out (about 2 s) */

/* logit element types */
#define SMCSD_F32 0
#define SMCSD_BF16 1

/* targets of the tilted SMC reweight (smc_reweight_tilted, smc_step_tilted) */
#define SMCSD_TARGET_TOKEN 0    /* per position: pi = softmax(alpha z / T), as smc_reweight */
#define SMCSD_TARGET_SEQUENCE 1 /* whole sequence: prod_t p_t(x_t)^alpha, p = softmax(z / T) */

/* operation ids for smcsd_workspace_size */
#define SMCSD_OP_SD_VERIFY 0
#define SMCSD_OP_SMC_REWEIGHT 1
#define SMCSD_OP_SMC_STEP 2
#define SMCSD_OP_ESS_RESAMPLE 3
#define SMCSD_OP_PAGETABLE_REMAP 4
#define SMCSD_OP_PACER_BLOCK_STOP 5
#define SMCSD_OP_DRAFT_SAMPLE 6 /* S = number of rows R; K is ignored */

/*
 * Scratch bytes that `op` needs for S sequences (or particles; for the resampling ops S is the
 * number of groups G), at most K draft positions and vocabulary V.
 */
size_t smcsd_workspace_size(int op, int S, int K, int V);

/* Zero-fill `ws` on `stream` (needed once before a buffer's first use). */
int smcsd_workspace_init(void* ws, size_t ws_bytes, void* stream);

/*
 * Wait for `stream`, then return the first device-side error recorded in `ws` since the last
 * check (SMCSD_OK if none) and clear it.
 */
int smcsd_check_status(void* ws, void* stream);

/* Static text for a status code. */
const char* smcsd_status_string(int code);

/*
 * Diagnostic for the failure path of the bounded waits (no counterpart on the pages): one warp
 * runs the streaming pass's two pipeline waits against a barrier and a slot tag that nothing
 * completes, each giving up after limit_us microseconds (1 .. 2000000) and recording
 * SMCSD_ERR_TIMEOUT in `ws` as a stalled pipeline would. Read it with smcsd_check_status; the
 * context stays usable. ws: any workspace of at least 4 bytes (zero-filled once, as always).
 */
int smcsd_selftest_wait(unsigned int limit_us, void* ws, size_t ws_bytes, void* stream);

/*
 * Speculative-decoding verify ([SMC] sec. 1; [UAG] sec. 1; ragged lengths from [PACER]
 * Methodik 2). For every sequence s, with p = softmax(z_t / T) and q = softmax(z_d / T):
 *   accept draft x_k iff u[s*(K+1)+k] < min(1, p_k(x_k) / q_k(x_k)), k = 0, 1, ... in order;
 *   accept_len[s] = index of the first rejection, or K_s if all pass;
 *   out_token[s]  = draw from normalise(max(0, p_acc - q_acc)) if a draft was rejected, else
 *                   the bonus draw from p at target row K_s; both by inverse CDF with
 *                   u[s*(K+1)+K]: the first token whose cumulative weight exceeds u * total.
 *                   A residual with zero mass (only reachable through rounding) falls back to p.
 * Layout, fixed (tgt_offsets == drf_offsets == NULL): target [S*(K+1), V] (row s*(K+1)+k),
 *   draft [S*K, V] (row s*K+k), draft_tokens [S*K].
 * Layout, ragged (both offsets given, int32 [S+1] device arrays): sequence s has
 *   K_s = drf_offsets[s+1]-drf_offsets[s] <= K drafts, target rows tgt_offsets[s] ..
 *   tgt_offsets[s+1]-1 (K_s+1 rows), draft rows and draft tokens drf_offsets[s] .. +K_s-1.
 *   Inconsistent offsets are reported as SMCSD_ERR_RANGE through smcsd_check_status.
 * uniforms: [S*(K+1)] (positions k >= K_s of a ragged sequence are unused).
 * accept_len, out_token: int32 [S]. lse_tgt / lse_drf: optional float [rows] (NULL to skip),
 *   the natural-log normaliser of each scaled row, log sum_i exp(z_i / T).
 */
int sd_verify(const void* tgt_logits, const void* drf_logits, int dtype,
              const int32_t* draft_tokens, const int32_t* tgt_offsets, const int32_t* drf_offsets,
              int S, int K, int V, float temperature, const float* uniforms,
              int32_t* accept_len, int32_t* out_token, float* lse_tgt, float* lse_drf,
              void* ws, size_t ws_bytes, void* stream);

/*
 * SMC-SD reweight and bonus token ([SMC] sec. 2 steps 3-4; power target from [SMC] sec. 3).
 * Target pi = softmax(alpha * z_t / T) (alpha = 1 is plain p; alpha != 1 is the power target
 * p^alpha renormalised), draft q = softmax(z_d / T). For each particle s:
 *   logw[s] += sum_{k<K} ( log pi_k(x_k) - log q_k(x_k) )   (float in/out)
 *   bonus_token[s] = inverse-CDF draw from pi at target row K with uniforms[s]
 *   (the (K+1)-th token; its weight factor is pi/pi = 1).
 * Layout: target [S*(K+1), V], draft [S*K, V], draft_tokens [S*K], uniforms [S].
 * lse_tgt [S*(K+1)] / lse_drf [S*K]: optional normalisers (NULL to skip).
 */
int smc_reweight(const void* tgt_logits, const void* drf_logits, int dtype,
                 const int32_t* draft_tokens, int S, int K, int V, float temperature, float alpha,
                 const float* uniforms, float* logw, int32_t* bonus_token,
                 float* lse_tgt, float* lse_drf, void* ws, size_t ws_bytes, void* stream);

/*
 * SMC-SD reweight toward a tilted target ([SMC] sec. 3 "flexibility": modified targets such as
 * power sampling and reward-weighted decoding; sec. 5: reward optimisation and hard
 * constraints through the same importance weights). Arguments and layout as smc_reweight, plus:
 *   target = SMCSD_TARGET_TOKEN: smc_reweight's per-position target pi = softmax(alpha z_t / T).
 *   target = SMCSD_TARGET_SEQUENCE: the unnormalised power of the sequence probability,
 *     prod_t p_t(x_t)^alpha with p = softmax(z_t / T). The draft tokens are proposed by q and
 *     the (K+1)-th token b_s is drawn from p at target row K (with uniforms[s]), so
 *       logw[s] += sum_{k<K} ( alpha log p_k(x_k) - log q_k(x_k) ) + (alpha - 1) log p_K(b_s).
 *     alpha = 1 gives smc_reweight's result. lse_tgt then holds the normalisers at 1/T.
 *   log_reward: optional float [S] (NULL for none); logw[s] += reward_scale * log_reward[s].
 *     A NaN or infinite reward is SMCSD_ERR_NONFINITE (device side, smcsd_check_status);
 *     reward_scale must be finite when log_reward is given.
 * target other than the two values above: SMCSD_ERR_INVALID_ARG.
 */
int smc_reweight_tilted(const void* tgt_logits, const void* drf_logits, int dtype,
                        const int32_t* draft_tokens, int S, int K, int V, float temperature,
                        float alpha, int target, const float* log_reward, float reward_scale,
                        const float* uniforms, float* logw, int32_t* bonus_token,
                        float* lse_tgt, float* lse_drf, void* ws, size_t ws_bytes, void* stream);

/*
 * Draft-token sampling ([SMC] sec. 2 step 1: the draft model proposes K tokens per particle,
 * each drawn from its tempered distribution). For each of R rows of `logits` ([R, V], dtype as
 * above), with q_r = softmax(z_r / T):
 *   tokens[r] = the first token whose cumulative q_r exceeds uniforms[r] (inverse CDF, the same
 *               draw as the verify's final token);
 *   logq[r]   = log q_r(tokens[r]) (optional, NULL to skip), what a verify needs from the draft;
 *   lse[r]    = log sum_i exp(z_{r,i} / T) (optional).
 * uniforms: float [R]; tokens: int32 [R]; logq, lse: float [R]. ws: see
 * smcsd_workspace_size(SMCSD_OP_DRAFT_SAMPLE, R, 0, V). An all-masked or non-finite row is
 * SMCSD_ERR_NONFINITE (device side) and its token is reported as 0.
 */
int draft_sample(const void* logits, int dtype, int R, int V, float temperature,
                 const float* uniforms, int32_t* tokens, float* logq, float* lse,
                 void* ws, size_t ws_bytes, void* stream);

/*
 * Effective sample size and systematic resampling per group of N particles ([SMC] sec. 2
 * step 4; the textbook forms, in double precision):
 *   w_i = exp(logw_i - max logw), ess[g] = (sum w)^2 / sum w^2;
 *   resampled[g] = ess[g] < ess_threshold (strict);
 *   if resampled: C_i = (sum_{j<=i} w_j)/W with C_{N-1} = 1, v_j = (j + uniforms[g]) / N,
 *                 ancestors[g*N+j] = min{ i : C_i > v_j }, and logw of the group is set to 0;
 *   else ancestors[g*N+j] = j and logw is unchanged.
 * logw [G*N] float in/out; uniforms [G]; ancestors [G*N] (group-local indices); ess [G] and
 * resampled [G] may be NULL. ws: see smcsd_workspace_size(SMCSD_OP_ESS_RESAMPLE, G, 0, 0).
 */
int smc_ess_resample(float* logw, int G, int N, float ess_threshold, const float* uniforms,
                     int32_t* ancestors, float* ess, int32_t* resampled,
                     void* ws, size_t ws_bytes, void* stream);

/*
 * Paged-KV page-table remap ([SMC] sec. 3: resampling moves no KV data, only metadata).
 *   table_out[g*N+j][:] = table_in[g*N+a][:], a = ancestors[g*N+j] if resampled[g] (or if
 *   resampled == NULL), else a = j;
 *   refcount (optional, int32 [num_pages]) is rebuilt: refcount[p] = entries of table_out == p.
 * Tables are int32 [G*N, pages_per_seq]; table_out must not alias table_in. -1 marks an empty
 * slot (copied, not counted). Other ids outside [0, num_pages) or ancestors outside [0, N) are
 * reported as SMCSD_ERR_RANGE through smcsd_check_status (the entry is then not counted).
 */
int kv_pagetable_remap(const int32_t* ancestors, const int32_t* resampled, int G, int N,
                       const int32_t* table_in, int32_t* table_out, int pages_per_seq,
                       int32_t* refcount, int num_pages, void* ws, size_t ws_bytes, void* stream);

/*
 * pacer_block_stop with position embeddings ([PACER] Methodik 1: the pre-verification layer
 * reads the block's hidden states together with position embeddings; the ablation under
 * "Ergebnisse" finds them essential). pos_emb: bf16 [max_blocks*b, d], row j for draft position
 * j, shared by all sequences (NULL: pacer_block_stop). The score of position j is
 *   score_j = sigmoid(w . (h_j + pos_emb_j) + c);
 * everything else is as in pacer_block_stop below.
 */
int pacer_block_stop_pos(const void* hidden, const void* w, const void* pos_emb, float c, int S,
                         int b, int max_blocks, int d, float t0, float rho, int32_t* lengths,
                         float* block_scores, int32_t* tgt_offsets, int32_t* drf_offsets,
                         void* ws, size_t ws_bytes, void* stream);

/*
 * PACER blockwise stop ([PACER] Methodik 1-3), with the pre-verification layer modelled as
 * score_j = sigmoid(w . h_j + c) over hidden states h (bf16 [S, max_blocks*b, d]) and a head
 * w (bf16 [d]):
 *   t = t0; for block i: m_i = mean of the b scores; if m_i < t: length = (i+1)*b, stop;
 *   else t = t * rho. No stop: length = max_blocks*b.
 * Only the blocks up to the stop are read. lengths: int32 [S]. block_scores: optional float
 * [S*max_blocks] (m_i of scored blocks, -1 after the stop). tgt_offsets / drf_offsets: optional
 * int32 [S+1], filled with the ragged layout that sd_verify takes for these lengths
 * (prefix sums of length+1 and of length).
 */
int pacer_block_stop(const void* hidden, const void* w, float c, int S, int b, int max_blocks,
                     int d, float t0, float rho, int32_t* lengths, float* block_scores,
                     int32_t* tgt_offsets, int32_t* drf_offsets,
                     void* ws, size_t ws_bytes, void* stream);

/*
 * One whole SMC-SD step in one pass over the logits ([SMC] sec. 2 steps 3-4 and sec. 3):
 * smc_reweight for S = G*N particles, then per group the effective sample size, systematic
 * resampling and the page-table remap, with the same semantics as the three calls above
 * (bonus_uniforms [G*N], resample_uniforms [G]). table_in / table_out / refcount may all be
 * NULL to skip the remap (pages_per_seq and num_pages are then ignored). ess and resampled
 * may be NULL.
 */
int smc_step(const void* tgt_logits, const void* drf_logits, int dtype,
             const int32_t* draft_tokens, int G, int N, int K, int V, float temperature,
             float alpha, const float* bonus_uniforms, float* logw, int32_t* bonus_token,
             float ess_threshold, const float* resample_uniforms, int32_t* ancestors,
             float* ess, int32_t* resampled, const int32_t* table_in, int32_t* table_out,
             int pages_per_seq, int32_t* refcount, int num_pages,
             void* ws, size_t ws_bytes, void* stream);

/*
 * smc_step with the draft's log-probabilities in place of its logits ([SMC] sec. 2 steps 1 and 3:
 * the draft proposes each token from its own distribution, and the weight needs only the
 * probability the draft gave the proposed token). drf_logq: float [G*N*K], log q_k(x_k) of draft
 * token draft_tokens[s*K+k] under the draft's tempered distribution at `temperature`, as
 * draft_sample returns it when it draws the tokens. The step then reads only the target logits
 * (target [G*N*(K+1), V]); its results are those of smc_step on draft logits whose normalised
 * log-probabilities at the draft tokens equal drf_logq:
 *   logw[s] += sum_{k<K} ( log pi_k(x_k) - drf_logq[s*K+k] ),
 * with pi = softmax(alpha z_t / T), then the bonus token, ESS, resampling and remap as smc_step.
 * The values of drf_logq are taken as given (non-positive and finite for a real distribution; a
 * NaN makes the particle's weight NaN, reported as SMCSD_ERR_NONFINITE by the group's ESS).
 * Arguments otherwise as smc_step; ws: smcsd_workspace_size(SMCSD_OP_SMC_STEP, G*N, K, V).
 */
int smc_step_logq(const void* tgt_logits, int dtype, const int32_t* draft_tokens,
                  const float* drf_logq, int G, int N, int K, int V, float temperature, float alpha,
                  const float* bonus_uniforms, float* logw, int32_t* bonus_token,
                  float ess_threshold, const float* resample_uniforms, int32_t* ancestors,
                  float* ess, int32_t* resampled, const int32_t* table_in, int32_t* table_out,
                  int pages_per_seq, int32_t* refcount, int num_pages, void* ws, size_t ws_bytes,
                  void* stream);

/*
 * smc_step toward a tilted target: target, log_reward and reward_scale as in
 * smc_reweight_tilted; everything else as in smc_step. The reward enters the log-weights
 * before the group's ESS and resampling.
 */
int smc_step_tilted(const void* tgt_logits, const void* drf_logits, int dtype,
                    const int32_t* draft_tokens, int G, int N, int K, int V, float temperature,
                    float alpha, int target, const float* log_reward, float reward_scale,
                    const float* bonus_uniforms, float* logw, int32_t* bonus_token,
                    float ess_threshold, const float* resample_uniforms, int32_t* ancestors,
                    float* ess, int32_t* resampled, const int32_t* table_in, int32_t* table_out,
                    int pages_per_seq, int32_t* refcount, int num_pages,
                    void* ws, size_t ws_bytes, void* stream);

/*
 * smc_step without a workspace argument. None of the pages has a counterpart: this is an
 * interface variant of smc_step (same step, same arguments and results, minus ws / ws_bytes)
 * for callers that cannot allocate device memory for a workspace, such as a host program with no
 * device allocator or a plugin that must not use its host's allocator. The call allocates
 * nothing: its scratch is a 32 MiB device area owned by this library (SMCSD_STATIC_SCRATCH_BYTES),
 * set aside when the library's device code is loaded.
 *   status: optional int32 device pointer; receives this call's device-side status (SMCSD_OK or
 *     a negative SMCSD_* code, as smcsd_check_status would report), written in stream order.
 *     Without it, device-side errors of the call are not reported.
 * Returns SMCSD_ERR_WORKSPACE, before any device work, when the shape needs more scratch than the
 * area holds (smcsd_workspace_size(SMCSD_OP_SMC_STEP, G*N, K, V) > SMCSD_STATIC_SCRATCH_BYTES),
 * and the host-side errors of smc_step otherwise.
 * Each call clears, on the stream, the part of the scratch that must start at zero. All calls on
 * one device share the one area: calls whose device work may overlap (different streams, or
 * several host threads without ordering between them) race on it and give wrong results, so
 * order them, for instance on one stream. The first call on a device looks the area's address up
 * with that device current; make that first call before any stream capture begins.
 */
#define SMCSD_STATIC_SCRATCH_BYTES (32u << 20)
int smc_step_static(const void* tgt_logits, const void* drf_logits, int dtype,
                    const int32_t* draft_tokens, int G, int N, int K, int V, float temperature,
                    float alpha, const float* bonus_uniforms, float* logw, int32_t* bonus_token,
                    float ess_threshold, const float* resample_uniforms, int32_t* ancestors,
                    float* ess, int32_t* resampled, const int32_t* table_in, int32_t* table_out,
                    int pages_per_seq, int32_t* refcount, int num_pages, int32_t* status,
                    void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SMCSD_H */
