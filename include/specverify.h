/*
 * specverify.h -- C ABI of the GB300 (sm_103a) speculative-sampling verification library.
 *
 * Batched verification of draft tokens against full-vocabulary target and draft logits:
 *  - temperature softmax of both rows, with one temperature for both ("standardized sampling",
 *    lossless-proof tutorial "Speculative Decoding 为什么是 Lossless 的 — 详细证明教程", §8 Q4);
 *  - the accept test r < min(1, p_target(t) / p_draft(t)), evaluated as r * p_draft(t) < p_target(t)
 *    (same tutorial, §5.1 SpecSampleOne);
 *  - on the first reject, one draw from the residual (p_target - p_draft)+ / Z, Z = sum (p_target - p_draft)+
 *    (§5.1, §6.4); the drafts after it are dropped; if every draft is accepted, one bonus draw from the
 *    target row K+1 (§9.1, the gamma-step chain);
 *  - HedgeSpec counterfactual acceptance gamma[i,b,j] = 1 - TV(p_target, q_i) = sum_x min(p_target, q_i)
 *    for every drafter i ("Not-a-Bandit: Provably No-Regret Drafter Selection in Speculative Decoding for
 *    LLMs", Key design 1) and its loss 1 - gamma (Key design 3);
 *  - Cactus constrained acceptance ("Cactus: Accelerating Auto-Regressive Decoding with Constrained
 *    Acceptance Speculative Sampling", Key design 2-3): gamma* = min(q(n) + sqrt(2 delta q(n)(1 - q(n))), 1)
 *    with q(n) the TARGET probability of the draft token n (that page calls the target q and the draft p),
 *    target h_n = gamma*, h_i = (1 - gamma*) / (1 - q(n)) * p_target(i), accept iff r * p_draft(n) < gamma*,
 *    residual (h - p_draft)+ / sum (h - p_draft)+.
 *
 * Conventions for every call:
 *  - Tensor pointers are DEVICE memory owned by the caller, contiguous, row-major. Logits are bf16 or fp32
 *    (spec_dtype). The library allocates nothing; it reads every logit once (plus, for the draw of each
 *    sequence, the one row pair it draws from) and writes only the outputs and the caller's workspace.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream). Calls are asynchronous:
 *    they enqueue kernels and return without synchronising.
 *  - Uniforms: Philox4x32-10 (Salmon et al., SC'11) with key = seeds[b] (low word, high word) and counter
 *    (position j, sequence b, stream, 0); output word 0 maps to ((w >> 9) + 0.5) * 2^-23. Stream 0 gives
 *    the accept uniform r of position j; stream 1 gives the resample uniform u of position j (or of the
 *    bonus row at j = K).
 *  - Inverse CDF in ascending token id: the emitted token is the smallest x whose running mass exceeds
 *    u * (total mass). A token with zero mass is never emitted.
 *  - Arguments are validated on the host before anything is launched; a bad argument returns
 *    SPEC_ERR_INVALID (message in spec_last_error()) and enqueues nothing. A CUDA launch failure returns
 *    SPEC_ERR_CUDA. Draft tokens live on the device and are checked there: a token outside [0, V) sets
 *    bit SPEC_STATUS_BAD_TOKEN of the workspace status word (read with spec_read_status) and that position
 *    is verified as if the draft had proposed a token of probability 0 under both models.
 *  - Every row must hold at least one finite logit; -inf logits are allowed (probability 0). NaN or +inf
 *    logits give unspecified results.
 *  - Limits: 1 <= K <= 64, 1 <= V <= 262144, 1 <= N <= 64, temperature > 0 and finite (temperature 0,
 *    greedy decoding, returns SPEC_ERR_UNSUPPORTED), delta >= 0 and finite. B = 0 is a no-op.
 *  - Workspace: caller-provided device memory of at least spec_workspace_size(B, K, V, N) bytes, 16-byte
 *    aligned. Its first word is the status word: zero it once before first use (spec_clear_status or a
 *    memset); calls only OR bits into it. The rest is scratch for per-position records and holds nothing
 *    a later call depends on. Calls that share a workspace must not overlap on the GPU.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID = 1,
    SPEC_ERR_CUDA = 2,
    SPEC_ERR_UNSUPPORTED = 3
} spec_status;

typedef enum { SPEC_BF16 = 0, SPEC_FP32 = 1 } spec_dtype;

/* Bits of the device status word. */
#define SPEC_STATUS_BAD_TOKEN 1u /* a draft token was outside [0, V) */
#define SPEC_STATUS_TIMEOUT 2u   /* a bounded wait for a bulk copy gave up (results invalid) */

/* Bytes of workspace the three calls need for these sizes (a pure function of the sizes; the same
 * buffer serves any call whose sizes are not larger). */
size_t spec_workspace_size(int B, int K, int V, int N);

/* Standard speculative sampling (tutorial §5.1 + §9.1).
 *  target_logits [B, K+1, V]  row K of each sequence is the bonus row
 *  draft_logits  [B, K, V]
 *  draft_tokens  int32 [B, K], the draft's proposals
 *  seeds         uint64 [B], Philox keys
 *  temperature   applied to both rows
 * Outputs (device):
 *  accept_len    int32 [B], number of accepted drafts L in [0, K]
 *  out_tokens    int32 [B, K+1]: the L accepted drafts, then the residual draw (L < K) or the bonus draw
 *                (L = K), then -1 padding
 *  diag          nullable float [B, K, 4]: per position (p_target(t), p_draft(t), Z, r) for every j, also
 *                after the chain stopped */
spec_status spec_verify(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                        const int32_t* draft_tokens, const uint64_t* seeds, int B, int K, int V,
                        float temperature, int32_t* accept_len, int32_t* out_tokens, float* diag,
                        void* workspace, size_t workspace_bytes, void* stream);

/* HedgeSpec counterfactual evaluation ("Not-a-Bandit ...", Key design 1 and 3).
 *  target_logits  [B, K+1, V]  (row K is read only when selected >= 0)
 *  drafter_logits [N, B, K, V]
 * Outputs: gamma float [N, B, K] = sum_x min(p_target, q_i) at every level j (all K levels; the caller
 * applies censoring with accept_len), loss nullable float [N, B, K] = 1 - gamma.
 * selected = -1: gamma only (draft_tokens, seeds, accept_len, out_tokens, diag may be NULL).
 * selected in [0, N): in the same pass, the chain of drafter `selected` is verified exactly as spec_verify
 * would with draft_logits = drafter_logits[selected]. */
spec_status spec_counterfactual_gamma(const void* target_logits, const void* drafter_logits,
                                      spec_dtype dtype, int N, int B, int K, int V, float temperature,
                                      float* gamma, float* loss, int selected,
                                      const int32_t* draft_tokens, const uint64_t* seeds,
                                      int32_t* accept_len, int32_t* out_tokens, float* diag,
                                      void* workspace, size_t workspace_bytes, void* stream);

/* Cactus constrained acceptance ("Cactus ...", Key design 1-3). Same layout and outputs as spec_verify,
 * plus delta >= 0 (the divergence budget) and gamma_star nullable float [B, K]. diag's first entry is
 * h(t) = gamma*. The bonus row is the plain target row. delta = 0 gives outputs bit-identical to
 * spec_verify. */
spec_status spec_cactus_verify(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                               const int32_t* draft_tokens, const uint64_t* seeds, int B, int K, int V,
                               float temperature, float delta, int32_t* accept_len, int32_t* out_tokens,
                               float* diag, float* gamma_star, void* workspace, size_t workspace_bytes,
                               void* stream);

/* Cactus with gamma* as the exact root of its divergence constraint ("Cactus ...", Key design 2: gamma* is
 * the root of D_KL(h || p_target) = delta on [q(n), +inf), clamped to [q(n), 1]; Key design 3 chooses the
 * KL divergence and then replaces the root by its second-order Taylor closed form, which spec_cactus_verify
 * uses). With h_n = g and the other tokens scaled by (1 - g) / (1 - q(n)) the divergence is
 * g ln(g / q(n)) + (1 - g) ln((1 - g) / (1 - q(n))); the root is found per position by a bracketed Newton
 * iteration in fp32. Same arguments, layout, outputs and errors as spec_cactus_verify; delta = 0 again gives
 * outputs bit-identical to spec_verify, and ln(1 / q(n)) <= delta gives gamma* = 1. */
spec_status spec_cactus_kl_verify(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                                  const int32_t* draft_tokens, const uint64_t* seeds, int B, int K, int V,
                                  float temperature, float delta, int32_t* accept_len, int32_t* out_tokens,
                                  float* diag, float* gamma_star, void* workspace, size_t workspace_bytes,
                                  void* stream);

/* Greedy verification: [SpS] §5.1 and the §9.1 chain at temperature 0, where the target and draft rows are
 * one-hot at their largest logit ("Speculative Decoding 为什么是 Lossless 的", §8 Q4: sampling transforms are
 * folded into p and q before the ratio). Then p(t) / q(t) is 1 when the draft token t is the argmax of
 * target row j and 0 otherwise, so draft j is accepted iff it is that argmax; the first rejecting row (or row
 * K when all K are accepted) emits its argmax. Ties among equal largest logits go to the smallest index (the
 * pages fix no rule). The draft logits and the uniforms drop out, so only the target rows are read.
 * target_logits: [B, K+1, V]; draft_tokens int32 [B, K]; outputs accept_len [B] and out_tokens [B, K+1]
 * (-1 padded) as spec_verify. A draft token outside [0, V) is a reject and sets SPEC_STATUS_BAD_TOKEN. A row
 * whose logits are all -inf has argmax 0. Workspace and errors as spec_verify (spec_workspace_size(B, K, V,
 * 1) bytes). */
spec_status spec_greedy_verify(const void* target_logits, spec_dtype dtype, const int32_t* draft_tokens, int B,
                               int K, int V, int32_t* accept_len, int32_t* out_tokens, void* workspace,
                               size_t workspace_bytes, void* stream);

/* HedgeSpec accept-length estimate and loss from the counterfactual gamma ("Not-a-Bandit ...", Key design
 * 2: a one-trajectory estimate of a drafter's expected accept length, in [1, K + 1]; Key design 3: the loss
 * is the accept length still available up to K + 1). The page's displays of both formulas are missing;
 * the reading taken is est[i, b] = 1 + sum_{k=1..K} prod_{j<=k} gamma[i, b, j] (the expected tokens of a
 * chain accepting level k with probability gamma_k given the levels before it) and loss[i, b] = K + 1 -
 * est[i, b]. gamma: device float [N, B, K], as written by spec_counterfactual_gamma; est: device float
 * [N, B]; loss: nullable device float [N, B]. All levels are used: a caller that censors by the accepted
 * length passes gamma with the censored levels as it wants them. Asynchronous on `stream`; allocates
 * nothing. */
spec_status spec_accept_length_estimate(const float* gamma, int N, int B, int K, float* est, float* loss,
                                        void* stream);

/* One round of NormalHedge (Chaudhuri, Freund, Hsu, "A parameter-free hedging algorithm", NIPS 2009), the
 * learner the HedgeSpec notes name for picking the drafter ("Not-a-Bandit ...", Key design 3; the pages
 * give no update rule). weights: device float [N], the distribution the learner played this round, replaced
 * by the next one; loss: device float [N], this round's loss per drafter (for example 1 - gamma at a level,
 * or the accept-length loss); regret: device float [N], the cumulative regret, updated in place by
 * (weights . loss) - loss. Next weights: p_i proportional to ([R_i]+ / c) exp([R_i]+^2 / (2 c)) with c solving
 * (1/N) sum_i exp([R_i]+^2 / (2 c)) = e; uniform when no regret is positive. Start from regret 0 and uniform
 * weights. For the notes' delayed, censored feedback, spec_hedge_feedback_push keeps the queue and applies
 * this rule to each loss as it becomes available. 1 <= N <= 64. One warp; asynchronous on `stream`; allocates nothing. */
spec_status spec_normalhedge_update(float* regret, const float* loss, float* weights, int N, void* stream);

/* NormalHedge under delayed, censored feedback, one learner per sequence ("Not-a-Bandit ...", Key design 3:
 * the accepted tokens of a round are revealed as one block when the round ends; the counterfactual feedback
 * is censored unless the selected drafter fills the chunk; the loss is 1 - gamma or the accept length still
 * available up to K + 1; the delay is at most 2K; in practice the learner keeps a queue of feedback and keeps
 * applying the next available one, the stochastic-setting reduction of Joulani, Gyorgy, Szepesvari, "Online
 * learning under delayed feedback", ICML 2013). The notes give no pseudo-code; the reading taken:
 *  - each round, spec_hedge_feedback_push receives the round's counterfactual gamma [N, B, K] (as written by
 *    spec_counterfactual_gamma) and the accepted length accept_len [B] of the selected drafter. For sequence
 *    b, levels j < min(accept_len[b] + 1, K) have a fully verified context and are appended, in level order,
 *    to the sequence's queue of feedback items; the levels after them are censored and never used;
 *  - objective 0 (acceptance probability): an item's loss is 1 - gamma, available at once;
 *    objective 1 (accept length): item n's loss is K + 1 minus the accept-length estimate of
 *    spec_accept_length_estimate over the window of items n .. n + K - 1, available once item n + K - 1 has
 *    arrived (so at most 2K - 1 items are ever pending);
 *  - every newly available loss is applied, oldest item first, as one NormalHedge round
 *    (spec_normalhedge_update's rule); items whose window never completes are never applied.
 * State: caller-owned device memory of spec_hedge_feedback_state_size(N, B, K) bytes, 16-byte aligned, set up
 * by spec_hedge_feedback_init (regrets 0, uniform weights, empty queues, the objective). Outputs of a push
 * (device, nullable): weights [B, N], the distribution for the next round; applied [B], the NormalHedge rounds
 * applied so far. An accepted length outside [0, K] skips that sequence's round and sets bit 1 of the status
 * word at byte 16 of the sequence's state. 1 <= N <= 64, 1 <= K <= 64; one warp per sequence; asynchronous on
 * `stream`; pushes on one state must not overlap on the GPU. Allocates nothing. */
size_t spec_hedge_feedback_state_size(int N, int B, int K);
spec_status spec_hedge_feedback_init(void* state, int N, int B, int K, int objective, void* stream);
spec_status spec_hedge_feedback_push(void* state, const float* gamma, const int32_t* accept_len, int N, int B, int K,
                                     float* weights, int32_t* applied, void* stream);

/* Bytes of workspace spec_verify_filtered needs: the spec_verify workspace; per target and draft row its
 * threshold and the kept logits' (max, sum); per target row a list of up to 1024 kept logits (index and
 * value) for the draw. No filtered copy of the logits is made: the kernels mask each logit as they read it.
 * 0 for invalid sizes or dtype. */
size_t spec_filter_workspace_size(int B, int K, int V, spec_dtype dtype);

/* spec_verify with standardised sampling ("Speculative Decoding 为什么是 Lossless 的", §8 Q4: temperature,
 * top-k and top-p are folded into p and q, the same transforms on the target and the draft row, before the
 * ratio). Each target and draft row keeps the logits at or above its threshold: top_k (0 or >= V: none)
 * keeps the values at or above the k-th largest, then top_p (1: none) keeps, of those, the values at or
 * above the one at which the renormalised mass summed from the largest logit down first reaches top_p. The
 * other logits become -inf, and the chain is spec_verify's on the filtered rows. Readings (the pages give
 * neither rule): ties at a threshold are all kept, top-k comes before top-p. Same arguments, outputs and
 * errors as spec_verify, plus top_k >= 0 and top_p in (0, 1]; the workspace must hold
 * spec_filter_workspace_size(B, K, V, dtype) bytes (its first 16 bytes zeroed once, as for spec_verify). The
 * thresholds come from an exact selection on order-preserving integer keys of the logits; top-p sums fp32
 * masses in 2^-44 fixed point, so a top-p decision within about 1e-6 of the mass boundary may differ from
 * an exact-arithmetic one. */
spec_status spec_verify_filtered(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                                 const int32_t* draft_tokens, const uint64_t* seeds, int B, int K, int V,
                                 float temperature, int top_k, float top_p, int32_t* accept_len, int32_t* out_tokens,
                                 float* diag, void* workspace, size_t workspace_bytes, void* stream);

/* spec_verify for callers that cannot allocate device memory: same inputs, outputs and semantics, but no
 * workspace argument. Some callers run where allocation is not allowed or not possible: inside a memory
 * budget fixed in advance, under an allocator that must not grow, or from code that has no allocator at all.
 * The pages have no counterpart of this entry point; it only changes where the scratch lives.
 *  - Scratch: a fixed 32 MiB region of device memory inside the library (one per device, part of the loaded
 *    library image). A call whose workspace would exceed it (spec_workspace_size(B, K, V, 1) > 32 MiB)
 *    returns SPEC_ERR_UNSUPPORTED before any CUDA call; spec_verify with a caller workspace has no such
 *    limit.
 *  - The first call on each device looks the region's address up (cudaGetSymbolAddress, with that device
 *    current); make it before any stream capture.
 *  - The region's first word is the status word, the only part that must start at zero: the region starts
 *    zeroed, and every call clears the word on `stream` before its kernels run.
 *  - All calls on one device share the region: calls that can overlap on the GPU (different streams, or
 *    several host threads) race on it and give wrong results. Serialise them.
 *  - status_out: nullable host pointer. When given, the call also waits for `stream` and stores this call's
 *    status bits (SPEC_STATUS_*) there.
 * Nothing is allocated: no cudaMalloc, no allocating library routine. */
spec_status spec_verify_static(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                               const int32_t* draft_tokens, const uint64_t* seeds, int B, int K, int V,
                               float temperature, int32_t* accept_len, int32_t* out_tokens, float* diag,
                               uint32_t* status_out, void* stream);

/* Copies the workspace status word to *status_out (host), synchronising `stream`. */
spec_status spec_read_status(const void* workspace, uint32_t* status_out, void* stream);

/* Zeroes the first 16 bytes of the workspace: the status word and three words the library keeps for its own
 * bookkeeping between calls (asynchronous on `stream`). */
spec_status spec_clear_status(void* workspace, void* stream);

/* Thread-local message describing the last non-OK status returned on this thread. */
const char* spec_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
