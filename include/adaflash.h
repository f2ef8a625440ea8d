/*
 * adaflash.h -- C ABI of the packed verify + on-policy-distillation (OPD) loss pass.
 *
 * The operations come from the page "AdaFlash: Adaptive Speculative Decoding with
 * Online Self-Improvement for High-Concurrency LLM Inference" (below: the AdaFlash
 * article) and the page "AdaFlash: Adaptive Speculative Decoding via On-Policy
 * Distilled Diffusion Drafters" (below: the AdaFlash README).
 *
 * Packed layout ("Variable-length request packing", AdaFlash article): R requests
 * with draft lengths 1 <= k_i <= 16 share one batch.  draft_offsets (int32, R+1
 * entries) is the exclusive prefix sum of the k_i, so draft_offsets[0] = 0 and
 * draft_offsets[R] = N_d, the number of draft rows.  Request i owns
 *   - draft rows   draft_offsets[i] .. draft_offsets[i+1]-1      (k_i rows),
 *   - target rows  draft_offsets[i]+i .. draft_offsets[i+1]+i    (k_i+1 rows),
 * so there are N_t = N_d + R target rows.  Draft row draft_offsets[i]+j is paired
 * with target row draft_offsets[i]+i+j (the target's distribution at the position
 * of draft token j); target row draft_offsets[i+1]+i is the request's bonus row.
 *
 * Logit matrices are row-major: row r of a matrix with leading dimension ld starts
 * at element r*ld; columns ld > vocab are never read.  Element types: float32 or
 * bfloat16 (ADAFLASH_FP32 / ADAFLASH_BF16); supported (draft, target) pairs are
 * (fp32, fp32), (bf16, bf16), (fp32, bf16) and (bf16, fp32).  Any element-aligned
 * base pointer and any ld >= vocab are accepted.  Every row is bulk-copied: the
 * entries before a target row's first 16-byte boundary (under 16 bytes of them) are
 * read one by one, and a draft row that is off that grid is copied from the 16-byte
 * boundary just below it.
 *
 * Empty batch: num_requests = num_draft_rows = 0 is valid.  Nothing is read and no
 * kernel is launched, so the row, token, offset and per-row output pointers may be
 * NULL; the scalar arguments are still checked, and an entry point with a loss
 * output sets *loss = 0 (its loss pointer must be valid).
 *
 * Ownership and ordering: every pointer argument of the GPU entry points is a
 * DEVICE pointer owned by the caller.  They allocate no device memory, keep no device
 * state between calls and never synchronise: each call enqueues its kernels on `stream` (a
 * cudaStream_t; NULL is the legacy default stream) and returns.  Calls on one stream
 * run in order.  Several host threads may call at once (each on its own stream): the
 * small host-side tables the library fills on first use (occupancy per kernel and
 * cluster size, kernel shared-memory limits, device attributes) are locked or atomic.
 * The packer entry points (below) work on host memory only.
 *
 * Errors:
 *   - Argument errors found on the host are returned at once and nothing is
 *     enqueued (ADAFLASH_ERR_INVALID_ARG, ADAFLASH_ERR_UNSUPPORTED).
 *   - A failed CUDA launch returns ADAFLASH_ERR_CUDA.
 *   - Errors only the device can see are OR-ed into *d_status as bit
 *     (1u << code), e.g. (1u << ADAFLASH_ERR_BAD_OFFSETS); d_status may be NULL
 *     to ignore them.  The library never clears *d_status.  A row or request
 *     with such an error is skipped (its outputs are left unwritten, or set to
 *     -1 where stated); the kernels never trap or fault on bad device data.
 *
 * Device: compute capability 10.3 (GB300, sm_103a).  Any other device gives
 * ADAFLASH_ERR_UNSUPPORTED.
 */
#ifndef ADAFLASH_H
#define ADAFLASH_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ADAFLASH_OK = 0,
  ADAFLASH_ERR_INVALID_ARG = 1, /* host: NULL pointer, vocab < 1, ld < vocab, bad dtype, bad counts, clip_c not > 0 */
  ADAFLASH_ERR_UNSUPPORTED = 2, /* host: device is not cc 10.3, or vocab above the supported maximum */
  ADAFLASH_ERR_CUDA = 3,        /* host: a CUDA runtime call or launch failed */
  ADAFLASH_ERR_TIMEOUT = 4,     /* device bit: a bounded wait gave up; that row's outputs are invalid */
  ADAFLASH_ERR_BAD_OFFSETS = 5, /* device bit: draft_offsets not a prefix sum of k_i in [1,16] ending at N_d */
  ADAFLASH_ERR_BAD_TOKEN = 6    /* device bit: a draft token outside [0, vocab); it never counts as accepted */
} adaflash_status;

typedef enum { ADAFLASH_FP32 = 0, ADAFLASH_BF16 = 1 } adaflash_dtype;

/* Largest vocabulary the kernels accept (8 CTAs x 65536 entries per row). */
#define ADAFLASH_MAX_VOCAB 524288
/* Largest draft length of one request (the fixed verification length k = 16 of
 * the AdaFlash article, section "2. Adaptive Length Head for Token-Level Variance"). */
#define ADAFLASH_MAX_K 16

/*
 * adaflash_verify_packed -- greedy verification of packed draft blocks.
 *
 * The draft model proposes k_i tokens and the target verifies them in parallel
 * (AdaFlash article, opening section); the true acceptance rate is the length
 * head's free label (section "2. Adaptive Length Head for Token-Level Variance").
 * Greedy reading: the target's choice at a position is the lowest index of the
 * row maximum; draft token j is accepted while it equals that choice.
 *
 *   target_logits  [N_t, ld_t] of t_dtype          in
 *   draft_tokens   int32 [N_d]                      in
 *   draft_offsets  int32 [R+1]                      in
 *   target_argmax  int32 [N_t]                      out: lowest index of each target row's maximum
 *   accept_len     int32 [R]                        out: L_i = first j with token != choice, else k_i
 *   bonus_token    int32 [R]                        out: target choice at target row draft_offsets[i]+i+L_i
 *   accept_rate    float [R]                        out: L_i / k_i rounded once to float32
 * A request with malformed offsets gets accept_len = bonus_token = -1.
 */
adaflash_status adaflash_verify_packed(
    const void* target_logits, adaflash_dtype t_dtype, int64_t ld_t,
    const int32_t* draft_tokens, const int32_t* draft_offsets,
    int32_t num_requests, int32_t num_draft_rows, int32_t vocab,
    int32_t* target_argmax, int32_t* accept_len, int32_t* bonus_token, float* accept_rate,
    uint32_t* d_status, void* stream);

/*
 * adaflash_opd_loss_fwd -- fused verification + OPD loss forward (one read of every logit).
 *
 * For each draft row d (request i, position j) with draft logits z and paired
 * target logits t, p = softmax(z), q = softmax(t), r_v = log p_v - log q_v:
 *   kl_row[d] = sum_v min(p_v r_v, clip_c)  -- the reverse KL(p||q) with each
 *               vocabulary term clipped before the sum (AdaFlash article,
 *               "Reverse KL + Top-1 hard labels" and "Per-vocabulary divergence
 *               clipping"; the clip bounds terms from above);
 *   ce_row[d] = -log p_a, a = target_argmax of the paired target row
 *               ("Top-1 hard labels from the target");
 *   loss[0]   = (1/N_d) sum_d (kl_row[d] + ce_weight * ce_row[d])  (the
 *               "mixture reverse-KL loss" of the AdaFlash README, "Released Checkpoint").
 * It also produces every output of adaflash_verify_packed, and
 *   row_stats [N_d, 4] float: {logsumexp(z), logsumexp(t), S, n_clipped} with
 *               S = sum_v [p_v r_v <= clip_c] p_v (r_v + 1); pass it to the backward.
 * clip_c must be > 0 (+inf disables the clip); ce_weight is the mixture weight.
 */
adaflash_status adaflash_opd_loss_fwd(
    const void* draft_logits, adaflash_dtype d_dtype, int64_t ld_d,
    const void* target_logits, adaflash_dtype t_dtype, int64_t ld_t,
    const int32_t* draft_tokens, const int32_t* draft_offsets,
    int32_t num_requests, int32_t num_draft_rows, int32_t vocab,
    float clip_c, float ce_weight,
    int32_t* target_argmax, int32_t* accept_len, int32_t* bonus_token, float* accept_rate,
    float* kl_row, float* ce_row, float* row_stats, float* loss,
    uint32_t* d_status, void* stream);

/*
 * adaflash_opd_loss_bwd -- gradient of the OPD loss with respect to the draft logits.
 *
 * Training updates the serving draft model from each round's verification
 * (AdaFlash article, "On-Policy Distillation (OPD) for Domain Adaptation"); the
 * target is a constant (it is never updated).  With g_r =
 * grad_row[r] (or grad_scale when grad_row is NULL), m_v = [p_v r_v <= clip_c]
 * and a the target argmax:
 *   grad_draft[r, v] = g_r * ( p_v (m_v (r_v + 1) - S) + ce_weight (p_v - [v == a]) )
 * where S and the two log-sum-exps come from row_stats of the forward and a from
 * its target_argmax.  grad_draft is float32 [N_d, ld_g]; columns >= vocab are not
 * written.  grad_scale = 1/N_d gives the gradient of the mean loss.
 */
adaflash_status adaflash_opd_loss_bwd(
    const void* draft_logits, adaflash_dtype d_dtype, int64_t ld_d,
    const void* target_logits, adaflash_dtype t_dtype, int64_t ld_t,
    const int32_t* draft_offsets, int32_t num_requests, int32_t num_draft_rows, int32_t vocab,
    float clip_c, float ce_weight,
    const int32_t* target_argmax, const float* row_stats,
    const float* grad_row, float grad_scale,
    float* grad_draft, int64_t ld_g,
    uint32_t* d_status, void* stream);

/*
 * adaflash_opd_loss_fwd_bwd -- the forward and the backward in one call.
 *
 * The drafter takes a training step right after each verification round (AdaFlash
 * article, "On-Policy Distillation (OPD) for Domain Adaptation"), so the upstream
 * weights are known when the forward runs.  Outputs and arguments are those of
 * adaflash_opd_loss_fwd followed by adaflash_opd_loss_bwd with the same clip_c,
 * ce_weight, grad_row and grad_scale; the integer outputs are equal to theirs and
 * the float outputs agree to float32 rounding (a row's partial sums may be combined
 * in another order).  When every row of draft_logits, target_logits and grad_draft
 * starts on a 16-byte boundary, each logit is read from HBM once for both passes:
 * for at most one wave of row units with every row pair held on chip (a cluster of
 * at most 8 CTAs) while its statistics are combined, then dz written from there;
 * for larger batches by a row pass that reads each slice again, from L2, once the
 * row's statistics are known.  Rows off that grid take the separate forward and
 * backward kernels.
 */
adaflash_status adaflash_opd_loss_fwd_bwd(
    const void* draft_logits, adaflash_dtype d_dtype, int64_t ld_d,
    const void* target_logits, adaflash_dtype t_dtype, int64_t ld_t,
    const int32_t* draft_tokens, const int32_t* draft_offsets,
    int32_t num_requests, int32_t num_draft_rows, int32_t vocab,
    float clip_c, float ce_weight, const float* grad_row, float grad_scale,
    int32_t* target_argmax, int32_t* accept_len, int32_t* bonus_token, float* accept_rate,
    float* kl_row, float* ce_row, float* row_stats, float* loss,
    float* grad_draft, int64_t ld_g,
    uint32_t* d_status, void* stream);

/*
 * adaflash_verify_sampled -- temperature-sampled verification of packed draft blocks.
 *
 * The target verifies the drafted tokens in parallel (AdaFlash article, opening
 * section) at the sampling temperature, a tunable of the method (page "Adaflash
 * Adaptive Speculative Decoding", section "Implementation Steps").  The rule is
 * speculative sampling, with p = softmax(z / T) of a draft row and q = softmax(t / T)
 * of its paired target row:
 *   - draft token x_j is accepted when u_accept[d] * p(x_j) < q(x_j), d its draft row;
 *     accept_len[i] = L_i is the number of tokens before the first rejection;
 *   - L_i < k_i: the emitted token is drawn from max(0, q - p) at position L_i
 *     (from q when that is all zero); L_i = k_i: from q at the bonus row;
 *   - a draw from weights pi with w = u_sample[i] is the smallest v whose prefix sum
 *     sum_{u<=v} pi_u exceeds w * sum_u pi_u (the inverse CDF in vocabulary order).
 * The uniforms are inputs, so the caller owns the random stream.  w is clamped to
 * [0, 1] (NaN -> 0); a NaN u rejects.  Logits are finite or -inf.
 *
 *   draft_logits   [N_d, ld_d] of d_dtype           in
 *   target_logits  [N_t, ld_t] of t_dtype           in
 *   draft_tokens   int32 [N_d]                      in
 *   draft_offsets  int32 [R+1]                      in
 *   temperature    T > 0 with 1/T finite            in
 *   u_accept       float [N_d]                      in: accept uniforms in [0, 1)
 *   u_sample       float [R]                        in: draw uniforms in [0, 1)
 *   row_lse        float [N_d + N_t]                out: logsumexp(x / T) of each draft row,
 *                                                        then of each target row
 *   accept_len     int32 [R]                        out: L_i
 *   next_token     int32 [R]                        out: the emitted token
 *   accept_rate    float [R]                        out: L_i / k_i rounded once to float32
 * A request with malformed offsets gets accept_len = next_token = -1, accept_rate = -1.
 * A draft token outside [0, vocab) is rejected and sets ADAFLASH_ERR_BAD_TOKEN.
 */
adaflash_status adaflash_verify_sampled(
    const void* draft_logits, adaflash_dtype d_dtype, int64_t ld_d,
    const void* target_logits, adaflash_dtype t_dtype, int64_t ld_t,
    const int32_t* draft_tokens, const int32_t* draft_offsets,
    int32_t num_requests, int32_t num_draft_rows, int32_t vocab,
    float temperature, const float* u_accept, const float* u_sample,
    float* row_lse, int32_t* accept_len, int32_t* next_token, float* accept_rate,
    uint32_t* d_status, void* stream);

/*
 * The logit-free forward: verification and OPD loss from final hidden states.
 *
 * A row's logits are its LM head applied to its final hidden state: z = W_d h_d for
 * a draft row, t = W_t h_t for a target row.  adaflash_lmhead_opd_fwd produces every
 * output of adaflash_opd_loss_fwd (same meaning, same layouts) from the hidden
 * states and the two heads, without writing the logits: a tensor-core GEMM (tcgen05,
 * bf16 x bf16 -> f32) reduces each 128-row x 256-entry tile of z and t to per-row
 * statistics in the caller's workspace, a per-row pass combines them and
 * re-evaluates exactly (dot products) only the entries whose clipped term can
 * exceed clip_c, then the acceptance scan and the loss follow.
 *
 *   draft_hidden   bf16 [N_d, ld_hd]    in   (row d: the draft's hidden state at draft row d)
 *   target_hidden  bf16 [N_t, ld_ht]    in   (packed like target_logits: N_t = N_d + R rows)
 *   draft_head     bf16 [V, ld_wd]      in
 *   target_head    bf16 [V, ld_wt]      in   (may be the same pointer as draft_head)
 *   hidden         H, a multiple of 64; every ld >= H and a multiple of 8; every matrix
 *                  16-byte aligned
 *   workspace      device memory of at least adaflash_lmhead_workspace_bytes(R, N_d, V, H)
 *                  bytes, 256-byte aligned, owned by the caller, overwritten
 *   other arguments and outputs: as adaflash_opd_loss_fwd
 * adaflash_lmhead_workspace_bytes returns -1 for invalid sizes.
 *
 * adaflash_lmhead_logits writes the logits of `rows` hidden rows under one head,
 * logits[r, v] = sum_k h[r, k] w[v, k] (float32 [rows, ld_out]), with the same GEMM;
 * it is there to check and time the tensor-core product on its own.
 */
int64_t adaflash_lmhead_workspace_bytes(int32_t num_requests, int32_t num_draft_rows, int32_t vocab, int32_t hidden);

adaflash_status adaflash_lmhead_logits(const void* hidden_rows, int64_t ld_h, int32_t rows, const void* head,
                                       int64_t ld_w, int32_t vocab, int32_t hidden, float* logits, int64_t ld_out,
                                       uint32_t* d_status, void* stream);

adaflash_status adaflash_lmhead_opd_fwd(
    const void* draft_hidden, int64_t ld_hd, const void* target_hidden, int64_t ld_ht,
    const void* draft_head, int64_t ld_wd, const void* target_head, int64_t ld_wt, int32_t hidden,
    const int32_t* draft_tokens, const int32_t* draft_offsets,
    int32_t num_requests, int32_t num_draft_rows, int32_t vocab,
    float clip_c, float ce_weight, void* workspace, int64_t workspace_bytes,
    int32_t* target_argmax, int32_t* accept_len, int32_t* bonus_token, float* accept_rate,
    float* kl_row, float* ce_row, float* row_stats, float* loss,
    uint32_t* d_status, void* stream);

/*
 * adaflash_lmhead_opd_fwd_static -- adaflash_lmhead_opd_fwd without a workspace argument.
 *
 * The pages have no counterpart: this entry point is for callers that cannot hand
 * the library device memory.  A plugin called by a host framework that owns every
 * allocation (an inference server's custom-op slot, a runtime with its own pooled
 * allocator) may have no way to call cudaMalloc, or may be forbidden to because an
 * allocation would synchronise the device or break the framework's memory
 * accounting.  Such a caller passes only its inputs and outputs; the scratch the
 * logit-free forward needs (the gathered hidden rows and the per-tile records) lives
 * in one static device array of ADAFLASH_LMHEAD_STATIC_SCRATCH_BYTES inside this
 * library, which every GPU that loads the library's LM-head code holds until the
 * process exits.
 *
 * Arguments, outputs and results are those of adaflash_lmhead_opd_fwd, and bad
 * arguments get the same status from both.  A batch whose
 * adaflash_lmhead_workspace_bytes(R, N_d, V, H) exceeds the array is rejected with
 * ADAFLASH_ERR_UNSUPPORTED before anything is enqueued.  The first call on a device
 * looks up the array's device address with that device current (set-up done once
 * per device); make that first call before any stream capture.  The array's device
 * memory is committed when the library's LM-head code is loaded on the device: with
 * CUDA's lazy module loading (the default) that is this first call, so make it
 * outside any region where the device may not allocate (a failure there returns
 * ADAFLASH_ERR_CUDA).  The address looked up is kept for the life of the process:
 * cudaDeviceReset, or destroying and recreating the device's primary context,
 * invalidates it, and this entry point is not supported after either.  Nothing here
 * calls cudaMalloc or cudaFree.  All calls share the one array and each leaves its contents
 * behind: a call writes every scratch byte it reads before reading it, so nothing is
 * cleared, but calls whose kernels overlap on the GPU (other streams, other host
 * threads) race on the array and must be serialised by the caller.
 */
#define ADAFLASH_LMHEAD_STATIC_SCRATCH_BYTES (48ll << 20)

adaflash_status adaflash_lmhead_opd_fwd_static(
    const void* draft_hidden, int64_t ld_hd, const void* target_hidden, int64_t ld_ht,
    const void* draft_head, int64_t ld_wd, const void* target_head, int64_t ld_wt, int32_t hidden,
    const int32_t* draft_tokens, const int32_t* draft_offsets,
    int32_t num_requests, int32_t num_draft_rows, int32_t vocab,
    float clip_c, float ce_weight,
    int32_t* target_argmax, int32_t* accept_len, int32_t* bonus_token, float* accept_rate,
    float* kl_row, float* ce_row, float* row_stats, float* loss,
    uint32_t* d_status, void* stream);

/*
 * Variable-length request packing with an EMA capacity estimate (host side).
 *
 * The AdaFlash article ("Infrastructure: Async Training & Variable-Length Batching",
 * "Variable-length request packing") packs requests of different predicted
 * verification lengths into compact batches and sizes the next round with an
 * exponential moving average, to use the GPU well without running out of memory.
 * Reading: a request of predicted draft length k (1..16) occupies 2k + 1 logit rows
 * (k draft rows, k + 1 target rows); a round holds at most row_budget rows; the
 * estimate e of rows per request follows e <- alpha*x + (1 - alpha)*e with x a
 * round's rows / requests (float64, that order); a round takes
 * capacity = max(1, floor(row_budget / e)) requests from the front of the queue,
 * gives back the last ones while their rows exceed row_budget, and packs the rest
 * back to back.
 *
 * All pointers here are HOST pointers; nothing touches the GPU.  The packer is a
 * small host object owned by the caller (create / destroy); calls on one packer
 * must not run concurrently.
 *
 *   adaflash_packer_create   row_budget >= 33, 0 < alpha <= 1, initial estimate > 0
 *   adaflash_packer_plan     queue_k int32 [n_queue] in 1..16 (queue order)    in
 *                            draft_offsets int32 [n_queue + 1]                  out: [0..num_admitted] written
 *                            num_admitted, capacity, rows (int32 each)          out
 *                            the estimate is not changed
 *   adaflash_packer_observe  a finished round's rows and requests: one EMA step (none if requests == 0)
 *   adaflash_packer_estimate the current estimate of rows per request
 * Errors: ADAFLASH_ERR_INVALID_ARG for NULL pointers, out-of-range arguments or a k
 * outside 1..16 (nothing is written then).
 */
typedef struct adaflash_packer adaflash_packer;

adaflash_status adaflash_packer_create(int32_t row_budget, double alpha, double initial_rows_per_request,
                                       adaflash_packer** out);
adaflash_status adaflash_packer_destroy(adaflash_packer* packer);
adaflash_status adaflash_packer_plan(const adaflash_packer* packer, const int32_t* queue_k, int32_t n_queue,
                                     int32_t* draft_offsets, int32_t* num_admitted, int32_t* capacity,
                                     int32_t* rows);
adaflash_status adaflash_packer_observe(adaflash_packer* packer, int32_t rows, int32_t requests);
adaflash_status adaflash_packer_estimate(const adaflash_packer* packer, double* rows_per_request);

/* Number of kernel launches this library has enqueued in this process so far
 * (all entry points, all devices).  For instrumentation: the difference over a
 * region of calls counts the kernels that region launched. */
uint64_t adaflash_kernel_launches(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* adaflash_status_string(adaflash_status status);

/*
 * adaflash_selftest_bounded_wait -- exercises the bounded-wait error path.
 *
 * Launches one block that waits on a shared-memory barrier nothing ever
 * completes, with a limit of `limit_us` microseconds (1 .. 1000000); the wait
 * gives up, the block sets bit (1u << ADAFLASH_ERR_TIMEOUT) in *d_status and
 * returns.  This is the same wait routine the streaming kernels use, so a test
 * can check on a real device that a stuck wait ends in a status, not a hang.
 * The pages have no counterpart: it is part of this library's failure handling.
 */
adaflash_status adaflash_selftest_bounded_wait(uint32_t* d_status, int32_t limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ADAFLASH_H */
