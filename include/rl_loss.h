/*
 * rl_loss.h — C ABI of the GB300 (sm_103a) fused token-level policy loss.
 *
 * What it computes: the GRPO objective with IcePop train/inference mismatch
 * suppression and no KL term, forward and backward in one call, as written in
 * "GLM-5: from Vibe Coding to Agentic Engineering", section 3.2 "Reasoning
 * RL", Eq. (1):
 *
 *   L = -(1/S) sum_i (1/|y_i|) sum_{t in i} m_t * pop(rho_t, 1/beta, beta)
 *                          * min(r_t A_i, clip(r_t, 1 - eps_low, 1 + eps_high) A_i)
 *
 *   rho_t = pi_old^train(y_t) / pi_old^infer(y_t)   = exp(logp_old - logp_infer)
 *   pop(rho) = rho if 1/beta <= rho <= beta, else 0  (pop_indicator: 1 instead of rho)
 *   r_t   = pi_theta^train(y_t) / pi_old^train(y_t) = exp(logp_t - logp_old)
 *   A_i   = (R_i - mean(R_group)) / (std(R_group) + adv_eps)    (group = G consecutive responses)
 *   logp_t = z_{t, y_t} - log sum_v exp(z_{t, v})   (log-softmax of the logits row z_t)
 *
 * with S responses in the batch (the expectation over prompts read as the
 * mean over the batch's S/G prompts, so 1/(S/G) * 1/G = 1/S), |y_i| the number
 * of mask=1 tokens of response i (tool/environment tokens carry mask 0:
 * "Zhipu AI / GLM: From Blank Infilling to Compaction-Aware Agentic
 * Reinforcement Learning", section 9.4), and m_t the loss mask. Alongside the
 * loss it writes dL/dlogits, the per-token log-prob and entropy (the entropy
 * collapse the GLM-5 page watches in section 3.2, "DSA RL insights"), the
 * per-token pop/clip flags and counters.
 *
 * Every floating-point reduction runs in a fixed order that depends only on
 * the shapes, so repeated calls on the same inputs give bit-identical outputs
 * (the section-3.2 lesson that non-deterministic GPU kernels collapsed RL).
 *
 * Conventions shared by every entry point:
 *  - Pointers inside rl_loss_inputs / rl_loss_outputs are DEVICE pointers on
 *    the handle's device (except the `host` inputs of
 *    rl_loss_forward_backward_from_host); the caller owns them. The handle owns
 *    only its workspace, allocated once by rl_loss_create and freed by
 *    rl_loss_destroy.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream). Work is enqueued asynchronously; no call below synchronises
 *    except rl_loss_get_device_status and rl_loss_profile_read. One handle must
 *    not be used on two streams at the same time (it has one workspace).
 *  - Argument, shape, alignment and capacity errors are detected on the host
 *    and returned before anything is launched; outputs are then untouched.
 *  - Data-dependent problems (a target id outside [0, V), a response with no
 *    mask=1 token, malformed cu_seqlens) are detected on the device and set
 *    bits (1u << rl_status code) in the handle's device status word, read with
 *    rl_loss_get_device_status. Kernels never trap.
 */
#ifndef RL_LOSS_H
#define RL_LOSS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define RL_LOSS_API __attribute__((visibility("default")))
#else
#define RL_LOSS_API
#endif

typedef enum rl_status {
    RL_OK = 0,
    RL_ERR_INVALID_ARG = 1,   /* NULL handle / required pointer, bad hyper-parameter */
    RL_ERR_SHAPE = 2,         /* num_tokens / num_seqs / ld out of range, S % G != 0 */
    RL_ERR_DTYPE = 3,         /* unknown dtype code */
    RL_ERR_ALIGNMENT = 4,     /* logits / dlogits base or row stride not 16-byte aligned */
    RL_ERR_CAPACITY = 5,      /* num_tokens > max_tokens or num_seqs > max_seqs */
    RL_ERR_CUDA = 6,          /* a CUDA runtime call or launch failed */
    RL_ERR_TARGET_RANGE = 7,  /* device bit: some target id outside [0, V) (token excluded) */
    RL_ERR_NONFINITE = 8,     /* device bit: a logits row holds NaN or +inf, or the loss is not finite */
    RL_ERR_EMPTY_SEQ = 9,     /* device bit (warning): a response has no mask=1 token; it adds 0 */
    RL_ERR_TIMEOUT = 10,      /* device bit: a bounded wait ran out */
    RL_ERR_UNSUPPORTED = 11,  /* valid request the library does not implement */
    RL_ERR_SEQLENS = 12,      /* device bit: cu_seqlens not monotone or not ending at num_tokens */
    RL_ERR_DEVICE = 13,       /* called with another CUDA device current than the handle's */
    RL_ERR_INTERNAL = 14      /* device bit: an internal consistency check failed; that result is invalid */
} rl_status;

typedef enum rl_dtype { RL_F32 = 0, RL_BF16 = 1 } rl_dtype;

typedef enum rl_adv_mode {
    RL_ADV_GROUP_REWARDS = 0, /* rewards_or_adv = R [S]; A_i normalised per group of G */
    RL_ADV_PER_SEQ = 1,       /* rewards_or_adv = A [S] given, e.g. teacher_score - student_score
                                 with G = 1 ("2.5 GLM-5 -- 异步 Agentic RL 工程", Cross-Stage Distillation) */
    RL_ADV_PER_TOKEN = 2,     /* rewards_or_adv = A [T] given per token (e.g. from a critic) */
    RL_ADV_TEACHER_LOGP = 3   /* rewards_or_adv = log pi_teacher(y_t) [T]: A_t = sg[log pi_teacher(y_t) - logp_t],
                                 on-policy distillation ("GLM-5: from Vibe Coding to Agentic Engineering",
                                 section 3.5, Eq. (2)); its sign is taken in fp32 from the kernel's logp */
} rl_adv_mode;

typedef enum rl_objective {
    RL_OBJ_GRPO_ICEPOP = 0,   /* Eq. (1): pop(rho) min(r A, clip(r) A), r = exp(logp - logp_old) */
    RL_OBJ_DIS = 1            /* direct double-sided importance sampling (section 4.1.2, Eqs. (3)-(5)):
                                 f(r) A logp with r = exp(logp - logp_infer) (the rollout log-prob) and
                                 f(r) = r on the open interval (1 - eps_low, 1 + eps_high), else 0;
                                 logp_old and beta are not used; not with RL_ADV_TEACHER_LOGP */
} rl_objective;

typedef enum rl_loss_norm {
    RL_NORM_PER_RESPONSE = 0, /* weight 1/(S |y_i|): the 1/G, 1/|y_i| of Eq. (1) with E_x the mean over prompts */
    RL_NORM_PER_TOKEN = 1     /* weight 1/sum_i |y_i|: the mean over every generated token of the batch */
} rl_loss_norm;

/* Per-token flag bits written to rl_loss_outputs.flags. */
#define RL_FLAG_POP_IN_BOUNDS 0x1u /* 1/beta <= rho <= beta (decided in fp32: -fl32(ln beta) <= fl32(lo - li) <= fl32(ln beta));
                                      with RL_OBJ_DIS: 1 - eps_low < r < 1 + eps_high (fl32(logp - li) strictly
                                      between fl32(ln(1 - eps_low)) and fl32(ln(1 + eps_high))) */
#define RL_FLAG_CLIP_ACTIVE 0x2u   /* clipped branch of min() taken: A>0 and fl32(logp - lo) > fl32(ln(1+eps_high)),
                                      or A<0 and fl32(logp - lo) < fl32(ln(1-eps_low)); its gradient is 0
                                      (RL_OBJ_GRPO_ICEPOP only) */
#define RL_FLAG_MASKED 0x4u        /* loss mask m_t == 0 */
#define RL_FLAG_BAD_TARGET 0x8u    /* target id outside [0, V): token excluded, logp = NaN */

typedef struct rl_loss_handle_s *rl_loss_t;

/* Static configuration; fixed for the life of a handle. */
typedef struct rl_loss_config {
    int32_t vocab_size;    /* V >= 1 */
    int32_t group_size;    /* G >= 1; responses of a group are consecutive */
    int32_t max_tokens;    /* capacity: largest num_tokens a call may pass (>= 0) */
    int32_t max_seqs;      /* capacity: largest num_seqs a call may pass (>= 1) */
    float eps_low;         /* 0 <= eps_low < 1 (0.2 on the page) */
    float eps_high;        /* eps_high >= 0 (0.28 on the page) */
    float beta;            /* beta > 1 (2 on the page) */
    float adv_eps;         /* >= 0, added to the group std (1e-6) */
    int32_t adv_mode;      /* rl_adv_mode */
    int32_t std_unbiased;  /* 0: population std (ddof 0), 1: ddof 1 (needs G >= 2) */
    int32_t pop_indicator; /* 0: pop returns rho (the printed operator), 1: returns 1 */
    int32_t logits_dtype;  /* rl_dtype of logits and of dlogits */
    int32_t objective;     /* rl_objective (0 = Eq. (1)) */
    int32_t loss_norm;     /* rl_loss_norm (0 = per response) */
    int32_t dis_stopgrad;  /* RL_OBJ_DIS only. The pages leave open whether f(r) is stop-gradient:
                              1 = f(r) is a constant (dL/dlogp = -w f(r) A),
                              0 = differentiated too (dL/dlogp = -w r A (1 + logp) inside the interval) */
} rl_loss_config;

/* One batch of T packed response tokens in S responses. */
typedef struct rl_loss_inputs {
    int32_t num_tokens;           /* T, 0 <= T <= max_tokens */
    int32_t num_seqs;             /* S, 1 <= S <= max_seqs, S % G == 0 */
    int64_t ld_logits;            /* row stride in elements, >= V; ld * elem_size % 16 == 0 */
    const void *logits;           /* [T, ld] logits_dtype, 16-byte aligned; rows are read up to V
                                     rounded up to 16 bytes (<= ld), the padding is never used */
    const int32_t *targets;       /* [T] sampled token ids y_t */
    const float *logp_old;        /* [T] log pi_old^train(y_t) */
    const float *logp_infer;      /* [T] log pi_old^infer(y_t), from the rollout engine */
    const uint8_t *mask;          /* [T] loss mask, nonzero = 1 */
    const int32_t *cu_seqlens;    /* [S+1] offsets: response i is tokens [cu[i], cu[i+1]); cu[0]=0, cu[S]=T */
    const float *rewards_or_adv;  /* [S] rewards (RL_ADV_GROUP_REWARDS) or advantages (RL_ADV_PER_SEQ);
                                     [T] advantages (RL_ADV_PER_TOKEN) or teacher log-probs (RL_ADV_TEACHER_LOGP) */
} rl_loss_inputs;

/* Where results go. Only `loss` and `dlogits` are required; NULL skips an output. */
typedef struct rl_loss_outputs {
    float *loss;          /* [1] L (rounded from loss_f64) */
    double *loss_f64;     /* [1] L accumulated in fp64, or NULL */
    void *dlogits;        /* [T, ld_dlogits] logits_dtype, dL/dlogits (columns >= V untouched).
                             May alias logits when ld_dlogits == ld_logits (in-place). */
    int64_t ld_dlogits;   /* >= V; ld * elem_size % 16 == 0 */
    float *logp;          /* [T] per-token log-prob, or NULL */
    float *entropy;       /* [T] per-token entropy of softmax(z_t) in nats, or NULL */
    uint8_t *flags;       /* [T] RL_FLAG_* bits, or NULL */
    float *seq_adv;       /* [S] A_i as used, or NULL */
    int32_t *counts;      /* [4] mask=1 tokens popped (DIS: outside the interval), mask=1 tokens clipped, mask=0 tokens,
                             responses with no mask=1 token; or NULL */
    float *mean_entropy;  /* [1] mean entropy over mask=1 tokens, or NULL */
} rl_loss_outputs;

/* Kernel timing collected with CUDA events (see rl_loss_profile_start). */
#define RL_PROFILE_MAX_KERNELS 12
typedef struct rl_loss_profile {
    int32_t num_kernels;
    char names[RL_PROFILE_MAX_KERNELS][32];
    int64_t launches[RL_PROFILE_MAX_KERNELS];
    double total_ms[RL_PROFILE_MAX_KERNELS];
} rl_loss_profile;

/* Validates `config`, binds the handle to the current CUDA device and
 * allocates its workspace (O(max_tokens + max_seqs) bytes). On failure *out is
 * NULL and nothing stays allocated. */
RL_LOSS_API rl_status rl_loss_create(const rl_loss_config *config, rl_loss_t *out);

/* Frees the workspace and the handle (synchronises the device first). NULL is a no-op. */
RL_LOSS_API rl_status rl_loss_destroy(rl_loss_t handle);

/* The fused forward + backward pass of Eq. (1) over one batch. Enqueues six
 * kernels on `stream` (per-response prep, per-token prep, the fused row
 * kernel, the entropy of the rows that hold -inf logits, two fixed-order
 * reductions) and returns without synchronising. A -inf logit is a valid
 * input (probability 0, e.g. a masked vocabulary entry): it adds nothing to
 * the entropy (0 log 0 = 0) and gets a zero gradient; NaN and +inf logits are
 * non-finite (RL_ERR_NONFINITE). */
RL_LOSS_API rl_status rl_loss_forward_backward(rl_loss_t handle, const rl_loss_inputs *inputs,
                                               const rl_loss_outputs *outputs, void *stream);

/* The same pass for inputs that start in HOST memory, with the host-to-device
 * copy overlapped with the computation. `host` holds the batch in host memory
 * (page-locked, e.g. cudaHostAlloc, for the copies to run asynchronously and
 * overlap); `device` names device buffers of the same shapes that receive it
 * (device->ld_logits may differ from host->ld_logits; num_tokens / num_seqs
 * are taken from `host` and those of `device` are ignored). Both follow the
 * rules of rl_loss_inputs; outputs as for rl_loss_forward_backward.
 * The small per-token and per-response arrays are copied on `stream` first.
 * The logits go in `num_chunks` blocks of consecutive rows (1 <= num_chunks
 * <= 64, fewer if T is smaller) on a copy stream of the handle, which starts
 * after the work enqueued on `stream` before the call; the token preparation
 * and the row kernel of a block start on `stream` as soon as that block has
 * landed, so all but the last block's computation hides under the copy. The
 * two reductions follow on `stream`, which at the end depends on every copy.
 * Results are bit-identical to rl_loss_forward_backward on the copied inputs
 * (every row is computed the same way; the reductions run once over all rows).
 * The first call on a handle creates its copy stream and events (kept until
 * rl_loss_destroy); nothing is allocated on the device. Returns without
 * synchronising: the host buffers must stay unchanged until `stream` has
 * passed the call. Not for use inside a CUDA graph capture. Argument errors
 * (those of rl_loss_forward_backward for `device` and `outputs`, a NULL host
 * array, host->ld_logits < V: RL_ERR_SHAPE, num_chunks outside [1, 64]:
 * RL_ERR_INVALID_ARG) return before anything is enqueued; a copy or launch the
 * runtime refuses (e.g. a host pointer that is not host memory) returns
 * RL_ERR_CUDA, possibly after part of the work was enqueued. */
RL_LOSS_API rl_status rl_loss_forward_backward_from_host(rl_loss_t handle, const rl_loss_inputs *host,
                                                         const rl_loss_inputs *device, const rl_loss_outputs *outputs,
                                                         int32_t num_chunks, void *stream);

/* ---- Sequence-chunked output projection + loss ------------------------------
 * "GLM-5: from Vibe Coding to Agentic Engineering", section 2.4.1, "Sequence-
 * chunked output projection for peak memory reduction" (also "GLM-5 Notes",
 * infrastructure item 5): the hidden states are split into chunks of rows; per
 * chunk the output projection z = h W^T, the loss above and their backward run
 * to completion before the next chunk reuses the buffers, so the logits of the
 * whole sequence never exist at once. All three products run on the tensor
 * cores (tcgen05, pairs of CTAs on 256 x 512 tiles, bf16 inputs, fp32
 * accumulation in a fixed order): the projection fused with the per-row
 * softmax statistics, its output kept as bf16 scaled probabilities
 * 2^{z log2e - m} (m a per-row reference of each 64-column block; the target's
 * logit kept in fp32); dZ is formed once per chunk in bf16 over them, in
 * place; dH = dZ W and dW += dZ^T H share one launch per chunk, dW
 * accumulated in fp32 chunk after chunk in chunk order, so every output
 * repeats bit for bit. */

/* Allocates the fused projection path's buffers for hidden size `hidden_dim`
 * (a multiple of 8) and chunks of `chunk_tokens` rows: one chunk_tokens x V
 * bf16 buffer (the scaled probabilities, then dL/dlogits), the per-row
 * statistics and block references (32 bytes per row per 256 columns) and the
 * target logits. Requires a handle with logits_dtype RL_BF16 (else
 * RL_ERR_UNSUPPORTED). Calling it again
 * replaces the buffers. Synchronises the device. */
RL_LOSS_API rl_status rl_loss_projection_setup(rl_loss_t handle, int32_t hidden_dim, int32_t chunk_tokens);

/* logits[rows x V] (fp32, row stride ld_logits >= V, 16-byte aligned rows) =
 * hidden[rows x H] (bf16, row stride ld_hidden) * w_lm[V x H]^T (bf16, row
 * stride ld_w), the projection of the fused path on the tensor cores, for
 * callers that want a chunk's logits themselves. Needs rl_loss_projection_setup
 * (for H). Device pointers, 16-byte aligned, row strides a multiple of 16 bytes. */
RL_LOSS_API rl_status rl_loss_projection_logits(rl_loss_t handle, const void *hidden, int64_t ld_hidden,
                                                const void *w_lm, int64_t ld_w, int32_t rows, float *logits,
                                                int64_t ld_logits, void *stream);

/* The fused forward + backward over T = inputs->num_tokens rows of hidden
 * states: hidden [T x H] bf16 (row stride ld_hidden), w_lm [V x H] bf16
 * (row stride ld_w). Writes dhidden [T x H] bf16 (row stride ld_dhidden) =
 * dL/dhidden and dw_lm [V x H] fp32 (row stride ld_dw, overwritten) = dL/dW.
 * inputs->logits / ld_logits and outputs->dlogits / ld_dlogits are ignored;
 * every other field of inputs / outputs means what it means for
 * rl_loss_forward_backward. Needs rl_loss_projection_setup; allocates nothing.
 * Device pointers, 16-byte aligned, row strides a multiple of 16 bytes. */
RL_LOSS_API rl_status rl_loss_fused_projection_forward_backward(rl_loss_t handle, const void *hidden,
                                                                int64_t ld_hidden, const void *w_lm, int64_t ld_w,
                                                                const rl_loss_inputs *inputs, void *dhidden,
                                                                int64_t ld_dhidden, float *dw_lm, int64_t ld_dw,
                                                                const rl_loss_outputs *outputs, void *stream);

/* ---- Generalized advantage estimation (the step before a critic-based loss) --
 * "Zhipu AI / GLM: From Blank Infilling to Compaction-Aware Agentic
 * Reinforcement Learning", section 11: skip-observation GAE of the
 * single-rollout critic, and CompactionRL's cross-trajectory discount. Per
 * response, walking backwards over its action (mask=1) tokens t with next
 * action token t' of the same response:
 *   A_t = r_t + gamma V_{t'} - V_t + gamma lambda A_{t'}   (V_{t'} = A_{t'} = 0 after the last)
 * observation (mask=0) tokens are skipped and get A = 0 (with
 * skip_observations = 0 every token is an action token). With
 * cross_trajectory, consecutive responses sharing a rollout id are segments
 * of one rollout and segment s is scaled by (gamma lambda)^{N_{>s}}, N_{>s}
 * the mask=1 tokens of its later segments. Computed in fp32 in one pass over
 * the token arrays: 8192-token chunks, each folded into an affine map, a fixed
 * tree inside a chunk and a look-back over the chunks to the right in a fixed
 * order; bit-identical run to run. The result feeds RL_ADV_PER_TOKEN. */
typedef struct rl_gae_config {
    double gamma;              /* discount, 0 <= gamma <= 1 (not disclosed on the pages: an input); double so
                                  that (gamma lambda)^N over a long rollout keeps its accuracy */
    double lambda;             /* GAE lambda, 0 <= lambda <= 1 */
    int32_t skip_observations; /* 1: mask=0 tokens are skipped; 0: every token is an action token */
    int32_t cross_trajectory;  /* 1: apply (gamma lambda)^{N_{>s}} over segments (needs rollout_ids) */
} rl_gae_config;

/* Bytes of device workspace rl_gae_advantages needs for num_tokens tokens
 * (a 256-byte header and a 64-byte slot per 8192-token chunk). */
RL_LOSS_API size_t rl_gae_workspace_bytes(int32_t num_tokens);

/* Device pointers: rewards [T], values [T] fp32, mask [T] u8 (nonzero =
 * action token), cu_seqlens [S+1] i32 non-decreasing within [0, T] (tokens
 * outside [cu_seqlens[0], cu_seqlens[S]) are not written), rollout_ids [S] i32
 * (read when cross_trajectory, else may be NULL); writes advantages [T] fp32
 * and, if non-NULL, returns [T] = A + V on action tokens, 0 elsewhere.
 * rewards, values, advantages and returns must be 4-byte aligned; with every
 * array 16-byte aligned the kernel uses 16-byte accesses.
 * `workspace` (device, 256-byte aligned, at least rl_gae_workspace_bytes(T))
 * is owned by the caller and must be zero-filled before its first use; every
 * call that completes clears its counters and flags again, so the same
 * workspace serves the next call of any size; one workspace per stream.
 * `device_status` (optional, device uint32) receives RL_ERR_SEQLENS and
 * RL_ERR_TIMEOUT bits (after a timeout, zero the workspace again).
 * Host-side errors: RL_ERR_INVALID_ARG (NULL pointer, gamma or lambda outside
 * [0, 1]), RL_ERR_SHAPE (T < 0 or S < 1), RL_ERR_CAPACITY (workspace too
 * small), RL_ERR_ALIGNMENT. Needs no handle and allocates nothing; one
 * launch on `stream`. */
RL_LOSS_API rl_status rl_gae_advantages(const rl_gae_config *config, int32_t num_tokens, int32_t num_seqs,
                                        const float *rewards, const float *values, const uint8_t *mask,
                                        const int32_t *cu_seqlens, const int32_t *rollout_ids, float *advantages,
                                        float *returns, void *workspace, size_t workspace_bytes,
                                        uint32_t *device_status, void *stream);

/* Failure injection for tests of the failure detection above (the pages have
 * no counterpart): rl_gae_advantages with the map of chunk `withhold_chunk`
 * (8192-token chunks, counted from token 0) never published, and each wait
 * for a neighbouring chunk's map bounded by `wait_limit_s` seconds
 * (0 < wait_limit_s <= 1; rl_gae_advantages uses 1 s). The chunks whose
 * look-back needs the withheld map wait that long, raise RL_ERR_TIMEOUT in
 * `device_status` and treat the chunk as a response end, so their advantages
 * are wrong but the launch always completes and the GPU stays usable. No
 * fault, trap or unbounded wait is involved. RL_ERR_INVALID_ARG for
 * withhold_chunk < 0 or wait_limit_s outside (0, 1]; otherwise as
 * rl_gae_advantages. */
RL_LOSS_API rl_status rl_gae_advantages_withheld(const rl_gae_config *config, int32_t num_tokens, int32_t num_seqs,
                                                 const float *rewards, const float *values, const uint8_t *mask,
                                                 const int32_t *cu_seqlens, const int32_t *rollout_ids,
                                                 float *advantages, float *returns, void *workspace,
                                                 size_t workspace_bytes, uint32_t *device_status, void *stream,
                                                 int32_t withhold_chunk, double wait_limit_s);

/* ---- Deterministic top-k over DSA indexer scores ----------------------
 * "GLM-5: from Vibe Coding to Agentic Engineering", section 3.2 ("DSA RL
 * insights"): the DSA indexer keeps the k = 2048 best-scoring key positions of
 * every query, and the top-k used in RL must be deterministic (a
 * non-deterministic CUDA top-k collapsed RL; torch.topk was used instead).
 * Selection: the first k positions of a row under one total order: NaN above
 * every number, then larger score, then lower position; -0 and +0 tie. The
 * result (set and order) is unique and bit-identical from run to run. A CTA
 * per row streams it once from HBM through a shared-memory candidate buffer
 * behind a lower bound taken from a 4% sample of the row (a row where fewer
 * than k scores reach that bound is read a second time from the start). */
typedef enum rl_topk_order {
    RL_TOPK_BY_SCORE = 0,    /* (score desc, position asc): what a sorted torch.topk returns, ties fixed */
    RL_TOPK_BY_POSITION = 1  /* the same set by increasing position */
} rl_topk_order;

typedef struct rl_topk_config {
    int32_t k;      /* 1 <= k <= rl_topk_max_k() */
    int32_t order;  /* rl_topk_order */
} rl_topk_config;

/* Largest k the library supports (4096). */
RL_LOSS_API int32_t rl_topk_max_k(void);

/* Device pointers: scores [rows x ld] fp32, row-major, 16-byte aligned with
 * ld % 4 == 0; lengths [rows] i32 (row q's valid scores are its first
 * lengths[q], 0 <= lengths[q] <= ld; NULL: all ld); writes out_idx [rows x ldo]
 * i32 positions and, if non-NULL, out_val [rows x ldo] fp32 (the scores
 * themselves, bit for bit). When lengths[q] < k the missing entries are -1 and
 * -inf. `device_status` (optional, device uint32) receives RL_ERR_SEQLENS for
 * a length outside [0, ld] (clamped), RL_ERR_TIMEOUT if a tile copy did not
 * land within its bounded wait, and RL_ERR_INTERNAL if an internal consistency
 * check failed; after either of the last two that row's output is not valid.
 * Host-side errors: RL_ERR_INVALID_ARG
 * (NULL pointer, bad order), RL_ERR_SHAPE (rows < 0, ld < 1, ldo < k),
 * RL_ERR_UNSUPPORTED (k outside [1, rl_topk_max_k()]), RL_ERR_ALIGNMENT.
 * Needs no handle and allocates nothing; one launch on `stream`. */
RL_LOSS_API rl_status rl_topk(const rl_topk_config *config, int32_t rows, const float *scores, int64_t ld,
                              const int32_t *lengths, int32_t *out_idx, float *out_val, int64_t ldo,
                              uint32_t *device_status, void *stream);

/* Synchronises `stream`, returns the accumulated device status bits
 * (1u << code for each rl_status code raised) in *bits and clears them. */
RL_LOSS_API rl_status rl_loss_get_device_status(rl_loss_t handle, void *stream, uint32_t *bits);

/* Static, human-readable name of a status code. */
RL_LOSS_API const char *rl_loss_status_string(rl_status status);

/* Starts recording a CUDA event pair around every kernel of the next
 * `max_calls` forward_backward calls (timing only; results are unchanged). */
RL_LOSS_API rl_status rl_loss_profile_start(rl_loss_t handle, int32_t max_calls);

/* Synchronises the recorded events, writes per-kernel launch counts and
 * summed durations into *out and stops recording. */
RL_LOSS_API rl_status rl_loss_profile_read(rl_loss_t handle, rl_loss_profile *out);

/* Name of the CUDA error (e.g. "cudaErrorInvalidValue") behind the most recent
 * RL_ERR_CUDA returned for this handle, "cudaSuccess" if there was none.
 * Static string; never NULL. */
RL_LOSS_API const char *rl_loss_last_cuda_error(rl_loss_t handle);

/* Number of kernels this handle has launched since it was created. */
RL_LOSS_API rl_status rl_loss_launch_count(rl_loss_t handle, int64_t *count);

/* Allocation-free variant of rl_loss_forward_backward, for callers that cannot
 * call cudaMalloc when they need the loss: code inside a framework whose
 * caching allocator owns all device memory, or a serving process with a fixed
 * memory budget, where an allocation could fail or synchronise the device.
 * (The pages describe no such entry point; it has no counterpart there.)
 *
 * It needs no handle and allocates nothing: its workspace is one static
 * 16 MiB device array of this library, which every GPU that loads the library
 * holds until the process exits. `config` is read as for rl_loss_create except
 * that max_tokens / max_seqs are ignored: calls accept at most 262144 tokens
 * and 8192 responses and return RL_ERR_CAPACITY beyond that, before launching
 * anything. The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current. Every call on a device
 * shares the one array and leaves its contents behind (the status word is
 * cleared at the start of each call), so calls that overlap on the GPU (two
 * streams, two threads) race and must be serialised by the caller.
 * `device_status` (optional, a device pointer to one uint32) receives this
 * call's status bits as rl_loss_get_device_status would report them.
 * Everything else (arguments, layouts, outputs, errors) is as for
 * rl_loss_forward_backward. */
RL_LOSS_API rl_status rl_loss_forward_backward_noalloc(const rl_loss_config *config, const rl_loss_inputs *inputs,
                                                       const rl_loss_outputs *outputs, uint32_t *device_status,
                                                       void *stream);

/* Library version as major * 10000 + minor * 100 + patch. */
RL_LOSS_API int32_t rl_loss_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RL_LOSS_H */
