/*
 * Oracle for the token-level GRPO + IcePop policy loss and its gradient.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file: only the tests, the package's smoke check and the benchmark's
 * CPU-baseline leg do. It shares no header, helper or constant with the CUDA
 * library. Plain, slow, obviously correct: every quantity is computed in
 * double precision straight from its definition.
 *
 * Sources (web pages, cited by title and section):
 *  - "GLM-5: from Vibe Coding to Agentic Engineering", section 3.2 "Reasoning
 *    RL", Eq. (1): the loss, the mismatch ratio rho, the pop operator, the PPO
 *    ratio r and the group-normalised advantage A; hyper-parameters beta = 2,
 *    eps_low = 0.2, eps_high = 0.28; the KL term of the original IcePop is
 *    removed.
 *  - "Zhipu AI / GLM: From Blank Infilling to Compaction-Aware Agentic
 *    Reinforcement Learning", section 9.4 (loss masks: tool results and
 *    incorrect action segments get loss mask 0) and section 9.5 (GRPO +
 *    IcePop, no KL, beta = 2, clip 0.2 / 0.28).
 *  - "2.5 GLM-5 -- 异步 Agentic RL 工程", section "Cross-Stage Distillation":
 *    group size 1 with a per-sequence advantage teacher_score - student_score
 *    (served here by adv_mode 1, a given per-sequence advantage).
 *
 * Readings taken where the pages are silent (each one is also listed in the
 * design notes of the repository):
 *  - E_x over a batch of P prompts is the mean over prompts, so every response
 *    carries weight 1/(P*G) = 1/S in total, split as 1/|y_i| over its tokens.
 *  - |y_i| is the number of mask=1 tokens of response i; a response with none
 *    contributes 0.
 *  - std() is the population standard deviation (ddof 0) unless std_unbiased,
 *    and the denominator carries a small adv_eps: (R - mean) / (std + adv_eps).
 *  - pop() returns rho inside [1/beta, beta] (the printed operator) or 1 when
 *    pop_indicator is set; 0 outside.
 *  - The in-bounds test of pop and the clip test are decided in IEEE fp32, the
 *    precision of the log-prob inputs: d = fl32(logp_old - logp_infer) is in
 *    bounds iff -B <= d <= B with B = fl32(ln beta); the clip branch is active
 *    (zero gradient) iff A > 0 and fl32(fl32(logp) - logp_old) > fl32(ln(1 +
 *    eps_high)), or A < 0 and that difference < fl32(ln(1 - eps_low)). On the
 *    boundary itself both branches of min() are equal and the unclipped
 *    derivative is taken.
 *  - Entropy is the full-vocabulary Shannon entropy of softmax(z) in nats.
 *    It is an output only and carries no gradient.
 *  - Logits are used as given (temperature 1).
 *  - A target id outside [0, V) excludes its token from the loss (objective
 *    and gradient 0), sets flag bit 3 and leaves logp as NaN.
 *
 * Two further objectives / advantages of the same pages (adv_mode, objective):
 *  - Per-token advantages (adv_mode 2, e.g. from a critic) and the on-policy
 *    distillation advantage A_t = sg[log pi_teacher(y_t) - log pi_theta(y_t)]
 *    (adv_mode 3, "GLM-5: from Vibe Coding to Agentic Engineering", section 3.5,
 *    Eq. (2)), which replaces A in Eq. (1). Its sign, which decides the clip
 *    side, is taken in fp32: fl32(logp_teacher - fl32(logp)).
 *  - Direct double-sided importance sampling (objective 1, section 4.1.2,
 *    Eqs. (3)-(5); "Zhipu AI / GLM: From Blank Infilling to Compaction-Aware
 *    Agentic Reinforcement Learning", section 11, "Direct Double-Sided
 *    Importance Sampling"): r = exp(logp - logp_rollout) with the rollout
 *    engine's log-prob (logp_infer), f(r) = r on the open interval
 *    (1 - eps_low, 1 + eps_high) and 0 outside (decided in fp32 on
 *    fl32(fl32(logp) - logp_rollout) against the clip thresholds), token term
 *    f(r) A logp. Readings: the loss is minus the printed objective (as for
 *    Eq. (1)); "E_t" is the mean over the generated tokens when loss_norm = 1;
 *    whether f is stop-gradient is unmarked on the pages, so both readings
 *    exist: dis_stopgrad = 1 differentiates A logp only (dL/dlogp = -w f A),
 *    0 differentiates f too (dL/dlogp = -w r A (1 + logp) inside the interval).
 *    Flag bit0 is then "inside the interval" and bit1 is unused.
 *
 * Flag bits per token: bit0 pop in bounds, bit1 clip branch active, bit2 mask
 * is 0, bit3 target id out of range.
 *
 * The functions are parallel over rows with OpenMP; every row is computed on
 * its own, in one thread, in index order, so results do not depend on the
 * thread count.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F64 2 /* oracle-only: lets finite-difference checks perturb logits finely */

/* One logit as a double. bf16 is the upper half of an IEEE binary32 word, so
 * widening it is exact; fp32 -> double is exact as well. */
static double logit_at(const void *row, int32_t dtype, int64_t v) {
    if (dtype == ORACLE_F32) return (double)((const float *)row)[v];
    if (dtype == ORACLE_F64) return ((const double *)row)[v];
    uint32_t bits = (uint32_t)((const uint16_t *)row)[v] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static int64_t elem_size(int32_t dtype) {
    return dtype == ORACLE_F32 ? 4 : (dtype == ORACLE_F64 ? 8 : 2);
}

/* Index i of the response whose token range [cu[i], cu[i+1]) holds token t,
 * or -1. Plain linear scan. */
static int64_t seq_of_token(int64_t S, const int32_t *cu, int64_t t) {
    for (int64_t i = 0; i < S; ++i)
        if (t >= cu[i] && t < cu[i + 1]) return i;
    return -1;
}

/* fp32 threshold constants of the pop and clip decisions (see header). */
float oracle_ln_beta_f32(float beta) { return (float)log((double)beta); }
float oracle_clip_hi_f32(float eps_high) { return (float)log1p((double)eps_high); }
float oracle_clip_lo_f32(float eps_low) { return (float)log1p(-(double)eps_low); }

/* pop in-bounds decision: 1/beta <= rho <= beta, rho = pi_old^train / pi^infer,
 * i.e. -ln beta <= logp_old - logp_infer <= ln beta, taken in fp32. */
int32_t oracle_pop_in_bounds(float logp_old, float logp_infer, float beta) {
    volatile float d = logp_old - logp_infer; /* one IEEE fp32 subtraction */
    float b = oracle_ln_beta_f32(beta);
    return (-b <= d && d <= b) ? 1 : 0;
}

/* Clip branch active (the zero-gradient side of min(r A, clip(r) A)), taken
 * in fp32 from a given fp32 log-prob. A > 0: r > 1 + eps_high. A < 0:
 * r < 1 - eps_low. A == 0: never. */
int32_t oracle_clip_active(float logp, float logp_old, double adv, float eps_low, float eps_high) {
    volatile float e = logp - logp_old; /* one IEEE fp32 subtraction: ln r */
    if (adv > 0.0) return e > oracle_clip_hi_f32(eps_high) ? 1 : 0;
    if (adv < 0.0) return e < oracle_clip_lo_f32(eps_low) ? 1 : 0;
    return 0;
}

/* Vector form of oracle_clip_active, for checking another side's flags
 * against the definition from that side's own fp32 log-probs. */
void oracle_clip_active_vec(int64_t n, const float *logp, const float *logp_old, const double *adv_per_token,
                            float eps_low, float eps_high, uint8_t *out) {
    for (int64_t k = 0; k < n; ++k)
        out[k] = (uint8_t)oracle_clip_active(logp[k], logp_old[k], adv_per_token[k], eps_low, eps_high);
}

/*
 * Sequence-level quantities ("GLM-5: from Vibe Coding to Agentic Engineering",
 * section 3.2, definitions under Eq. (1)).
 *   n_i   = |y_i| = number of mask=1 tokens of response i
 *   A_i   = (R_i - mean(R_group)) / (std(R_group) + adv_eps)   (adv_mode 0)
 *         = rewards_or_adv[i]                                 (adv_mode 1)
 *   w_i   = 1 / (S * n_i), or 0 when n_i == 0          (loss_norm 0, Eq. (1))
 *         = 1 / sum_j n_j, or 0 when n_i == 0         (loss_norm 1, mean over tokens)
 * Groups are G consecutive responses. Returns 0, or -1 on bad arguments.
 */
int32_t oracle_seq_prep(int64_t S, int64_t G, const int32_t *cu_seqlens, const uint8_t *mask,
                        const float *rewards_or_adv, int32_t adv_mode, float adv_eps, int32_t std_unbiased,
                        int32_t loss_norm, int64_t *n_tokens, double *adv, double *w) {
    if (S < 1 || G < 1 || S % G != 0) return -1;
    if (adv_mode < 0 || adv_mode > 3) return -1;
    if (adv_mode == 0 && std_unbiased && G < 2) return -1;
    int64_t total = 0;
    for (int64_t i = 0; i < S; ++i) {
        if (cu_seqlens[i + 1] < cu_seqlens[i]) return -1;
        int64_t n = 0;
        for (int64_t t = cu_seqlens[i]; t < cu_seqlens[i + 1]; ++t) n += mask[t] ? 1 : 0;
        n_tokens[i] = n;
        total += n;
        w[i] = n > 0 ? 1.0 / ((double)S * (double)n) : 0.0;
    }
    if (loss_norm == 1) /* the mean over every generated token of the batch */
        for (int64_t i = 0; i < S; ++i) w[i] = n_tokens[i] > 0 ? 1.0 / (double)total : 0.0;
    if (adv_mode >= 2) { /* per-token advantages: no per-response value */
        for (int64_t i = 0; i < S; ++i) adv[i] = 0.0;
        return 0;
    }
    if (adv_mode == 1) {
        for (int64_t i = 0; i < S; ++i) adv[i] = (double)rewards_or_adv[i];
        return 0;
    }
    for (int64_t g0 = 0; g0 < S; g0 += G) {
        double mean = 0.0;
        for (int64_t k = 0; k < G; ++k) mean += (double)rewards_or_adv[g0 + k];
        mean /= (double)G;
        double ss = 0.0;
        for (int64_t k = 0; k < G; ++k) {
            double c = (double)rewards_or_adv[g0 + k] - mean;
            ss += c * c;
        }
        double std = sqrt(ss / (double)(std_unbiased ? G - 1 : G));
        for (int64_t k = 0; k < G; ++k)
            adv[g0 + k] = ((double)rewards_or_adv[g0 + k] - mean) / (std + (double)adv_eps);
    }
    return 0;
}

/*
 * Per-token forward and backward for a list of rows.
 *
 * logits holds n_rows rows of ld elements each, row k being token row_ids[k];
 * targets / logp_old / logp_infer / mask are indexed by token id. adv and w
 * come from oracle_seq_prep. Per row k this writes:
 *   logp[k]    = z_y - log sum_v exp(z_v)                  (log-softmax gather)
 *   entropy[k] = -sum_v p_v log p_v
 *   flags[k]   = bit0 pop in bounds | bit1 clip active | bit2 masked | bit3 bad target
 *   tok_obj[k] = m_t * pop(rho_t) * min(r_t A_i, clip(r_t, 1-eps_low, 1+eps_high) A_i)
 *   g[k]       = dL/dlogp_t = -w_i * m_t * pop(rho_t) * A_i * r_t  on the unclipped branch, else 0
 *   dz[k, v]   = dL/dz_v    = g[k] * (1[v == y_t] - p_v)          (if dz != NULL; [n_rows, V])
 * where rho_t = exp(logp_old - logp_infer), r_t = exp(logp_t - logp_old) and
 * L = -sum_i w_i sum_{t in i} tok_obj_t ("GLM-5: from Vibe Coding to Agentic
 * Engineering", section 3.2, Eq. (1)). Returns 0, or -1 on bad arguments.
 */
int32_t oracle_rows(int64_t n_rows, const int64_t *row_ids, int64_t V, int64_t ld, int32_t dtype, const void *logits,
                    const int32_t *targets, const float *logp_old, const float *logp_infer, const uint8_t *mask,
                    int64_t S, const int32_t *cu_seqlens, const double *adv, const double *w, float eps_low,
                    float eps_high, float beta, int32_t pop_indicator, int32_t objective, int32_t dis_stopgrad,
                    const float *adv_token, const float *teacher_logp, double *logp, double *entropy,
                    uint8_t *flags, double *tok_obj, double *g, double *dz) {
    if (V < 1 || ld < V || n_rows < 0) return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F64) return -1;
    const double lo_clip = 1.0 - (double)eps_low, hi_clip = 1.0 + (double)eps_high;
    int32_t bad = 0;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t k = 0; k < n_rows; ++k) {
        const int64_t t = row_ids[k];
        const void *row = (const char *)logits + (size_t)(k * ld * elem_size(dtype));
        const int64_t i = seq_of_token(S, cu_seqlens, t);
        if (i < 0) {
#pragma omp atomic write
            bad = 1;
            continue;
        }
        /* log-softmax: logZ = log sum_v exp(z_v), shifted by the max for range */
        double zmax = -INFINITY;
        for (int64_t v = 0; v < V; ++v) {
            double z = logit_at(row, dtype, v);
            if (z > zmax) zmax = z;
        }
        double sum = 0.0;
        for (int64_t v = 0; v < V; ++v) sum += exp(logit_at(row, dtype, v) - zmax);
        const double logZ = zmax + log(sum);
        double H = 0.0;
        for (int64_t v = 0; v < V; ++v) {
            double lp = logit_at(row, dtype, v) - logZ;
            const double pv = exp(lp);
            if (pv > 0.0) H -= pv * lp; /* p log p -> 0 as p -> 0: a -inf logit adds nothing */
        }
        entropy[k] = H;

        const int32_t y = targets[t];
        const int target_ok = (y >= 0 && (int64_t)y < V);
        const double lp_y = target_ok ? logit_at(row, dtype, y) - logZ : NAN;
        logp[k] = lp_y;

        /* the advantage of this token, and the sign that decides the clip side */
        double A = adv[i], A_sign = adv[i];
        if (adv_token) A = A_sign = (double)adv_token[t];
        if (teacher_logp) {
            A = target_ok ? (double)teacher_logp[t] - lp_y : 0.0;
            volatile float a32 = teacher_logp[t] - (float)lp_y; /* fp32, as the kernel decides it */
            A_sign = target_ok ? (double)a32 : 0.0;
        }
        const int m = mask[t] ? 1 : 0;

        double obj = 0.0, gt = 0.0;
        if (objective == 1) {
            /* direct double-sided importance sampling against the rollout log-prob */
            volatile float e = (float)lp_y - logp_infer[t];
            const int gate = target_ok && e > oracle_clip_lo_f32(eps_low) && e < oracle_clip_hi_f32(eps_high);
            flags[k] = (uint8_t)(gate | ((!m) << 2) | ((!target_ok) << 3));
            if (target_ok && m && gate) {
                const double r = exp(lp_y - (double)logp_infer[t]);
                obj = r * A * lp_y; /* f(r) A log pi, f(r) = r inside the interval */
                gt = dis_stopgrad ? -w[i] * r * A : -w[i] * r * A * (1.0 + lp_y);
            }
        } else {
        const int in_bounds = oracle_pop_in_bounds(logp_old[t], logp_infer[t], beta);
        const int clip = target_ok ? oracle_clip_active((float)lp_y, logp_old[t], A_sign, eps_low, eps_high) : 0;
        flags[k] = (uint8_t)(in_bounds | (clip << 1) | ((!m) << 2) | ((!target_ok) << 3));
        if (target_ok && m) {
            const double rho = exp((double)logp_old[t] - (double)logp_infer[t]);
            const double pop = in_bounds ? (pop_indicator ? 1.0 : rho) : 0.0;
            const double r = exp(lp_y - (double)logp_old[t]);
            const double r_clipped = fmin(fmax(r, lo_clip), hi_clip);
            obj = pop * fmin(r * A, r_clipped * A);
            /* d/dlogp of min(r A, clip(r) A): r A on the unclipped branch, 0 on the clipped one */
            gt = clip ? 0.0 : -w[i] * pop * A * r;
        }
        }
        tok_obj[k] = obj;
        g[k] = gt;
        if (dz) {
            double *out = dz + (size_t)(k * V);
            for (int64_t v = 0; v < V; ++v) {
                double p = exp(logit_at(row, dtype, v) - logZ);
                out[v] = gt * (((target_ok && v == y) ? 1.0 : 0.0) - p);
            }
        }
    }
    return bad ? -1 : 0;
}

/* L = -sum_i w_i sum_{t in response i} tok_obj_t ("GLM-5: from Vibe Coding to
 * Agentic Engineering", section 3.2, Eq. (1)); tok_obj indexed by token id. */
double oracle_loss(int64_t S, const int32_t *cu_seqlens, const double *w, const double *tok_obj) {
    double L = 0.0;
    for (int64_t i = 0; i < S; ++i) {
        double s = 0.0;
        for (int64_t t = cu_seqlens[i]; t < cu_seqlens[i + 1]; ++t) s += tok_obj[t];
        L -= w[i] * s;
    }
    return L;
}

/*
 * Generalized advantage estimation over packed responses, with observation
 * tokens skipped ("Zhipu AI / GLM: From Blank Infilling to Compaction-Aware
 * Agentic Reinforcement Learning", section 11, "Restoring a critic at group
 * size one": skip-observation GAE, and "Token loss and cross-trajectory GAE").
 *
 * Within response i the action tokens are the mask=1 tokens; observation
 * (mask=0) tokens are skipped: the recursion links an action token directly to
 * the next action token of the same response. Walking backwards over the
 * action tokens t with next action token t' (none after the last one):
 *   delta_t = r_t + gamma * V_{t'} - V_t           (V_{t'} = 0 after the last action token)
 *   A_t     = delta_t + gamma * lambda * A_{t'}    (A_{t'} = 0 after the last action token)
 * Observation tokens get A = 0. With skip_observations = 0 every token is an
 * action token (plain token-level GAE).
 *
 * Cross-trajectory discount (rollout_ids != NULL): consecutive responses with
 * the same rollout id are the segments of one rollout; segment s's advantages
 * are multiplied by (gamma * lambda)^{N_{>s}}, N_{>s} being the number of
 * trainable (mask=1) tokens in the later segments of the same rollout.
 * Readings: gamma and lambda are inputs (the pages leave them undisclosed);
 * rewards are per token (zero except where the environment pays out).
 * Everything in double. Returns 0, or -1 on bad arguments.
 */
int32_t oracle_gae(int64_t S, const int32_t *cu_seqlens, const float *rewards, const float *values,
                   const uint8_t *mask, double gamma, double lambda, int32_t skip_observations,
                   const int32_t *rollout_ids, double *adv) {
    if (S < 0) return -1;
    for (int64_t i = 0; i < S; ++i) {
        if (cu_seqlens[i + 1] < cu_seqlens[i]) return -1;
        double A_next = 0.0, V_next = 0.0;
        for (int64_t t = cu_seqlens[i + 1] - 1; t >= cu_seqlens[i]; --t) {
            const int action = skip_observations ? (mask[t] != 0) : 1;
            if (!action) {
                adv[t] = 0.0;
                continue;
            }
            const double delta = (double)rewards[t] + gamma * V_next - (double)values[t];
            const double A = delta + gamma * lambda * A_next;
            adv[t] = A;
            A_next = A;
            V_next = (double)values[t];
        }
    }
    if (rollout_ids) {
        for (int64_t s = 0; s < S; ++s) {
            int64_t later = 0;
            for (int64_t u = s + 1; u < S && rollout_ids[u] == rollout_ids[s]; ++u)
                for (int64_t t = cu_seqlens[u]; t < cu_seqlens[u + 1]; ++t) later += mask[t] ? 1 : 0;
            const double f = pow(gamma * lambda, (double)later);
            for (int64_t t = cu_seqlens[s]; t < cu_seqlens[s + 1]; ++t) adv[t] *= f;
        }
    }
    return 0;
}
