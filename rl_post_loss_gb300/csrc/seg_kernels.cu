// Per-response preparation, per-token records and the fixed-order reductions.
//
// seg_prep:     |y_i|, A_i and w_i = 1/(S |y_i|) per response ("GLM-5: from
//               Vibe Coding to Agentic Engineering", section 3.2: the
//               group-normalised advantage and the 1/G, 1/|y_i| factors of Eq. (1)).
// token_prep:   the row-independent part of each token's objective (rho, pop,
//               mask, the advantage sign, z_y) packed for the row kernel.
// seg_reduce:   per-response sums of the token objectives, in token order.
// final_reduce: L = -sum_i w_i * (sum over response i), in response order.
//
// All floating-point sums use a tree whose shape depends only on the sizes,
// never on timing or on how many SMs are free, so results are bit-identical
// from run to run. No float atomics.
#include "common.cuh"

namespace rlk {

namespace {

constexpr int kPrepThreads = 256;
constexpr int kTokenThreads = 256;
constexpr int kReduceThreads = 256;

// One block per response.
__global__ void __launch_bounds__(kPrepThreads) seg_prep_kernel(SeqPrepParams p) {
    __shared__ int iscratch[32];
    const int i = blockIdx.x;
    const int T = p.num_tokens;
    int b = __ldg(p.cu_seqlens + i), e = __ldg(p.cu_seqlens + i + 1);
    const bool bad = (b < 0) || (e < b) || (e > T) || (i == 0 && b != 0) || (i == p.num_seqs - 1 && e != T);
    if (bad) {
        if (threadIdx.x == 0) raise_status(p.status, RL_ERR_SEQLENS);
        b = min(max(b, 0), T);
        e = min(max(e, b), T);
    }
    int n = 0;
#pragma unroll 4
    for (int t = b + threadIdx.x; t < e; t += kPrepThreads) n += __ldg(p.mask + t) ? 1 : 0;
    n = block_sum_i32(n, iscratch);
    if (threadIdx.x != 0) return;
    p.seq_n[i] = n;
    const double w = n > 0 ? 1.0 / ((double)p.num_seqs * (double)n) : 0.0;
    p.seq_w64[i] = w;
    p.seq_w[i] = (float)w;
    if (n == 0) raise_status(p.status, RL_ERR_EMPTY_SEQ);
    float a;
    if (p.adv_mode == RL_ADV_PER_TOKEN || p.adv_mode == RL_ADV_TEACHER_LOGP) {
        a = 0.f;  // per-token advantages: nothing per response
    } else if (p.adv_mode == RL_ADV_PER_SEQ) {
        a = p.rewards_or_adv[i];
    } else {
        // group statistics in double, fixed order over the group's G rewards;
        // every response of the group computes the same values
        const int G = p.group_size;
        const int g0 = (i / G) * G;
        double mean = 0.0;
        for (int k = 0; k < G; ++k) mean += (double)p.rewards_or_adv[g0 + k];
        mean /= (double)G;
        double ss = 0.0;
        for (int k = 0; k < G; ++k) {
            const double c = (double)p.rewards_or_adv[g0 + k] - mean;
            ss += c * c;
        }
        const double sd = sqrt(ss / (double)(p.std_unbiased ? G - 1 : G));
        a = (float)(((double)p.rewards_or_adv[i] - mean) / (sd + (double)p.adv_eps));
    }
    p.seq_adv[i] = a;
    if (p.seq_adv_out) p.seq_adv_out[i] = a;
}

// One block: the number of generated tokens of the batch (fixed-order sum of
// |y_i|) and w_i = 1 / that number for the mean over tokens.
__global__ void __launch_bounds__(kReduceThreads) seg_token_norm_kernel(SeqPrepParams p) {
    __shared__ int iscratch[32];
    int n = 0;
    for (int i = threadIdx.x; i < p.num_seqs; i += blockDim.x) n += p.seq_n[i];
    n = block_sum_i32(n, iscratch);
    const double w = n > 0 ? 1.0 / (double)n : 0.0;
    for (int i = threadIdx.x; i < p.num_seqs; i += blockDim.x) {
        const double wi = p.seq_n[i] > 0 ? w : 0.0;
        p.seq_w64[i] = wi;
        p.seq_w[i] = (float)wi;
    }
}

// One thread per token.
__global__ void __launch_bounds__(kTokenThreads) token_prep_kernel(TokenPrepParams p) {
    const int i_row = blockIdx.x * kTokenThreads + threadIdx.x;
    if (i_row >= p.rows) return;
    const int t = p.row0 + i_row;
    if (!RLK_CHECK(p.status, t < p.num_tokens)) return;
    const int i = find_seq(p.cu_seqlens, p.num_seqs, t);
    if (i < 0) raise_status(p.status, RL_ERR_SEQLENS);
    if (!RLK_CHECK(p.status, i < 0 || (i < p.num_seqs && __ldg(p.cu_seqlens + i) <= t &&
                                        t < __ldg(p.cu_seqlens + i + 1))))
        return;
    const float A = p.token_adv ? __ldg(p.token_adv + t) : (i >= 0 ? p.seq_adv[i] : 0.f);
    const float w = i >= 0 ? p.seq_w[i] : 0.f;
    const int y = __ldg(p.targets + t);
    const bool ok = (y >= 0) && (y < p.vocab);
    if (!ok) raise_status(p.status, RL_ERR_TARGET_RANGE);
    const bool m = (i >= 0) && (__ldg(p.mask + t) != 0);
    const float lo = __ldg(p.logp_old + t);
    const float d = __fsub_rn(lo, __ldg(p.logp_infer + t));  // ln rho, one fp32 subtraction
    const bool in_bounds = (-p.c.ln_beta <= d) && (d <= p.c.ln_beta);
    float zy = 0.f;
    if (ok && p.target_logit) {
        zy = __ldg(p.target_logit + i_row);
    } else if (ok) {
        const size_t off = (size_t)i_row * (size_t)p.ld_logits + (size_t)y;
        if (p.logits_dtype == RL_F32) {
            zy = __ldg(reinterpret_cast<const float *>(p.logits) + off);
        } else {
            const unsigned short b = __ldg(reinterpret_cast<const unsigned short *>(p.logits) + off);
            zy = __uint_as_float(static_cast<uint32_t>(b) << 16);
        }
    }
    uint32_t pre = (m ? 0u : RL_FLAG_MASKED) | (ok ? 0u : RL_FLAG_BAD_TARGET) | (A > 0.f ? kPreAPos : 0u) |
                   (A < 0.f ? kPreANeg : 0u);
    float cf = 0.f, lref = lo;
    if (p.c.objective == RL_OBJ_DIS) {
        // the gate needs logp: the token carries m * A and the rollout log-prob
        lref = __ldg(p.logp_infer + t);
        if (m && ok) cf = A;
    } else {
        pre |= in_bounds ? RL_FLAG_POP_IN_BOUNDS : 0u;
        const float pop = (m && ok && in_bounds) ? (p.c.pop_indicator ? 1.f : expf(d)) : 0.f;
        cf = p.c.adv_teacher ? pop : pop * A;  // the distillation advantage is applied once logp is known
    }
    p.rec[t] = make_float4(zy, lref, cf, w * cf);
    p.meta[t] = (ok ? (uint32_t)y : 0u) | (pre << 24);
}

// One block per response: sums over its tokens in token order (strided per
// thread, then a fixed tree).
__global__ void __launch_bounds__(kReduceThreads) seg_reduce_kernel(ReduceParams p) {
    __shared__ double dscratch[32];
    __shared__ int iscratch[32];
    const int i = blockIdx.x;
    const int T = p.num_tokens;
    int b = __ldg(p.cu_seqlens + i), e = __ldg(p.cu_seqlens + i + 1);
    b = min(max(b, 0), T);
    e = min(max(e, b), T);
    double obj = 0.0, ent = 0.0;
    int popped = 0, clipped = 0, masked = 0;
#pragma unroll 4
    for (int t = b + threadIdx.x; t < e; t += kReduceThreads) {
        const uint32_t f = p.flags[t];
        obj += (double)p.tok_obj[t];
        const bool m = !(f & RL_FLAG_MASKED);
        if (m) ent += (double)p.entropy[t];
        popped += (m && !(f & RL_FLAG_POP_IN_BOUNDS)) ? 1 : 0;
        clipped += (m && (f & RL_FLAG_CLIP_ACTIVE)) ? 1 : 0;
        masked += m ? 0 : 1;
    }
    obj = block_sum_f64(obj, dscratch);
    ent = block_sum_f64(ent, dscratch);
    popped = block_sum_i32(popped, iscratch);
    clipped = block_sum_i32(clipped, iscratch);
    masked = block_sum_i32(masked, iscratch);
    if (threadIdx.x == 0) {
        p.seq_obj[i] = obj;
        p.seq_ent[i] = ent;
        p.seq_cnt[4 * i + 0] = popped;
        p.seq_cnt[4 * i + 1] = clipped;
        p.seq_cnt[4 * i + 2] = masked;
        p.seq_cnt[4 * i + 3] = p.seq_n[i] == 0 ? 1 : 0;
    }
}

// One block: L = -sum_i w_i * seq_obj_i, in response order.
__global__ void __launch_bounds__(kReduceThreads) final_reduce_kernel(ReduceParams p) {
    __shared__ double dscratch[32];
    __shared__ int iscratch[32];
    double L = 0.0, ent = 0.0;
    int n = 0, c0 = 0, c1 = 0, c2 = 0, c3 = 0;
    for (int i = threadIdx.x; i < p.num_seqs; i += blockDim.x) {
        L += p.seq_w64[i] * p.seq_obj[i];
        ent += p.seq_ent[i];
        n += p.seq_n[i];
        c0 += p.seq_cnt[4 * i + 0];
        c1 += p.seq_cnt[4 * i + 1];
        c2 += p.seq_cnt[4 * i + 2];
        c3 += p.seq_cnt[4 * i + 3];
    }
    L = -block_sum_f64(L, dscratch);
    ent = block_sum_f64(ent, dscratch);
    n = block_sum_i32(n, iscratch);
    c0 = block_sum_i32(c0, iscratch);
    c1 = block_sum_i32(c1, iscratch);
    c2 = block_sum_i32(c2, iscratch);
    c3 = block_sum_i32(c3, iscratch);
    if (threadIdx.x == 0) {
        p.loss[0] = (float)L;
        if (p.loss_f64) p.loss_f64[0] = L;
        if (p.counts) {
            p.counts[0] = c0;
            p.counts[1] = c1;
            p.counts[2] = c2;
            p.counts[3] = c3;
        }
        if (p.mean_entropy) p.mean_entropy[0] = n > 0 ? (float)(ent / (double)n) : 0.f;
        if (!isfinite(L)) raise_status(p.status, RL_ERR_NONFINITE);
    }
}

}  // namespace

cudaError_t launch_seg_prep(const SeqPrepParams &p, cudaStream_t stream) {
    seg_prep_kernel<<<p.num_seqs, kPrepThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_seg_token_norm(const SeqPrepParams &p, cudaStream_t stream) {
    seg_token_norm_kernel<<<1, kReduceThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_token_prep(const TokenPrepParams &p, cudaStream_t stream) {
    if (p.rows <= 0) return cudaSuccess;
    token_prep_kernel<<<(p.rows + kTokenThreads - 1) / kTokenThreads, kTokenThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_seg_reduce(const ReduceParams &p, cudaStream_t stream) {
    seg_reduce_kernel<<<p.num_seqs, kReduceThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_final_reduce(const ReduceParams &p, cudaStream_t stream) {
    final_reduce_kernel<<<1, kReduceThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace rlk
