// Per-response preparation and the fixed-order reductions of the loss.
//
// seg_prep:     |y_i|, A_i and w_i = 1/(S |y_i|) per response ("GLM-5: from
//               Vibe Coding to Agentic Engineering", section 3.2: the
//               group-normalised advantage and the 1/G, 1/|y_i| factors of Eq. (1)).
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
constexpr int kReduceThreads = 256;

// One block per group of G consecutive responses.
__global__ void __launch_bounds__(kPrepThreads) seg_prep_kernel(SeqPrepParams p) {
    __shared__ int iscratch[32];
    const int G = p.group_size;
    const int g0 = blockIdx.x * G;
    const int T = p.num_tokens;
    for (int k = 0; k < G; ++k) {
        const int i = g0 + k;
        int b = __ldg(p.cu_seqlens + i), e = __ldg(p.cu_seqlens + i + 1);
        const bool bad = (b < 0) || (e < b) || (e > T) || (i == 0 && b != 0) ||
                         (i == p.num_seqs - 1 && e != T);
        if (bad) {
            if (threadIdx.x == 0) raise_status(p.status, RL_ERR_SEQLENS);
            b = min(max(b, 0), T);
            e = min(max(e, b), T);
        }
        int n = 0;
        for (int t = b + threadIdx.x; t < e; t += blockDim.x) n += __ldg(p.mask + t) ? 1 : 0;
        n = block_sum_i32(n, iscratch);
        if (threadIdx.x == 0) {
            p.seq_n[i] = n;
            const double w = n > 0 ? 1.0 / ((double)p.num_seqs * (double)n) : 0.0;
            p.seq_w64[i] = w;
            p.seq_w[i] = (float)w;
            if (n == 0) raise_status(p.status, RL_ERR_EMPTY_SEQ);
        }
    }
    if (threadIdx.x != 0) return;
    // advantages in double, fixed order over the group, rounded once to fp32
    if (p.adv_mode == RL_ADV_PER_SEQ) {
        for (int k = 0; k < G; ++k) {
            const float a = p.rewards_or_adv[g0 + k];
            p.seq_adv[g0 + k] = a;
            if (p.seq_adv_out) p.seq_adv_out[g0 + k] = a;
        }
        return;
    }
    double mean = 0.0;
    for (int k = 0; k < G; ++k) mean += (double)p.rewards_or_adv[g0 + k];
    mean /= (double)G;
    double ss = 0.0;
    for (int k = 0; k < G; ++k) {
        const double c = (double)p.rewards_or_adv[g0 + k] - mean;
        ss += c * c;
    }
    const double sd = sqrt(ss / (double)(p.std_unbiased ? G - 1 : G));
    for (int k = 0; k < G; ++k) {
        const float a = (float)(((double)p.rewards_or_adv[g0 + k] - mean) / (sd + (double)p.adv_eps));
        p.seq_adv[g0 + k] = a;
        if (p.seq_adv_out) p.seq_adv_out[g0 + k] = a;
    }
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
    for (int t = b + threadIdx.x; t < e; t += blockDim.x) {
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
    seg_prep_kernel<<<p.num_seqs / p.group_size, kPrepThreads, 0, stream>>>(p);
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
