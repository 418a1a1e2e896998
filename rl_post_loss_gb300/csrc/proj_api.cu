// C ABI of the fused sequence-chunked output projection + loss ("GLM-5: from
// Vibe Coding to Agentic Engineering", section 2.4.1, "Sequence-chunked output
// projection for peak memory reduction"; "GLM-5 Notes", infrastructure item 5):
// the hidden states are split into chunks of rows; per chunk the projection,
// the loss of Eq. (1) (section 3.2) and its backward are computed and the
// chunk's buffers reused, so logits for the whole sequence never exist.
//
// Per chunk c of rows [r0, r0 + m):
//   proj_gemm   Z_c = H_c W^T (tcgen05, fp32 accumulators), stored as bf16 scaled
//               probabilities 2^{z log2e - m} (m a per-row, per-64-column reference),
//               with per-row, per-256-column softmax statistics and the exact
//               target logits
//   token_prep  per-token records (z_y from the target logits)
//   proj_rows   statistics merged per row in tile order, token objective, dZ_c (bf16,
//               over the scaled probabilities, in place)
//   proj_bwd    one tcgen05 launch over both backward products:
//               dH_c = dZ_c W (bf16 out) and
//               dW  (+)= dZ_c^T H_c (fp32; stored by chunk 0, added into by the later chunks)
// then the fixed-order per-response and batch reductions give the loss.
#include <cmath>

#include "handle.cuh"
#include "proj.cuh"

void rl_loss_handle_s::proj_release() {
    if (proj_ws) cudaFree(proj_ws);
    proj_ws = nullptr;
    proj_p = nullptr;
    proj_stats = nullptr;
    proj_refs = nullptr;
    proj_zy = nullptr;
    proj_hidden = proj_chunk = proj_n_tiles = 0;
}

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

rl_status cuda_fail(rl_loss_handle_s *h, cudaError_t e) {
    h->last_cuda_error = e;
    return RL_ERR_CUDA;
}

}  // namespace

extern "C" {

RL_LOSS_API rl_status rl_loss_projection_setup(rl_loss_t h, int32_t hidden_dim, int32_t chunk_tokens) {
    if (!h) return RL_ERR_INVALID_ARG;
    if (hidden_dim < 1 || hidden_dim % 8 != 0 || chunk_tokens < 1) return RL_ERR_SHAPE;
    if (h->cfg.logits_dtype != RL_BF16) return RL_ERR_UNSUPPORTED;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) return RL_ERR_DEVICE;
    cudaDeviceSynchronize();
    h->proj_release();
    const int64_t V = h->cfg.vocab_size;
    const int tile = rlk::proj_gemm_tile_cols();
    const int n_tiles = (int)((V + tile - 1) / tile);
    const int64_t ldp = (V + 7) / 8 * 8;
    const size_t p_bytes = align_up((size_t)chunk_tokens * ldp * 2, 256);
    const size_t st_bytes = align_up((size_t)chunk_tokens * n_tiles * sizeof(float4), 256);
    const size_t zy_bytes = align_up((size_t)chunk_tokens * sizeof(float), 256);
    void *ws = nullptr;
    cudaError_t e = cudaMalloc(&ws, p_bytes + 2 * st_bytes + zy_bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return cuda_fail(h, e);
    }
    char *b = reinterpret_cast<char *>(ws);
    h->proj_ws = ws;
    h->proj_p = b;
    h->proj_stats = reinterpret_cast<float4 *>(b + p_bytes);
    h->proj_refs = reinterpret_cast<float4 *>(b + p_bytes + st_bytes);
    h->proj_zy = reinterpret_cast<float *>(b + p_bytes + 2 * st_bytes);
    h->proj_hidden = hidden_dim;
    h->proj_chunk = chunk_tokens;
    h->proj_n_tiles = n_tiles;
    h->proj_ldp = ldp;
    return RL_OK;
}

RL_LOSS_API rl_status rl_loss_projection_logits(rl_loss_t h, const void *hidden, int64_t ld_hidden, const void *w_lm,
                                                int64_t ld_w, int32_t rows, float *logits, int64_t ld_logits,
                                                void *stream_ptr) {
    if (!h || !hidden || !w_lm || !logits) return RL_ERR_INVALID_ARG;
    if (h->proj_hidden == 0) return RL_ERR_INVALID_ARG;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) return RL_ERR_DEVICE;
    const int H = h->proj_hidden, V = h->cfg.vocab_size;
    if (rows < 0 || ld_hidden < H || ld_w < H || ld_logits < V) return RL_ERR_SHAPE;
    if (!aligned16(hidden) || !aligned16(w_lm) || (ld_hidden * 2) % 16 || (ld_w * 2) % 16 ||
        (reinterpret_cast<uintptr_t>(logits) & 15u) || (ld_logits * 4) % 16)
        return RL_ERR_ALIGNMENT;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_ptr);
    rlk::ProjGemmParams gp{};
    gp.M = rows;
    gp.N = V;
    gp.K = H;
    gp.z = logits;
    gp.ldz = ld_logits;
    gp.stats = nullptr;
    gp.status = h->status;
    const int slot = h->prof_begin(kProjGemm, stream);
    cudaError_t e = rlk::launch_proj_gemm(hidden, ld_hidden, w_lm, ld_w, gp, stream);
    h->prof_end(slot, stream);
    if (e != cudaSuccess) return cuda_fail(h, e);
    h->launches += rows > 0 ? 1 : 0;
    return RL_OK;
}

RL_LOSS_API rl_status rl_loss_fused_projection_forward_backward(
    rl_loss_t h, const void *hidden, int64_t ld_hidden, const void *w_lm, int64_t ld_w, const rl_loss_inputs *in,
    void *dhidden, int64_t ld_dhidden, float *dw_lm, int64_t ld_dw, const rl_loss_outputs *out, void *stream_ptr) {
    if (!h || !in || !out) return RL_ERR_INVALID_ARG;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) return RL_ERR_DEVICE;
    if (h->proj_hidden == 0) return RL_ERR_INVALID_ARG;
    const rl_loss_config &c = h->cfg;
    const int T = in->num_tokens, S = in->num_seqs, V = c.vocab_size, H = h->proj_hidden;
    if (T < 0 || S < 1 || S % c.group_size != 0) return RL_ERR_SHAPE;
    if (T > c.max_tokens || S > c.max_seqs) return RL_ERR_CAPACITY;
    if (!in->cu_seqlens || !in->rewards_or_adv || !out->loss) return RL_ERR_INVALID_ARG;
    if (T > 0) {
        if (!hidden || !w_lm || !dhidden || !dw_lm || !in->targets || !in->logp_old || !in->logp_infer || !in->mask)
            return RL_ERR_INVALID_ARG;
        if (ld_hidden < H || ld_w < H || ld_dhidden < H || ld_dw < H) return RL_ERR_SHAPE;
        if (!aligned16(hidden) || !aligned16(w_lm) || !aligned16(dhidden) || !aligned16(dw_lm) ||
            (ld_hidden * 2) % 16 || (ld_w * 2) % 16 || (ld_dhidden * 2) % 16 || (ld_dw * 4) % 16)
            return RL_ERR_ALIGNMENT;
    }
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_ptr);

    rlk::SeqPrepParams sp{};
    sp.cu_seqlens = in->cu_seqlens;
    sp.mask = in->mask;
    sp.rewards_or_adv = in->rewards_or_adv;
    sp.num_seqs = S;
    sp.num_tokens = T;
    sp.group_size = c.group_size;
    sp.adv_mode = c.adv_mode;
    sp.std_unbiased = c.std_unbiased;
    sp.loss_norm = c.loss_norm;
    sp.adv_eps = c.adv_eps;
    sp.seq_adv = h->seq_adv;
    sp.seq_w = h->seq_w;
    sp.seq_w64 = h->seq_w64;
    sp.seq_n = h->seq_n;
    sp.seq_adv_out = out->seq_adv;
    sp.status = h->status;
    int slot = h->prof_begin(kSegPrep, stream);
    cudaError_t e = rlk::launch_seg_prep(sp, stream);
    if (e == cudaSuccess && c.loss_norm == RL_NORM_PER_TOKEN) e = rlk::launch_seg_token_norm(sp, stream);
    h->prof_end(slot, stream);
    if (e != cudaSuccess) return cuda_fail(h, e);
    int64_t launches = 1;

    float *entropy = out->entropy ? out->entropy : h->tok_ent;
    uint8_t *flags = out->flags ? out->flags : h->tok_flags;
    for (int r0 = 0, ci = 0; r0 < T; r0 += h->proj_chunk, ++ci) {
        const int m = T - r0 < h->proj_chunk ? T - r0 : h->proj_chunk;
        const char *hc = reinterpret_cast<const char *>(hidden) + (size_t)r0 * ld_hidden * 2;

        rlk::GemmProblem fw{};
        fw.M = m;
        fw.N = V;
        fw.K = H;
        fw.a = rlk::GemmOperand{hc, ld_hidden, 0};
        fw.b = rlk::GemmOperand{w_lm, ld_w, 0};
        fw.epi = rlk::GemmProblem::kProbStats;
        fw.n_fastest = 0;  // pairs running at once share the LM-head tiles through L2
        fw.d = h->proj_p;
        fw.ldd = h->proj_ldp;
        fw.stats = h->proj_stats;
        fw.refs = h->proj_refs;
        fw.targets = in->targets + r0;
        fw.target_logit = h->proj_zy;
        slot = h->prof_begin(kProjGemm, stream);
        e = rlk::launch_gemm_problems(&fw, 1, h->status, stream);
        h->prof_end(slot, stream);
        if (e != cudaSuccess) return cuda_fail(h, e);

        rlk::TokenPrepParams tp{};
        tp.target_logit = h->proj_zy;
        tp.row0 = r0;
        tp.rows = m;
        tp.logits_dtype = RL_F32;
        tp.targets = in->targets;
        tp.logp_old = in->logp_old;
        tp.logp_infer = in->logp_infer;
        tp.mask = in->mask;
        tp.cu_seqlens = in->cu_seqlens;
        tp.num_seqs = S;
        tp.num_tokens = T;
        tp.vocab = V;
        tp.seq_adv = h->seq_adv;
        tp.seq_w = h->seq_w;
        tp.token_adv = c.adv_mode == RL_ADV_PER_TOKEN ? in->rewards_or_adv : nullptr;
        tp.c = h->consts;
        tp.rec = h->tok_rec;
        tp.meta = h->tok_meta;
        tp.status = h->status;
        slot = h->prof_begin(kTokenPrep, stream);
        e = rlk::launch_token_prep(tp, stream);
        h->prof_end(slot, stream);
        if (e != cudaSuccess) return cuda_fail(h, e);

        rlk::ProjRowParams rp{};
        rp.probs = h->proj_p;
        rp.ldp = h->proj_ldp;
        rp.stats = h->proj_stats;
        rp.refs = h->proj_refs;
        rp.n_tiles = h->proj_n_tiles;
        rp.row0 = r0;
        rp.rows = m;
        rp.vocab = V;
        rp.rec = h->tok_rec;
        rp.meta = h->tok_meta;
        rp.teacher = c.adv_mode == RL_ADV_TEACHER_LOGP ? in->rewards_or_adv : nullptr;
        rp.c = h->consts;
        rp.logp_out = out->logp;
        rp.entropy_out = entropy;
        rp.flags_out = flags;
        rp.tok_obj = h->tok_obj;
        rp.status = h->status;
        slot = h->prof_begin(kProjRows, stream);
        e = rlk::launch_proj_rows(rp, stream);
        h->prof_end(slot, stream);
        if (e != cudaSuccess) return cuda_fail(h, e);
        launches += 3;

        // dH_c [m x H] = dZ_c [m x V] W [V x H]: dZ_c is K-major, W MN-major (H contiguous)
        // dW [V x H] (+)= dZ_c^T [V x m] H_c [m x H]: dZ_c and H_c both MN-major
        rlk::GemmProblem bw[2] = {};
        bw[0].M = m;
        bw[0].N = H;
        bw[0].K = V;
        bw[0].a = rlk::GemmOperand{h->proj_p, h->proj_ldp, 0};
        bw[0].b = rlk::GemmOperand{w_lm, ld_w, 1};
        bw[0].epi = rlk::GemmProblem::kBf16;
        bw[0].n_fastest = 0;  // pairs running at once share W's column blocks through L2
        bw[0].d = reinterpret_cast<char *>(dhidden) + (size_t)r0 * ld_dhidden * 2;
        bw[0].ldd = ld_dhidden;
        bw[1].M = V;
        bw[1].N = H;
        bw[1].K = m;
        bw[1].a = rlk::GemmOperand{h->proj_p, h->proj_ldp, 1};
        bw[1].b = rlk::GemmOperand{hc, ld_hidden, 1};
        bw[1].epi = rlk::GemmProblem::kF32;
        bw[1].accumulate = ci > 0;
        bw[1].n_fastest = 1;  // a pair's consecutive tiles reuse one block of dZ_c from L2
        bw[1].d = dw_lm;
        bw[1].ldd = ld_dw;
        slot = h->prof_begin(kProjBwd, stream);
        e = rlk::launch_gemm_problems(bw, 2, h->status, stream);
        h->prof_end(slot, stream);
        if (e != cudaSuccess) return cuda_fail(h, e);
        launches += 1;
    }

    if (T == 0 && dw_lm) {  // no chunk ran: the weight gradient is zero
        e = cudaMemset2DAsync(dw_lm, (size_t)ld_dw * 4, 0, (size_t)H * 4, (size_t)V, stream);
        if (e != cudaSuccess) return cuda_fail(h, e);
    }

    rlk::ReduceParams rd{};
    rd.cu_seqlens = in->cu_seqlens;
    rd.num_seqs = S;
    rd.num_tokens = T;
    rd.tok_obj = h->tok_obj;
    rd.entropy = entropy;
    rd.flags = flags;
    rd.seq_w64 = h->seq_w64;
    rd.seq_n = h->seq_n;
    rd.seq_obj = h->seq_obj;
    rd.seq_ent = h->seq_ent;
    rd.seq_cnt = h->seq_cnt;
    rd.loss = out->loss;
    rd.loss_f64 = out->loss_f64;
    rd.counts = out->counts;
    rd.mean_entropy = out->mean_entropy;
    rd.status = h->status;
    slot = h->prof_begin(kSegReduce, stream);
    e = rlk::launch_seg_reduce(rd, stream);
    h->prof_end(slot, stream);
    if (e != cudaSuccess) return cuda_fail(h, e);
    slot = h->prof_begin(kFinalReduce, stream);
    e = rlk::launch_final_reduce(rd, stream);
    h->prof_end(slot, stream);
    if (e != cudaSuccess) return cuda_fail(h, e);
    h->launches += launches + 2;
    return RL_OK;
}

}  // extern "C"
