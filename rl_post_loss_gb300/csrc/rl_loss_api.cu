// C ABI of the fused GRPO + IcePop loss (declared in include/rl_loss.h):
// handle life cycle, host-side validation, workspace layout, launches,
// device status and event-based kernel timing.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "common.cuh"
#include "scan_select.cuh"

#include "handle.cuh"

static size_t workspace_layout(const rl_loss_config &c, rl_loss_handle_s *h, char *base) {
    const size_t S = (size_t)c.max_seqs, T = (size_t)c.max_tokens;
    size_t off = 0;
    auto carve = [&](size_t bytes) {
        off = align_up(off, 256);
        char *p = base ? base + off : nullptr;
        off += bytes;
        return p;
    };
    char *status = carve(sizeof(uint32_t));
    char *seq_adv = carve(S * sizeof(float));
    char *seq_w = carve(S * sizeof(float));
    char *seq_w64 = carve(S * sizeof(double));
    char *seq_obj = carve(S * sizeof(double));
    char *seq_ent = carve(S * sizeof(double));
    char *seq_n = carve(S * sizeof(int32_t));
    char *seq_cnt = carve(S * 4 * sizeof(int32_t));
    char *tok_obj = carve(T * sizeof(float));
    char *tok_ent = carve(T * sizeof(float));
    char *tok_flags = carve(T * sizeof(uint8_t));
    char *tok_fix = carve(T * sizeof(uint8_t));
    char *tok_rec = carve(T * sizeof(float4));
    char *tok_meta = carve(T * sizeof(uint32_t));
    char *loss_scratch = carve(4 * sizeof(float));
    if (h) {
        h->status = reinterpret_cast<uint32_t *>(status);
        h->seq_adv = reinterpret_cast<float *>(seq_adv);
        h->seq_w = reinterpret_cast<float *>(seq_w);
        h->seq_w64 = reinterpret_cast<double *>(seq_w64);
        h->seq_obj = reinterpret_cast<double *>(seq_obj);
        h->seq_ent = reinterpret_cast<double *>(seq_ent);
        h->seq_n = reinterpret_cast<int32_t *>(seq_n);
        h->seq_cnt = reinterpret_cast<int32_t *>(seq_cnt);
        h->tok_obj = reinterpret_cast<float *>(tok_obj);
        h->tok_ent = reinterpret_cast<float *>(tok_ent);
        h->tok_flags = reinterpret_cast<uint8_t *>(tok_flags);
        h->tok_fix = reinterpret_cast<uint8_t *>(tok_fix);
        h->tok_rec = reinterpret_cast<float4 *>(tok_rec);
        h->tok_meta = reinterpret_cast<uint32_t *>(tok_meta);
        h->loss_scratch = reinterpret_cast<float *>(loss_scratch);
    }
    return align_up(off, 256);
}

static int elem_size(int32_t dtype) { return dtype == RL_F32 ? 4 : 2; }

// Objective / advantage / normalisation codes of a configuration are known and compatible.
static bool config_modes_valid(const rl_loss_config &c) {
    if (c.adv_mode < RL_ADV_GROUP_REWARDS || c.adv_mode > RL_ADV_TEACHER_LOGP) return false;
    if (c.std_unbiased && c.adv_mode == RL_ADV_GROUP_REWARDS && c.group_size < 2) return false;
    if (c.objective != RL_OBJ_GRPO_ICEPOP && c.objective != RL_OBJ_DIS) return false;
    if (c.objective == RL_OBJ_DIS && c.adv_mode == RL_ADV_TEACHER_LOGP) return false;
    if (c.loss_norm != RL_NORM_PER_RESPONSE && c.loss_norm != RL_NORM_PER_TOKEN) return false;
    if (c.dis_stopgrad != 0 && c.dis_stopgrad != 1) return false;
    return true;
}

// fp32 decision thresholds, each rounded once from a double, and the modes.
static rlk::LossConsts loss_consts(const rl_loss_config &c) {
    rlk::LossConsts k{};
    k.ln_beta = (float)std::log((double)c.beta);
    k.clip_hi = (float)std::log1p((double)c.eps_high);
    k.clip_lo = (float)std::log1p(-(double)c.eps_low);
    k.one_plus_eps_high = 1.f + c.eps_high;
    k.one_minus_eps_low = 1.f - c.eps_low;
    k.pop_indicator = c.pop_indicator ? 1 : 0;
    k.objective = c.objective;
    k.dis_stopgrad = c.dis_stopgrad;
    k.adv_teacher = c.adv_mode == RL_ADV_TEACHER_LOGP ? 1 : 0;
    return k;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The parameters of one loss call's kernels.
struct LossLaunch {
    rlk::SeqPrepParams sp;
    rlk::TokenPrepParams tp;
    rlk::RowParams rp;
    rlk::ReduceParams rd;
    int T;
    int es;
};

// Checks what rl_loss_forward_backward requires of the handle, `in` and `out`, and fills the
// parameters of its kernels.
static rl_status prepare_call(rl_loss_handle_s *h, const rl_loss_inputs *in, const rl_loss_outputs *out,
                              LossLaunch &L) {
    if (!h || !in || !out) return RL_ERR_INVALID_ARG;
    int cur = -1;
    if (cudaError_t e0 = cudaGetDevice(&cur); e0 != cudaSuccess) {
        h->last_cuda_error = e0;
        return RL_ERR_CUDA;
    }
    if (cur != h->device) return RL_ERR_DEVICE;
    const rl_loss_config &c = h->cfg;
    const int T = in->num_tokens, S = in->num_seqs, V = c.vocab_size;
    const int es = elem_size(c.logits_dtype);
    if (T < 0 || S < 1 || S % c.group_size != 0) return RL_ERR_SHAPE;
    if (T > c.max_tokens || S > c.max_seqs) return RL_ERR_CAPACITY;
    if (!in->cu_seqlens || !in->rewards_or_adv || !out->loss) return RL_ERR_INVALID_ARG;
    if (T > 0) {
        if (!in->logits || !in->targets || !in->logp_old || !in->logp_infer || !in->mask || !out->dlogits)
            return RL_ERR_INVALID_ARG;
        if (in->ld_logits < V || out->ld_dlogits < V) return RL_ERR_SHAPE;
        if (!aligned16(in->logits) || !aligned16(out->dlogits) || (in->ld_logits * es) % 16 != 0 ||
            (out->ld_dlogits * es) % 16 != 0)
            return RL_ERR_ALIGNMENT;
        if (in->logits == out->dlogits && in->ld_logits != out->ld_dlogits) return RL_ERR_INVALID_ARG;
    }
    L.T = T;
    L.es = es;

    rlk::SeqPrepParams &sp = L.sp;
    sp = rlk::SeqPrepParams{};
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

    rlk::TokenPrepParams &tp = L.tp;
    tp = rlk::TokenPrepParams{};
    tp.logits = in->logits;
    tp.ld_logits = in->ld_logits;
    tp.row0 = 0;
    tp.rows = T;
    tp.logits_dtype = c.logits_dtype;
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

    rlk::RowParams &rp = L.rp;
    rp = rlk::RowParams{};
    rp.logits = in->logits;
    rp.ld_logits = in->ld_logits;
    rp.dlogits = out->dlogits;
    rp.ld_dlogits = out->ld_dlogits;
    rp.rec = h->tok_rec;
    rp.meta = h->tok_meta;
    rp.teacher = c.adv_mode == RL_ADV_TEACHER_LOGP ? in->rewards_or_adv : nullptr;
    rp.num_tokens = T;
    rp.vocab = V;
    rp.c = h->consts;
    rp.logp_out = out->logp;
    rp.entropy_out = out->entropy ? out->entropy : h->tok_ent;
    rp.flags_out = out->flags ? out->flags : h->tok_flags;
    rp.tok_obj = h->tok_obj;
    rp.status = h->status;
    rp.fix_rows = h->tok_fix;

    rlk::ReduceParams &rd = L.rd;
    rd = rlk::ReduceParams{};
    rd.cu_seqlens = in->cu_seqlens;
    rd.num_seqs = S;
    rd.num_tokens = T;
    rd.tok_obj = h->tok_obj;
    rd.entropy = rp.entropy_out;
    rd.flags = rp.flags_out;
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
    return RL_OK;
}

// The token preparation and row kernel parameters restricted to tokens [r0, r1).
static void restrict_rows(LossLaunch &B, const LossLaunch &L, int r0, int r1) {
    B = L;
    const size_t es = (size_t)L.es;
    B.tp.logits = static_cast<const char *>(L.tp.logits) + (size_t)r0 * (size_t)L.tp.ld_logits * es;
    B.tp.row0 = r0;
    B.tp.rows = r1 - r0;
    rlk::RowParams &rp = B.rp;
    rp.logits = static_cast<const char *>(L.rp.logits) + (size_t)r0 * (size_t)L.rp.ld_logits * es;
    rp.dlogits = static_cast<char *>(L.rp.dlogits) + (size_t)r0 * (size_t)L.rp.ld_dlogits * es;
    rp.rec = L.rp.rec + r0;
    rp.meta = L.rp.meta + r0;
    if (L.rp.teacher) rp.teacher = L.rp.teacher + r0;
    if (L.rp.logp_out) rp.logp_out = L.rp.logp_out + r0;
    rp.entropy_out = L.rp.entropy_out + r0;
    rp.flags_out = L.rp.flags_out + r0;
    rp.tok_obj = L.rp.tok_obj + r0;
    rp.fix_rows = L.rp.fix_rows + r0;
    rp.num_tokens = r1 - r0;
}

// Enqueues one loss call on `stream`. With nb > 0 blocks (rows[b] .. rows[b + 1]), the token
// preparation and row kernel of block b wait for h->copy_done[b] first.
static rl_status launch_loss(rl_loss_handle_s *h, const LossLaunch &L, const int *rows, int nb, cudaStream_t stream) {
    const rl_loss_config &c = h->cfg;
    cudaError_t err;
    auto failed = [&](cudaError_t e) {
        h->last_cuda_error = e;
        return RL_ERR_CUDA;
    };
    int slot = h->prof_begin(kSegPrep, stream);
    err = rlk::launch_seg_prep(L.sp, stream);
    if (err == cudaSuccess && c.loss_norm == RL_NORM_PER_TOKEN) err = rlk::launch_seg_token_norm(L.sp, stream);
    h->prof_end(slot, stream);
    if (err != cudaSuccess) return failed(err);
    int64_t row_launches = 0;
    const int blocks = nb > 0 ? nb : 1;
    for (int b = 0; b < blocks; ++b) {
        LossLaunch B;
        if (nb > 0) {
            restrict_rows(B, L, rows[b], rows[b + 1]);
            err = cudaStreamWaitEvent(stream, h->copy_done[b], 0);
            if (err != cudaSuccess) return failed(err);
        } else {
            B = L;
        }
        if (B.tp.rows <= 0) continue;
        slot = h->prof_begin(kTokenPrep, stream);
        err = rlk::launch_token_prep(B.tp, stream);
        h->prof_end(slot, stream);
        if (err != cudaSuccess) return failed(err);
        slot = h->prof_begin(kRowLoss, stream);
        err = rlk::launch_row_loss(B.rp, c.logits_dtype, stream);
        h->prof_end(slot, stream);
        if (err != cudaSuccess) return failed(err);
        row_launches += 2;
    }
    if (L.rp.num_tokens > 0) {  // after every row block: the entropy of rows holding -inf logits
        slot = h->prof_begin(kEntropyFix, stream);
        err = rlk::launch_entropy_fix(L.rp, c.logits_dtype, stream);
        h->prof_end(slot, stream);
        if (err != cudaSuccess) return failed(err);
        row_launches += 1;
    }
    slot = h->prof_begin(kSegReduce, stream);
    err = rlk::launch_seg_reduce(L.rd, stream);
    h->prof_end(slot, stream);
    if (err != cudaSuccess) return failed(err);
    slot = h->prof_begin(kFinalReduce, stream);
    err = rlk::launch_final_reduce(L.rd, stream);
    h->prof_end(slot, stream);
    if (err != cudaSuccess) return failed(err);
    h->launches += 3 + row_launches + (c.loss_norm == RL_NORM_PER_TOKEN ? 1 : 0);
    return RL_OK;
}

extern "C" {

RL_LOSS_API int32_t rl_loss_version(void) { return 100; }

RL_LOSS_API const char *rl_loss_status_string(rl_status s) {
    switch (s) {
        case RL_OK: return "ok";
        case RL_ERR_INVALID_ARG: return "invalid argument";
        case RL_ERR_SHAPE: return "bad shape";
        case RL_ERR_DTYPE: return "unsupported dtype";
        case RL_ERR_ALIGNMENT: return "pointer or row stride not 16-byte aligned";
        case RL_ERR_CAPACITY: return "batch exceeds the handle's capacity";
        case RL_ERR_CUDA: return "CUDA error";
        case RL_ERR_TARGET_RANGE: return "target id outside [0, V)";
        case RL_ERR_NONFINITE: return "non-finite logits or loss";
        case RL_ERR_EMPTY_SEQ: return "response without mask=1 tokens";
        case RL_ERR_TIMEOUT: return "bounded wait ran out";
        case RL_ERR_UNSUPPORTED: return "unsupported request";
        case RL_ERR_SEQLENS: return "malformed cu_seqlens";
        case RL_ERR_DEVICE: return "handle used on another device";
        case RL_ERR_INTERNAL: return "internal consistency check failed";
    }
    return "unknown status";
}

RL_LOSS_API rl_status rl_loss_create(const rl_loss_config *config, rl_loss_t *out) {
    if (!out) return RL_ERR_INVALID_ARG;
    *out = nullptr;
    if (!config) return RL_ERR_INVALID_ARG;
    const rl_loss_config &c = *config;
    if (c.logits_dtype != RL_F32 && c.logits_dtype != RL_BF16) return RL_ERR_DTYPE;
    if (c.vocab_size < 1 || c.vocab_size >= rlk::kMaxVocab || c.group_size < 1 || c.max_tokens < 0 ||
        c.max_seqs < 1)
        return RL_ERR_SHAPE;
    if (!(c.beta > 1.f) || !std::isfinite(c.beta)) return RL_ERR_INVALID_ARG;
    if (!(c.eps_low >= 0.f && c.eps_low < 1.f) || !(c.eps_high >= 0.f) || !std::isfinite(c.eps_high))
        return RL_ERR_INVALID_ARG;
    if (!(c.adv_eps >= 0.f) || !std::isfinite(c.adv_eps)) return RL_ERR_INVALID_ARG;
    if (!config_modes_valid(c)) return RL_ERR_INVALID_ARG;

    rl_loss_handle_s *h = new (std::nothrow) rl_loss_handle_s();
    if (!h) return RL_ERR_INVALID_ARG;
    h->cfg = c;
    if (cudaGetDevice(&h->device) != cudaSuccess) {
        delete h;
        return RL_ERR_CUDA;
    }
    h->consts = loss_consts(c);

    h->ws_bytes = workspace_layout(c, nullptr, nullptr);
    if (cudaMalloc(&h->ws, h->ws_bytes) != cudaSuccess) {
        cudaGetLastError();
        delete h;
        return RL_ERR_CUDA;
    }
    workspace_layout(c, h, reinterpret_cast<char *>(h->ws));
    if (cudaMemset(h->status, 0, sizeof(uint32_t)) != cudaSuccess ||
        cudaMemset(h->tok_fix, 0, (size_t)c.max_tokens) != cudaSuccess) {
        cudaFree(h->ws);
        delete h;
        return RL_ERR_CUDA;
    }
    h->launches = 0;
    h->last_cuda_error = cudaSuccess;
    *out = h;
    return RL_OK;
}

RL_LOSS_API rl_status rl_loss_destroy(rl_loss_t h) {
    if (!h) return RL_OK;
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != h->device) cudaSetDevice(h->device);
    cudaDeviceSynchronize();
    for (cudaEvent_t e : h->prof_events) cudaEventDestroy(e);
    h->proj_release();
    h->copy_release();
    cudaError_t err = cudaFree(h->ws);
    if (cur != h->device && cur >= 0) cudaSetDevice(cur);
    delete h;
    return err == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

RL_LOSS_API rl_status rl_loss_forward_backward(rl_loss_t h, const rl_loss_inputs *in, const rl_loss_outputs *out,
                                               void *stream_ptr) {
    LossLaunch L;
    const rl_status st = prepare_call(h, in, out, L);
    if (st != RL_OK) return st;
    return launch_loss(h, L, nullptr, 0, reinterpret_cast<cudaStream_t>(stream_ptr));
}

RL_LOSS_API rl_status rl_loss_forward_backward_from_host(rl_loss_t h, const rl_loss_inputs *host,
                                                         const rl_loss_inputs *dev, const rl_loss_outputs *out,
                                                         int32_t num_chunks, void *stream_ptr) {
    if (!h || !host || !dev || !out) return RL_ERR_INVALID_ARG;
    if (num_chunks < 1 || num_chunks > kMaxCopyChunks) return RL_ERR_INVALID_ARG;
    const rl_loss_config &c = h->cfg;
    const int T = host->num_tokens, S = host->num_seqs, V = c.vocab_size;
    const int es = elem_size(c.logits_dtype);
    // the device side must pass every check of rl_loss_forward_backward, with the host's sizes
    rl_loss_inputs d = *dev;
    d.num_tokens = T;
    d.num_seqs = S;
    LossLaunch L;
    rl_status st = prepare_call(h, &d, out, L);
    if (st != RL_OK) return st;
    if (!host->cu_seqlens || !host->rewards_or_adv) return RL_ERR_INVALID_ARG;
    if (T > 0) {
        if (!host->logits || !host->targets || !host->logp_old || !host->logp_infer || !host->mask)
            return RL_ERR_INVALID_ARG;
        if (host->ld_logits < V) return RL_ERR_SHAPE;
    }
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_ptr);
    auto failed = [&](cudaError_t e) {
        h->last_cuda_error = e;
        return RL_ERR_CUDA;
    };
    cudaError_t err = h->copy_setup();
    if (err != cudaSuccess) return failed(err);

    // the logits blocks start once the work enqueued before this call (which may still read the
    // device buffers) is done
    const int nb = T > 0 ? std::min(num_chunks, T) : 0;
    if (nb > 0) {
        err = cudaEventRecord(h->copy_entry, stream);
        if (err == cudaSuccess) err = cudaStreamWaitEvent(h->copy_stream, h->copy_entry, 0);
        if (err != cudaSuccess) return failed(err);
    }
    // the small arrays, on the caller's stream
    const bool adv_per_token = c.adv_mode == RL_ADV_PER_TOKEN || c.adv_mode == RL_ADV_TEACHER_LOGP;
    const size_t tok = (size_t)T;
    struct Part {
        void *dst;
        const void *src;
        size_t bytes;
    } parts[] = {
        {const_cast<int32_t *>(d.cu_seqlens), host->cu_seqlens, ((size_t)S + 1) * sizeof(int32_t)},
        {const_cast<float *>(d.rewards_or_adv), host->rewards_or_adv, (adv_per_token ? tok : (size_t)S) * sizeof(float)},
        {const_cast<int32_t *>(d.targets), host->targets, tok * sizeof(int32_t)},
        {const_cast<float *>(d.logp_old), host->logp_old, tok * sizeof(float)},
        {const_cast<float *>(d.logp_infer), host->logp_infer, tok * sizeof(float)},
        {const_cast<uint8_t *>(d.mask), host->mask, tok * sizeof(uint8_t)},
    };
    for (const Part &q : parts) {
        if (q.bytes == 0 || !q.dst) continue;
        err = cudaMemcpyAsync(q.dst, q.src, q.bytes, cudaMemcpyHostToDevice, stream);
        if (err != cudaSuccess) return failed(err);
    }
    // the logits, block by block, on the copy stream
    int rows[kMaxCopyChunks + 1];
    for (int b = 0; b <= nb; ++b) rows[b] = (int)((int64_t)T * b / std::max(nb, 1));
    for (int b = 0; b < nb; ++b) {
        const int r0 = rows[b], n = rows[b + 1] - r0;
        char *dst = const_cast<char *>(static_cast<const char *>(d.logits)) + (size_t)r0 * d.ld_logits * es;
        const char *src = static_cast<const char *>(host->logits) + (size_t)r0 * host->ld_logits * es;
        // one flat copy only when rows are packed on both sides: with ld > V it would touch the
        // padding columns and read past the end of a host buffer of (T - 1) * ld + V elements
        if (host->ld_logits == V && d.ld_logits == V)
            err = cudaMemcpyAsync(dst, src, (size_t)n * V * es, cudaMemcpyHostToDevice, h->copy_stream);
        else
            err = cudaMemcpy2DAsync(dst, (size_t)d.ld_logits * es, src, (size_t)host->ld_logits * es, (size_t)V * es,
                                    (size_t)n, cudaMemcpyHostToDevice, h->copy_stream);
        if (err == cudaSuccess) err = cudaEventRecord(h->copy_done[b], h->copy_stream);
        if (err != cudaSuccess) return failed(err);
    }
    return launch_loss(h, L, rows, nb, stream);
}

RL_LOSS_API rl_status rl_loss_get_device_status(rl_loss_t h, void *stream_ptr, uint32_t *bits) {
    if (!h || !bits) return RL_ERR_INVALID_ARG;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_ptr);
    uint32_t v = 0;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess) e = cudaMemcpy(&v, h->status, sizeof v, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(h->status, 0, sizeof v);
    if (e != cudaSuccess) {
        h->last_cuda_error = e;
        return RL_ERR_CUDA;
    }
    *bits = v;
    return RL_OK;
}

RL_LOSS_API rl_status rl_loss_profile_start(rl_loss_t h, int32_t max_calls) {
    if (!h || max_calls < 0) return RL_ERR_INVALID_ARG;
    return h->prof_reset((size_t)max_calls * kProfSlotsPerCall) ? RL_OK : RL_ERR_CUDA;
}

RL_LOSS_API rl_status rl_loss_profile_read(rl_loss_t h, rl_loss_profile *out) {
    if (!h || !out) return RL_ERR_INVALID_ARG;
    std::memset(out, 0, sizeof *out);
    out->num_kernels = kNumKernels;
    for (int k = 0; k < kNumKernels; ++k) std::snprintf(out->names[k], sizeof out->names[k], "%s", kKernelNames[k]);
    for (int i = 0; i < h->prof_used; ++i) {
        cudaEvent_t a = h->prof_events[2 * (size_t)i], b = h->prof_events[2 * (size_t)i + 1];
        if (cudaEventSynchronize(b) != cudaSuccess) return RL_ERR_CUDA;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, a, b) != cudaSuccess) return RL_ERR_CUDA;
        out->launches[h->prof_cls[i]] += 1;
        out->total_ms[h->prof_cls[i]] += ms;
    }
    h->prof_capacity = 0;
    h->prof_used = 0;
    return RL_OK;
}

RL_LOSS_API const char *rl_loss_last_cuda_error(rl_loss_t h) {
    if (!h) return "no handle";
    return cudaGetErrorName(h->last_cuda_error);
}

RL_LOSS_API rl_status rl_loss_launch_count(rl_loss_t h, int64_t *count) {
    if (!h || !count) return RL_ERR_INVALID_ARG;
    *count = h->launches;
    return RL_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- allocation-free entry point
//
// Some callers cannot call cudaMalloc at the moment they need the loss: code
// inside a framework whose caching allocator owns all device memory, or a
// serving process with a fixed memory budget where an allocation could fail or
// synchronise the device. rl_loss_forward_backward_noalloc serves them without a handle: its
// workspace is one statically sized device array of this library, which every
// GPU that loads the library holds until the process exits.
namespace {

constexpr int32_t kNoAllocMaxTokens = 262144;
constexpr int32_t kNoAllocMaxSeqs = 8192;
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the static scratch on `device` (the current device),
// looked up once per device.
rl_status noalloc_scratch(int device, void **ptr) {
    if (device < 0 || device >= kNoAllocMaxDevices) return RL_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[device]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return RL_ERR_CUDA;
        }
        g_noalloc_ptr[device] = p;
    }
    *ptr = g_noalloc_ptr[device];
    return RL_OK;
}

}  // namespace

extern "C" RL_LOSS_API rl_status rl_loss_forward_backward_noalloc(const rl_loss_config *config,
                                                                  const rl_loss_inputs *inputs,
                                                                  const rl_loss_outputs *outputs,
                                                                  uint32_t *device_status, void *stream_ptr) {
    if (!config || !inputs || !outputs) return RL_ERR_INVALID_ARG;
    const rl_loss_config &c = *config;
    if (c.logits_dtype != RL_F32 && c.logits_dtype != RL_BF16) return RL_ERR_DTYPE;
    if (c.vocab_size < 1 || c.vocab_size >= rlk::kMaxVocab || c.group_size < 1) return RL_ERR_SHAPE;
    if (!(c.beta > 1.f) || !std::isfinite(c.beta)) return RL_ERR_INVALID_ARG;
    if (!(c.eps_low >= 0.f && c.eps_low < 1.f) || !(c.eps_high >= 0.f) || !std::isfinite(c.eps_high))
        return RL_ERR_INVALID_ARG;
    if (!(c.adv_eps >= 0.f) || !std::isfinite(c.adv_eps)) return RL_ERR_INVALID_ARG;
    if (!config_modes_valid(c)) return RL_ERR_INVALID_ARG;
    if (inputs->num_tokens > kNoAllocMaxTokens || inputs->num_seqs > kNoAllocMaxSeqs) return RL_ERR_CAPACITY;

    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) return RL_ERR_CUDA;
    void *scratch = nullptr;
    rl_status st = noalloc_scratch(device, &scratch);
    if (st != RL_OK) return st;

    // A handle that lives on the stack and points into the static scratch.
    rl_loss_handle_s h{};
    h.cfg = c;
    h.cfg.max_tokens = kNoAllocMaxTokens;
    h.cfg.max_seqs = kNoAllocMaxSeqs;
    h.device = device;
    h.consts = loss_consts(c);
    h.ws_bytes = workspace_layout(h.cfg, nullptr, nullptr);
    if (h.ws_bytes > kNoAllocScratchBytes) return RL_ERR_CAPACITY;
    h.ws = scratch;
    workspace_layout(h.cfg, &h, reinterpret_cast<char *>(scratch));

    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_ptr);
    // the scratch keeps the previous call's contents: the status word must start at zero
    if (cudaMemsetAsync(h.status, 0, sizeof(uint32_t), stream) != cudaSuccess) return RL_ERR_CUDA;
    st = rl_loss_forward_backward(&h, inputs, outputs, stream_ptr);
    if (st != RL_OK) return st;
    if (device_status &&
        cudaMemcpyAsync(device_status, h.status, sizeof(uint32_t), cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
        return RL_ERR_CUDA;
    return RL_OK;
}

extern "C" RL_LOSS_API size_t rl_gae_workspace_bytes(int32_t num_tokens) {
    return rlk::gae_workspace_bytes(num_tokens < 0 ? 0 : num_tokens);
}

namespace {

rl_status gae_call(const rl_gae_config *config, int32_t num_tokens, int32_t num_seqs, const float *rewards,
                   const float *values, const uint8_t *mask, const int32_t *cu_seqlens, const int32_t *rollout_ids,
                   float *advantages, float *returns, void *workspace, size_t workspace_bytes,
                   uint32_t *device_status, void *stream_ptr, uint64_t wait_ns, int32_t withhold_chunk) {
    if (!config) return RL_ERR_INVALID_ARG;
    const rl_gae_config &c = *config;
    if (!(c.gamma >= 0.0 && c.gamma <= 1.0) || !(c.lambda >= 0.0 && c.lambda <= 1.0)) return RL_ERR_INVALID_ARG;
    if (num_tokens < 0 || num_seqs < 1) return RL_ERR_SHAPE;
    if (!cu_seqlens || (num_tokens > 0 && (!rewards || !values || !mask || !advantages || !workspace)))
        return RL_ERR_INVALID_ARG;
    if (c.cross_trajectory && !rollout_ids) return RL_ERR_INVALID_ARG;
    if (num_tokens > 0 && workspace_bytes < rlk::gae_workspace_bytes(num_tokens)) return RL_ERR_CAPACITY;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return RL_ERR_ALIGNMENT;
    if ((reinterpret_cast<uintptr_t>(rewards) | reinterpret_cast<uintptr_t>(values) |
         reinterpret_cast<uintptr_t>(advantages) | reinterpret_cast<uintptr_t>(returns)) & 3u)
        return RL_ERR_ALIGNMENT;
    rlk::GaeParams p{};
    p.cu_seqlens = cu_seqlens;
    p.num_seqs = num_seqs;
    p.num_tokens = num_tokens;
    p.rewards = rewards;
    p.values = values;
    p.mask = mask;
    const double gl = c.gamma * c.lambda;
    p.gamma = (float)c.gamma;
    p.gl = (float)gl;
    p.gl_kind = gl == 0.0 ? 1 : (gl == 1.0 ? 2 : 0);
    p.log2_gl = p.gl_kind == 0 ? std::log2(gl) : 0.0;
    p.log2_gl_hi = (float)p.log2_gl;
    p.log2_gl_lo = (float)(p.log2_gl - (double)p.log2_gl_hi);
    p.skip_observations = c.skip_observations ? 1 : 0;
    p.rollout_ids = c.cross_trajectory ? rollout_ids : nullptr;
    p.adv = advantages;
    p.returns = returns;
    p.workspace = workspace;
    p.status = device_status;  // may be NULL: the bits are then not reported
    p.wait_ns = wait_ns;
    p.withhold_chunk = withhold_chunk;
    if (rlk::launch_gae(p, reinterpret_cast<cudaStream_t>(stream_ptr)) != cudaSuccess) return RL_ERR_CUDA;
    return RL_OK;
}

}  // namespace

extern "C" RL_LOSS_API rl_status rl_gae_advantages(const rl_gae_config *config, int32_t num_tokens, int32_t num_seqs,
                                                   const float *rewards, const float *values, const uint8_t *mask,
                                                   const int32_t *cu_seqlens, const int32_t *rollout_ids,
                                                   float *advantages, float *returns, void *workspace,
                                                   size_t workspace_bytes, uint32_t *device_status,
                                                   void *stream_ptr) {
    return gae_call(config, num_tokens, num_seqs, rewards, values, mask, cu_seqlens, rollout_ids, advantages, returns,
                    workspace, workspace_bytes, device_status, stream_ptr, 1000000000ull, -1);
}

extern "C" RL_LOSS_API rl_status rl_gae_advantages_withheld(const rl_gae_config *config, int32_t num_tokens,
                                                            int32_t num_seqs, const float *rewards,
                                                            const float *values, const uint8_t *mask,
                                                            const int32_t *cu_seqlens, const int32_t *rollout_ids,
                                                            float *advantages, float *returns, void *workspace,
                                                            size_t workspace_bytes, uint32_t *device_status,
                                                            void *stream_ptr, int32_t withhold_chunk,
                                                            double wait_limit_s) {
    if (withhold_chunk < 0 || !(wait_limit_s > 0.0 && wait_limit_s <= 1.0)) return RL_ERR_INVALID_ARG;
    return gae_call(config, num_tokens, num_seqs, rewards, values, mask, cu_seqlens, rollout_ids, advantages, returns,
                    workspace, workspace_bytes, device_status, stream_ptr, (uint64_t)(wait_limit_s * 1e9),
                    withhold_chunk);
}

extern "C" RL_LOSS_API int32_t rl_topk_max_k(void) { return rlk::topk_max_k(); }

extern "C" RL_LOSS_API rl_status rl_topk(const rl_topk_config *config, int32_t rows, const float *scores, int64_t ld,
                                         const int32_t *lengths, int32_t *out_idx, float *out_val, int64_t ldo,
                                         uint32_t *device_status, void *stream_ptr) {
    if (!config) return RL_ERR_INVALID_ARG;
    const rl_topk_config &c = *config;
    if (c.order != RL_TOPK_BY_SCORE && c.order != RL_TOPK_BY_POSITION) return RL_ERR_INVALID_ARG;
    if (c.k < 1 || c.k > rlk::topk_max_k()) return RL_ERR_UNSUPPORTED;
    if (rows < 0 || ld < 1 || ld > INT32_MAX || ldo < c.k) return RL_ERR_SHAPE;
    if (rows == 0) return RL_OK;
    if (!scores || !out_idx) return RL_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(scores) & 15u) || (ld & 3) || (reinterpret_cast<uintptr_t>(out_idx) & 3u) ||
        (reinterpret_cast<uintptr_t>(out_val) & 3u) || (reinterpret_cast<uintptr_t>(lengths) & 3u))
        return RL_ERR_ALIGNMENT;
    rlk::TopkParams p{};
    p.scores = scores;
    p.ld = ld;
    p.lengths = lengths;
    p.rows = rows;
    p.k = c.k;
    p.order_by_score = c.order == RL_TOPK_BY_SCORE ? 1 : 0;
    p.out_idx = out_idx;
    p.out_val = out_val;
    p.ldo = ldo;
    p.status = device_status;
    if (rlk::launch_topk(p, reinterpret_cast<cudaStream_t>(stream_ptr)) != cudaSuccess) return RL_ERR_CUDA;
    return RL_OK;
}
