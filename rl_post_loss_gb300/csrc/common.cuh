// Shared device helpers of the fused GRPO + IcePop loss kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "rl_loss.h"

namespace rlk {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// 2^x on the MUFU unit (PTX ex2.approx.ftz.f32: relative error about 2^-22).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Round two floats to bf16 (round-to-nearest-even) and pack: `a` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Loss constants shared by every kernel that evaluates the token objective.
struct LossConsts {
    float ln_beta;        // fl32(ln beta): pop bound on fl32(logp_old - logp_infer)
    float clip_hi;        // fl32(ln(1 + eps_high)): A > 0 clipped when fl32(logp - logp_old) > clip_hi
    float clip_lo;        // fl32(ln(1 - eps_low)):  A < 0 clipped when fl32(logp - logp_old) < clip_lo
    float one_plus_eps_high;
    float one_minus_eps_low;
    int32_t pop_indicator;
    int32_t objective;     // rl_objective
    int32_t dis_stopgrad;  // RL_OBJ_DIS: f(r) held constant in the gradient
    int32_t adv_teacher;   // A_t = fl32(logp_teacher - logp) (RL_ADV_TEACHER_LOGP)
};

// ---------------------------------------------------------------- per-token record
//
// Everything a row kernel needs about token t besides its logits row, prepared
// once per call by token_prep (the parts of the objective that do not depend
// on the row's softmax):
//   rec[t]  = {z_y, l_ref, c, w * c}   with l_ref = logp_old (Eq. (1)) or the
//             rollout log-prob logp_infer (DIS), and c = m * pop(rho) * A
//             (Eq. (1)), m * pop(rho) (Eq. (1) with the distillation advantage,
//             whose A needs logp), or m * A (DIS); c = 0 for masked, popped or
//             bad-target tokens
//   meta[t] = y (low 24 bits) | pre-flags << 24
// pre-flags: RL_FLAG_POP_IN_BOUNDS, RL_FLAG_MASKED, RL_FLAG_BAD_TARGET, and the
// sign of A in the two internal bits below (stripped from the output flags).
constexpr uint32_t kMetaYMask = 0x00FFFFFFu;
constexpr uint32_t kPreAPos = 0x10u;
constexpr uint32_t kPreANeg = 0x20u;
constexpr uint32_t kPreOut = RL_FLAG_POP_IN_BOUNDS | RL_FLAG_MASKED | RL_FLAG_BAD_TARGET;
constexpr int32_t kMaxVocab = 1 << 24;

// ---------------------------------------------------------------- row statistics (base 2)
//
// Running softmax statistics of part of a row, with exponents in log2 units:
//   m2 = a reference point (the part's max of z * log2 e), s = sum 2^{z log2e - m2},
//   u2 = sum 2^{z log2e - m2} (z log2e - m2).
// For a whole row with M2, S2, U2: logZ = (M2 + log2 S2) ln 2 and the entropy
// H = -sum p ln p = (log2 S2 - U2 / S2) ln 2.
struct RowStats2 {
    float m2, s, u2;
};

__device__ __forceinline__ RowStats2 empty_stats() { return RowStats2{-INFINITY, 0.f, 0.f}; }

// Merge two partial statistics. Symmetric in its arguments (explicit _rn
// operations, no FMA contraction), so a butterfly gives every lane bit-identical
// results, and exact for empty parts.
__device__ __forceinline__ RowStats2 merge_stats2(RowStats2 a, RowStats2 b) {
    const float M = fmaxf(a.m2, b.m2);
    if (M == -INFINITY) return empty_stats();
    const bool ea = a.m2 == -INFINITY, eb = b.m2 == -INFINITY;
    const float da = ea ? 0.f : __fsub_rn(a.m2, M), db = eb ? 0.f : __fsub_rn(b.m2, M);
    const float fa = ea ? 0.f : ex2_approx(da), fb = eb ? 0.f : ex2_approx(db);
    const float ua = ea ? 0.f : __fmul_rn(fa, __fadd_rn(a.u2, __fmul_rn(da, a.s)));
    const float ub = eb ? 0.f : __fmul_rn(fb, __fadd_rn(b.u2, __fmul_rn(db, b.s)));
    return RowStats2{M, __fadd_rn(__fmul_rn(a.s, fa), __fmul_rn(b.s, fb)), __fadd_rn(ua, ub)};
}

__device__ __forceinline__ RowStats2 warp_merge_stats2(RowStats2 r) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        RowStats2 o{__shfl_xor_sync(0xffffffffu, r.m2, off), __shfl_xor_sync(0xffffffffu, r.s, off),
                    __shfl_xor_sync(0xffffffffu, r.u2, off)};
        r = merge_stats2(r, o);
    }
    return r;
}

// Per-row results of the token objective ("GLM-5: from Vibe Coding to Agentic
// Engineering", section 3.2, Eq. (1)) from the row's statistics and record.
struct RowOut {
    float logp;   // z_y - logZ (NaN for a bad target)
    float H;      // entropy of softmax(z)
    float g;      // dL/dlogp_t
    float obj;    // m * pop * min(r A, clip(r) A)
    float logZ2;  // logZ in log2 units
    uint32_t y;
    uint32_t flags;
};

// `teacher` is log pi_teacher(y_t) when c.adv_teacher (ignored otherwise).
__device__ __forceinline__ RowOut finish_row(RowStats2 st, float4 rec, uint32_t meta, const LossConsts &c,
                                             float teacher = 0.f) {
    RowOut o;
    const float log2S = log2f(st.s);
    o.logZ2 = st.m2 + log2S;
    const float logZ = o.logZ2 * kLn2;
    o.H = (log2S - st.u2 / st.s) * kLn2;
    uint32_t pre = meta >> 24;
    o.y = meta & kMetaYMask;
    const bool ok = !(pre & RL_FLAG_BAD_TARGET);
    o.logp = ok ? __fsub_rn(rec.x, logZ) : __int_as_float(0x7fc00000);
    const float e = __fsub_rn(o.logp, rec.y);  // ln r, one fp32 subtraction
    o.obj = 0.f;
    o.g = 0.f;
    if (c.objective == RL_OBJ_DIS) {
        // direct double-sided importance sampling: f(r) = r on the open interval
        const bool gate = ok && e > c.clip_lo && e < c.clip_hi;
        o.flags = (pre & (RL_FLAG_MASKED | RL_FLAG_BAD_TARGET)) | (gate ? RL_FLAG_POP_IN_BOUNDS : 0u);
        if (gate && rec.z != 0.f) {  // m * A != 0
            const float ratio = expf(e);
            o.obj = rec.z * ratio * o.logp;
            o.g = c.dis_stopgrad ? -rec.w * ratio : -rec.w * ratio * (1.f + o.logp);
        }
        return o;
    }
    float A = 1.f;  // rec.z / rec.w already carry A unless it comes from the teacher
    if (c.adv_teacher) {
        A = ok ? __fsub_rn(teacher, o.logp) : 0.f;  // sg[log pi_teacher - log pi_theta], in fp32
        pre = (pre & ~(kPreAPos | kPreANeg)) | (A > 0.f ? kPreAPos : 0u) | (A < 0.f ? kPreANeg : 0u);
    }
    const bool clip = ok && (((pre & kPreAPos) && e > c.clip_hi) || ((pre & kPreANeg) && e < c.clip_lo));
    o.flags = (pre & kPreOut) | (clip ? RL_FLAG_CLIP_ACTIVE : 0u);
    if (rec.z != 0.f && A != 0.f) {  // m * pop * A != 0
        const float ratio = expf(e);
        const float branch = clip ? ((pre & kPreAPos) ? c.one_plus_eps_high : c.one_minus_eps_low) : ratio;
        o.obj = rec.z * A * branch;
        o.g = clip ? 0.f : -rec.w * A * ratio;
    }
    return o;
}

// Index i with cu[i] <= t < cu[i+1], or -1 (binary search over S+1 offsets).
__device__ __forceinline__ int find_seq(const int32_t *__restrict__ cu, int S, int t) {
    int lo = 0, hi = S;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(cu + mid) <= t) lo = mid; else hi = mid;
    }
    return (__ldg(cu + lo) <= t && t < __ldg(cu + lo + 1)) ? lo : -1;
}

__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ int warp_sum_i32(int v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Fixed-order block sum of a double (blockDim.x a multiple of 32, <= 1024).
// Every thread returns the same total. `scratch` holds >= 32 doubles.
__device__ __forceinline__ double block_sum_f64(double v, double *scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_sum_f64(v);
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    double t = lane < nw ? scratch[lane] : 0.0;
    t = warp_sum_f64(t);
    return t;
}

__device__ __forceinline__ int block_sum_i32(int v, int *scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_sum_i32(v);
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    int t = lane < nw ? scratch[lane] : 0;
    return warp_sum_i32(t);
}

__device__ __forceinline__ void raise_status(uint32_t *status, rl_status code) {
    atomicOr(status, 1u << static_cast<int>(code));
}

// Invariant checks of the debug build (RL_LOSS_DEBUG_CHECKS, see build.py): a failed check
// raises RL_ERR_INTERNAL and the guarded access is skipped. In the normal build the check is
// `true` and compiles away.
#ifdef RL_LOSS_DEBUG_CHECKS
__device__ __forceinline__ bool debug_check_failed(uint32_t *status) {
    if (status) raise_status(status, RL_ERR_INTERNAL);  // the status word is optional for some entry points
    return false;
}
#define RLK_CHECK(status, cond) ((cond) ? true : ::rlk::debug_check_failed(status))
#else
#define RLK_CHECK(status, cond) true
#endif

// ---------------------------------------------------------------- kernel parameters

struct SeqPrepParams {
    const int32_t *cu_seqlens;
    const uint8_t *mask;
    const float *rewards_or_adv;
    int32_t num_seqs, num_tokens, group_size, adv_mode, std_unbiased, loss_norm;
    float adv_eps;
    float *seq_adv;      // workspace [S]
    float *seq_w;        // workspace [S] fp32 1/(S n_i)
    double *seq_w64;     // workspace [S] fp64 1/(S n_i)
    int32_t *seq_n;      // workspace [S]
    float *seq_adv_out;  // optional user output [S]
    uint32_t *status;
};

struct TokenPrepParams {
    const void *logits;  // row i holds token row0 + i
    int64_t ld_logits;
    const float *target_logit;  // [rows] z_y of row i, read instead of the logits (the projection path), else null
    int32_t row0, rows;  // tokens [row0, row0 + rows) are prepared
    int32_t logits_dtype;
    const int32_t *targets;
    const float *logp_old;
    const float *logp_infer;
    const uint8_t *mask;
    const int32_t *cu_seqlens;
    int32_t num_seqs, num_tokens, vocab;
    const float *seq_adv;
    const float *seq_w;
    const float *token_adv;  // [T] per-token advantages (RL_ADV_PER_TOKEN), else null
    LossConsts c;
    float4 *rec;     // workspace [T]
    uint32_t *meta;  // workspace [T]
    uint32_t *status;
};

struct RowParams {
    const void *logits;
    int64_t ld_logits;
    void *dlogits;
    int64_t ld_dlogits;
    const float4 *rec;
    const uint32_t *meta;
    const float *teacher;  // [T] log pi_teacher (RL_ADV_TEACHER_LOGP), else null
    int32_t num_tokens, vocab;
    LossConsts c;
    float *logp_out;     // optional
    float *entropy_out;
    uint8_t *flags_out;
    float *tok_obj;
    uint32_t *status;
    uint8_t *fix_rows;   // workspace [T], zero: rows whose entropy the fix kernel redoes
};

struct ReduceParams {
    const int32_t *cu_seqlens;
    int32_t num_seqs, num_tokens;
    const float *tok_obj;
    const float *entropy;
    const uint8_t *flags;
    const double *seq_w64;
    const int32_t *seq_n;
    double *seq_obj;      // workspace [S]
    double *seq_ent;      // workspace [S]
    int32_t *seq_cnt;     // workspace [S * 4]
    float *loss;
    double *loss_f64;
    int32_t *counts;
    float *mean_entropy;
    uint32_t *status;
};

cudaError_t launch_seg_prep(const SeqPrepParams &p, cudaStream_t stream);
// RL_NORM_PER_TOKEN: w_i = 1 / sum_j |y_j| (one block, fixed order); after seg_prep.
cudaError_t launch_seg_token_norm(const SeqPrepParams &p, cudaStream_t stream);
cudaError_t launch_token_prep(const TokenPrepParams &p, cudaStream_t stream);
cudaError_t launch_seg_reduce(const ReduceParams &p, cudaStream_t stream);
cudaError_t launch_final_reduce(const ReduceParams &p, cudaStream_t stream);

// The fused row kernel (one block per logits row).
cudaError_t launch_row_loss(const RowParams &p, int dtype, cudaStream_t stream);
// The entropy of the rows launch_row_loss marked in p.fix_rows (rows holding -inf logits).
cudaError_t launch_entropy_fix(const RowParams &p, int dtype, cudaStream_t stream);

}  // namespace rlk
