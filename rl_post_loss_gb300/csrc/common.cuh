// Shared device helpers of the fused GRPO + IcePop loss kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "rl_loss.h"

namespace rlk {

constexpr float kLog2e = 1.4426950408889634f;

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
};

struct TokenResult {
    float logp;   // z_y - logZ (NaN for a bad target)
    float g;      // dL/dlogp_t
    float obj;    // m * pop * min(r A, clip(r) A)
    uint32_t flags;
};

// Per-token part of Eq. (1) of the GLM-5 report page, section 3.2: rho, pop,
// r, the clipped min and dL/dlogp. `w` is 1/(S |y_i|) of the token's response.
__device__ __forceinline__ TokenResult token_objective(float zy, float logZ, bool target_ok, float logp_old,
                                                       float logp_infer, bool m, float A, float w,
                                                       const LossConsts &c) {
    TokenResult r;
    const float d = __fsub_rn(logp_old, logp_infer);  // ln rho, one fp32 subtraction
    const bool in_bounds = (-c.ln_beta <= d) && (d <= c.ln_beta);
    r.logp = target_ok ? __fsub_rn(zy, logZ) : __int_as_float(0x7fc00000);
    const float e = __fsub_rn(r.logp, logp_old);      // ln r, one fp32 subtraction
    const bool clip = target_ok && ((A > 0.f && e > c.clip_hi) || (A < 0.f && e < c.clip_lo));
    r.flags = (in_bounds ? RL_FLAG_POP_IN_BOUNDS : 0u) | (clip ? RL_FLAG_CLIP_ACTIVE : 0u) |
              (m ? 0u : RL_FLAG_MASKED) | (target_ok ? 0u : RL_FLAG_BAD_TARGET);
    r.obj = 0.f;
    r.g = 0.f;
    if (m && target_ok && in_bounds) {
        const float pop = c.pop_indicator ? 1.f : expf(d);
        const float ratio = expf(e);
        const float branch = clip ? (A > 0.f ? c.one_plus_eps_high : c.one_minus_eps_low) : ratio;
        r.obj = pop * A * branch;
        r.g = clip ? 0.f : -w * pop * A * ratio;
    }
    return r;
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

// Running softmax statistics of part of a row: M = max, S = sum e^{z-M},
// U = sum e^{z-M} (z-M).
struct RowStats {
    float m, s, u;
};

// Merge two partial statistics. Symmetric in its arguments (so a butterfly
// gives every lane bit-identical results) and exact for empty parts.
__device__ __forceinline__ RowStats merge_stats(RowStats a, RowStats b) {
    const float M = fmaxf(a.m, b.m);
    if (M == -INFINITY) return RowStats{M, 0.f, 0.f};
    const float da = a.m - M, db = b.m - M;
    const float fa = (a.m == -INFINITY) ? 0.f : ex2_approx(da * kLog2e);
    const float fb = (b.m == -INFINITY) ? 0.f : ex2_approx(db * kLog2e);
    // explicit _rn operations: no FMA contraction, so merge(a, b) == merge(b, a) bitwise
    const float ua = (a.m == -INFINITY) ? 0.f : __fmul_rn(fa, fmaf(da, a.s, a.u));
    const float ub = (b.m == -INFINITY) ? 0.f : __fmul_rn(fb, fmaf(db, b.s, b.u));
    return RowStats{M, __fadd_rn(__fmul_rn(a.s, fa), __fmul_rn(b.s, fb)), __fadd_rn(ua, ub)};
}

__device__ __forceinline__ RowStats warp_merge_stats(RowStats r) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        RowStats o{__shfl_xor_sync(0xffffffffu, r.m, off), __shfl_xor_sync(0xffffffffu, r.s, off),
                   __shfl_xor_sync(0xffffffffu, r.u, off)};
        r = merge_stats(r, o);
    }
    return r;
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

// ---------------------------------------------------------------- kernel parameters

struct SeqPrepParams {
    const int32_t *cu_seqlens;
    const uint8_t *mask;
    const float *rewards_or_adv;
    int32_t num_seqs, num_tokens, group_size, adv_mode, std_unbiased;
    float adv_eps;
    float *seq_adv;      // workspace [S]
    float *seq_w;        // workspace [S] fp32 1/(S n_i)
    double *seq_w64;     // workspace [S] fp64 1/(S n_i)
    int32_t *seq_n;      // workspace [S]
    float *seq_adv_out;  // optional user output [S]
    uint32_t *status;
};

struct RowParams {
    const void *logits;
    int64_t ld_logits;
    void *dlogits;
    int64_t ld_dlogits;
    const int32_t *targets;
    const float *logp_old;
    const float *logp_infer;
    const uint8_t *mask;
    const int32_t *cu_seqlens;
    int32_t num_seqs, num_tokens, vocab;
    const float *seq_adv;
    const float *seq_w;
    LossConsts c;
    float *logp_out;
    float *entropy_out;
    uint8_t *flags_out;
    float *tok_obj;
    uint32_t *status;
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

__device__ __forceinline__ void raise_status(uint32_t *status, rl_status code) {
    atomicOr(status, 1u << static_cast<int>(code));
}

cudaError_t launch_seg_prep(const SeqPrepParams &p, cudaStream_t stream);
cudaError_t launch_row_loss(const RowParams &p, int dtype, cudaStream_t stream);
cudaError_t launch_seg_reduce(const ReduceParams &p, cudaStream_t stream);
cudaError_t launch_final_reduce(const ReduceParams &p, cudaStream_t stream);

}  // namespace rlk
