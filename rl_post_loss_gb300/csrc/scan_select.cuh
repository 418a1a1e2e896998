// Internal interface of the two kernels outside the loss path: the GAE scan
// (gae.cu) and the deterministic top-k (topk.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace rlk {

struct GaeParams {
    const int32_t *cu_seqlens;
    int32_t num_seqs, num_tokens;
    const float *rewards;      // [T]
    const float *values;       // [T]
    const uint8_t *mask;       // [T] nonzero = action token
    float gamma, gl;           // gamma and gamma * lambda, rounded to fp32 once
    float log2_gl_hi, log2_gl_lo;  // log2(gamma lambda) as an unevaluated fp32 sum
    double log2_gl;
    int32_t gl_kind;           // 0: 0 < gamma lambda < 1; 1: gamma lambda == 0; 2: gamma lambda == 1
    int32_t skip_observations;
    const int32_t *rollout_ids;  // [S] or null (no cross-trajectory discount)
    float *adv;                // [T]
    float *returns;            // [T] adv + V, or null
    void *workspace;           // gae_workspace_bytes(T), zeroed before the first launch
    int32_t vec;               // set by launch_gae: every array 16-byte aligned
    uint32_t *status;
    uint64_t wait_ns;          // bound on each wait for a neighbouring chunk's map (1 s)
    int32_t withhold_chunk;    // failure injection: this chunk never publishes its map (-1: none)
    // set by launch_gae: the first wave's blocks on an SM start stagger_ns apart (0: no stagger);
    // block b of that wave is taken to run in slot b / stagger_sms of its SM
    uint32_t stagger_ns;
    int32_t stagger_sms, stagger_slots;
};

// Row-wise deterministic top-k (see topk.cu).
struct TopkParams {
    const float *scores;     // [rows x ld], 16-byte aligned, ld % 4 == 0
    int64_t ld;
    const int32_t *lengths;  // [rows] valid scores per row, or null (all ld)
    int32_t rows, k;
    int32_t order_by_score;  // 1: (score desc, position asc); 0: position asc
    int32_t *out_idx;        // [rows x ldo]
    float *out_val;          // [rows x ldo] or null
    int64_t ldo;
    uint32_t *status;        // optional
};

int topk_max_k();
cudaError_t launch_topk(const TopkParams &p, cudaStream_t stream);

size_t gae_workspace_bytes(int64_t num_tokens);
cudaError_t launch_gae(GaeParams p, cudaStream_t stream);

}  // namespace rlk
