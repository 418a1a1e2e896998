// Internal interface of the fused projection path (sequence-chunked output
// projection + loss).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace rlk {

struct ProjGemmParams {
    int M, N, K;     // Z [M x N] = A [M x K] * B [N x K]^T
    float *z;        // optional fp32 output, row stride ldz
    int64_t ldz;
    float4 *stats;   // optional [M x ceil(N / 256)] partial row statistics (m2, s, u2, 0)
    uint32_t *status;
};

// Columns of one statistics tile of launch_proj_gemm (256).
int proj_gemm_tile_cols();

// tcgen05 GEMM with the statistics epilogue. A and B are bf16, row-major,
// K contiguous, 16-byte aligned with ld * 2 a multiple of 16.
cudaError_t launch_proj_gemm(const void *A, int64_t lda, const void *B, int64_t ldb, const ProjGemmParams &p,
                             cudaStream_t stream);

// One bf16 operand of a GEMM problem, row-major with row stride `ld`
// elements (16-byte aligned base, ld * 2 a multiple of 16). K-major: the
// operand's M (or N) index is the row and K the column; MN-major: K is the row
// and M (or N) the column.
struct GemmOperand {
    const void *base;
    int64_t ld;
    int mn_major;
};

// D [M x N] = A [M x K] B [K x N] (fp32 accumulation over K in a fixed order).
struct GemmProblem {
    enum Epi { kZStats = 0, kBf16 = 1, kF32 = 2, kProbStats = 3 };
    int M, N, K;
    GemmOperand a, b;
    int epi;         // kZStats: fp32 D (optional) + per-row, per-256-column softmax statistics;
                     // kProbStats: bf16 scaled probabilities 2^{z log2e - m} in D, the statistics,
                     //   each 64-column block's reference m and the target logits;
                     // kBf16: D rounded to bf16; kF32: D in fp32
    int accumulate;  // kF32: D += A B instead of D = A B
    int n_fastest;   // tile order of the problem (consecutive tiles of a CTA pair walk N, else M)
    void *d;
    int64_t ldd;     // elements
    float4 *stats;   // kZStats, kProbStats: [M x ceil(N / 256)]
    float4 *refs;    // kProbStats: [M x ceil(N / 256)], the references of a tile's four 64-column blocks
    const int32_t *targets;  // kProbStats: [M] target column per row
    float *target_logit;     // kProbStats: [M] written for rows whose target is in [0, N)
};

// One launch over one or two problems. With two, the tiles of the first are
// strided over the CTA pairs and those of the second follow in strided rounds
// that the pairs with one more tile of the first join later.
cudaError_t launch_gemm_problems(const GemmProblem *probs, int nprob, uint32_t *status, cudaStream_t stream);

struct ProjRowParams {
    void *probs;          // [rows x ldp] bf16: in, the scaled probabilities of the chunk; out, dZ (in place)
    int64_t ldp;
    const float4 *stats;  // [rows x n_tiles]
    const float4 *refs;   // [rows x n_tiles]: base-2 reference of each 64-column block
    int32_t n_tiles;
    int32_t row0;        // token index of the chunk's first row
    int32_t rows, vocab;
    const float4 *rec;   // per-token records (indexed by token)
    const uint32_t *meta;
    const float *teacher; // [T] log pi_teacher (RL_ADV_TEACHER_LOGP), else null
    LossConsts c;
    float *logp_out;     // optional, indexed by token
    float *entropy_out;
    uint8_t *flags_out;
    float *tok_obj;
    uint32_t *status;
};

// Per row of the chunk: merge the partial statistics in tile order, finish the
// token objective, write dZ = g (onehot - softmax(z)) as bf16.
cudaError_t launch_proj_rows(const ProjRowParams &p, cudaStream_t stream);

}  // namespace rlk
