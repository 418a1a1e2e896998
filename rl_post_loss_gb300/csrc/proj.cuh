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

struct ProjRowParams {
    const float *z;      // [rows x ldz] fp32 logits of the chunk
    int64_t ldz;
    const float4 *stats; // [rows x n_tiles]
    int32_t n_tiles;
    void *dz;            // [rows x lddz] bf16 dL/dlogits of the chunk
    int64_t lddz;
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
