// Logits projection of one sequence chunk on the 5th-generation tensor cores,
// fused with the softmax-statistics epilogue of the loss:
//
//   Z = H_c W^T            H_c [M x K] bf16 (a chunk of hidden states), W [N x K] bf16 (LM head)
//   Z -> global (fp32, optional) and, per row and per 256-column tile, the
//   partial base-2 softmax statistics (max, sum 2^{z log2e - m}, sum 2^{...}(...)).
//
// This is the first GEMM of the sequence-chunked output projection + loss
// ("GLM-5: from Vibe Coding to Agentic Engineering", section 2.4.1,
// "Sequence-chunked output projection"): the statistics let the loss finish a
// row without a second pass over the full-vocabulary logits, and the logits of
// the whole sequence never exist at once.
//
// Kernel structure (persistent, one CTA per SM, 192 threads):
//   warp 0      TMA producer: 128-byte-swizzled K-major tiles of H_c (128 x 64)
//               and W (256 x 64) into a 4-stage shared-memory ring (mbarriers).
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M=128, N=256, K=16,
//               kind::f16 bf16 -> fp32) into one of two TMEM accumulators and
//               commits stage releases / accumulator completion to mbarriers.
//   warps 2..5  epilogue: each thread owns one row of the 128-row tile, reads
//               its 256 accumulator columns from TMEM (tcgen05.ld), updates the
//               row's statistics and stores the row's values.
// The two TMEM accumulators let the epilogue of tile i overlap the MMAs of
// tile i+1. Every wait is bounded; a timeout raises RL_ERR_TIMEOUT and the
// kernel stops waiting, so it always finishes.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "proj.cuh"
#include "ptx.cuh"

namespace rlk {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, NSTAGE = 4;
constexpr int kGemmThreads = 192;
constexpr uint32_t kStageA = BM * BK * 2;  // 16 KB
constexpr uint32_t kStageB = BN * BK * 2;  // 32 KB
constexpr uint32_t kTmemCols = 2 * BN;     // two fp32 accumulators of 128 x 256
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(BM, BN);

struct GemmSmem {
    // offsets from the 1024-aligned base
    static constexpr uint32_t a_off = 0;
    static constexpr uint32_t b_off = NSTAGE * kStageA;
    static constexpr uint32_t bar_off = b_off + NSTAGE * kStageB;
    // full[NSTAGE], empty[NSTAGE], accf[2], acce[2], done
    static constexpr uint32_t tmem_off = bar_off + 8 * (2 * NSTAGE + 5);
    static constexpr uint32_t total = tmem_off + 16;
};

__global__ void __launch_bounds__(kGemmThreads, 1)
    proj_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     ProjGemmParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // the swizzled tiles need 1024-byte alignment
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    unsigned char *smem = smem_raw + (sbase - raw);

    const uint32_t full0 = sbase + GemmSmem::bar_off;
    const uint32_t empty0 = full0 + 8 * NSTAGE;
    const uint32_t accf0 = empty0 + 8 * NSTAGE;
    const uint32_t acce0 = accf0 + 16;
    const uint32_t done_bar = acce0 + 16;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + GemmSmem::tmem_off);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tiles = (p.M + BM - 1) / BM, n_tiles = (p.N + BN - 1) / BN;
    const int k_blocks = (p.K + BK - 1) / BK;
    const int tiles = m_tiles * n_tiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            ptx::mbar_init(full0 + 8 * s, 1);
            ptx::mbar_init(empty0 + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(accf0 + 8 * a, 1);
            ptx::mbar_init(acce0 + 8 * a, 4);  // one arrival per epilogue warp
        }
        ptx::mbar_init(done_bar, 1);
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
    }
    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    bool timed_out = false;
    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
                const int m0 = (tile % m_tiles) * BM, n0 = (tile / m_tiles) * BN;
                for (int kb = 0; kb < k_blocks; ++kb, ++it) {
                    const uint32_t s = it % NSTAGE, ph = (it / NSTAGE) & 1u;
                    if (!timed_out && !ptx::mbar_wait(empty0 + 8 * s, ph ^ 1u)) timed_out = true;
                    ptx::mbar_arrive_expect_tx(full0 + 8 * s, kStageA + kStageB);
                    ptx::tma_load_2d(sbase + GemmSmem::a_off + s * kStageA, &tmA, kb * BK, m0, full0 + 8 * s);
                    ptx::tma_load_2d(sbase + GemmSmem::b_off + s * kStageB, &tmB, kb * BK, n0, full0 + 8 * s);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            uint32_t it = 0, tcount = 0;
            for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++tcount) {
                const uint32_t acc = tcount & 1u, aph = (tcount >> 1) & 1u;
                if (!timed_out && !ptx::mbar_wait(acce0 + 8 * acc, aph ^ 1u)) timed_out = true;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < k_blocks; ++kb, ++it) {
                    const uint32_t s = it % NSTAGE, ph = (it / NSTAGE) & 1u;
                    if (!timed_out && !ptx::mbar_wait(full0 + 8 * s, ph)) timed_out = true;
                    ptx::tc_fence_after();
                    const uint32_t a_addr = sbase + GemmSmem::a_off + s * kStageA;
                    const uint32_t b_addr = sbase + GemmSmem::b_off + s * kStageB;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t ad = ptx::smem_desc_kmajor_sw128(a_addr + kk * 32);
                        const uint64_t bd = ptx::smem_desc_kmajor_sw128(b_addr + kk * 32);
                        ptx::mma_bf16_ss(d_tmem, ad, bd, kIdesc, (kb > 0 || kk > 0) ? 1u : 0u);
                    }
                    ptx::mma_commit(empty0 + 8 * s);  // the stage is free once these MMAs have read it
                }
                ptx::mma_commit(accf0 + 8 * acc);  // accumulator complete
            }
            ptx::mma_commit(done_bar);  // every MMA of this CTA has completed
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int r_in_tile = q * 32 + lane;
        uint32_t tcount = 0;
        for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++tcount) {
            const int mt = tile % m_tiles, nt = tile / m_tiles;
            const int row = mt * BM + r_in_tile;
            const int n0 = nt * BN;
            const uint32_t acc = tcount & 1u, aph = (tcount >> 1) & 1u;
            if (!timed_out && !ptx::mbar_wait(accf0 + 8 * acc, aph)) timed_out = true;
            ptx::tc_fence_after();
            RowStats2 st = empty_stats();
            float *zrow = (p.z && row < p.M) ? p.z + (size_t)row * (size_t)p.ldz : nullptr;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN + c * 32, r);
                ptx::tmem_ld_wait();
                const int col0 = n0 + c * 32;
                const int nvalid = min(32, p.N - col0);
                if (nvalid <= 0) continue;
                float mv = -INFINITY;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j < nvalid) mv = fmaxf(mv, __uint_as_float(r[j]));
                const float mv2 = mv * kLog2e;
                if (mv2 > st.m2) {
                    if (st.m2 != -INFINITY) {
                        const float dm = st.m2 - mv2;
                        const float f = ex2_approx(dm);
                        st.u2 = f * fmaf(dm, st.s, st.u2);
                        st.s = f * st.s;
                    }
                    st.m2 = mv2;
                }
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    if (j < nvalid) {
                        const float d2 = fmaf(__uint_as_float(r[j]), kLog2e, -st.m2);
                        const float e = ex2_approx(d2);
                        st.s += e;
                        st.u2 = fmaf(e, d2, st.u2);
                    }
                }
                if (zrow) {
                    if (nvalid == 32 && (p.ldz & 3) == 0) {
                        float4 *dst = reinterpret_cast<float4 *>(zrow + col0);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                 __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < nvalid) zrow[col0 + j] = __uint_as_float(r[j]);
                    }
                }
            }
            if (p.stats && row < p.M) p.stats[(size_t)row * n_tiles + nt] = make_float4(st.m2, st.s, st.u2, 0.f);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(acce0 + 8 * acc);
        }
    }

    __syncthreads();
    if (warp == 0) {
        // every MMA has completed before the accumulators are released
        if (!ptx::mbar_wait(done_bar, 0, timed_out ? 100000000ull : 2000000000ull)) timed_out = true;
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
    if (timed_out) raise_status(p.status, RL_ERR_TIMEOUT);
}

// ------------------------------------------------------------------ host side

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
        cudaGetLastError();
    });
    return fn;
}

// 2-D bf16 tensor map over a row-major [rows x cols] matrix with row stride
// `ld` elements, boxes of box_rows x 64 columns, 128-byte swizzle.
bool make_tmap(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int64_t ld, uint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 2u};
    const cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

std::mutex g_gemm_mu;
int g_gemm_sms[64] = {};
bool g_gemm_attr[64] = {};

}  // namespace

int proj_gemm_tile_cols() { return BN; }

cudaError_t launch_proj_gemm(const void *A, int64_t lda, const void *B, int64_t ldb, const ProjGemmParams &p,
                             cudaStream_t stream) {
    if (p.M <= 0 || p.N <= 0) return cudaSuccess;
    if (p.K <= 0 || (lda * 2) % 16 != 0 || (ldb * 2) % 16 != 0 || (reinterpret_cast<uintptr_t>(A) & 15u) ||
        (reinterpret_cast<uintptr_t>(B) & 15u))
        return cudaErrorInvalidValue;
    CUtensorMap ta, tb;
    if (!make_tmap(&ta, A, p.M, p.K, lda, BM) || !make_tmap(&tb, B, p.N, p.K, ldb, BN)) return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int smem = (int)GemmSmem::total + 1024;
    int sms = 0;
    {
        std::lock_guard<std::mutex> lock(g_gemm_mu);
        if (dev < 64 && !g_gemm_attr[dev]) {
            e = cudaFuncSetAttribute(proj_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            cudaDeviceGetAttribute(&g_gemm_sms[dev], cudaDevAttrMultiProcessorCount, dev);
            g_gemm_attr[dev] = true;
        }
        sms = dev < 64 ? g_gemm_sms[dev] : 0;
    }
    if (sms <= 0) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int tiles = ((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN);
    const int grid = tiles < sms ? tiles : sms;
    proj_gemm_kernel<<<grid, kGemmThreads, smem, stream>>>(ta, tb, p);
    return cudaGetLastError();
}

}  // namespace rlk
