// The three GEMMs of the sequence-chunked output projection + loss, on the
// 5th-generation tensor cores ("GLM-5: from Vibe Coding to Agentic
// Engineering", section 2.4.1, "Sequence-chunked output projection"): per
// chunk of rows, the forward projection and both products of its backward.
//
//   forward   Z_c  = H_c W^T      A = H_c [m x H] (K-major), B = W [V x H] (K-major)
//             epilogue: Z_c in fp32 and, per row and per 256-column tile, the
//             partial base-2 softmax statistics (max, sum 2^{z log2e - m},
//             sum 2^{...}(...)), so the loss can finish a row without another
//             pass over the full-vocabulary logits
//   backward  dH_c = dZ_c W       A = dZ_c [m x V] (K-major), B = W [V x H] (MN-major), bf16 out
//             dW  (+)= dZ_c^T H_c A = dZ_c (MN-major), B = H_c [m x H] (MN-major), fp32 out,
//             stored by the first chunk and added into by the later ones
//
// The two backward products of a chunk run in one launch over one combined
// tile list: the long dH tiles (K = V) go first, strided over the CTA pairs,
// and the short dW tiles (K = m) follow in contiguous ranges sized so that
// every pair gets about the same number of k-blocks. Every output tile is
// owned by one pair and accumulated over K in a fixed order, and dW is added
// into chunk after chunk in chunk order: the results do not depend on
// scheduling and repeat bit for bit.
//
// Kernel structure (persistent; clusters of 2 CTAs, one CTA per SM, 192
// threads). A pair of CTAs computes a 256 x 256 tile with tcgen05.mma
// cta_group::2 (M = 256, N = 256, K = 16, kind::f16, bf16 -> fp32): each CTA
// stages 128 rows of A and 128 columns of B per k-block, and holds 128 rows of
// the accumulator in its own TMEM.
//   warp 0      TMA producer (both CTAs): 128-byte-swizzled tiles into a
//               6-stage ring; the loads of both CTAs complete on the even
//               CTA's "full" mbarrier.
//   warp 1      MMA issuer (one thread of the even CTA): 4 MMAs per k-block
//               into one of two TMEM accumulators; each stage's release and
//               each accumulator's completion are committed to the mbarriers
//               of both CTAs.
//   warps 2..5  epilogue (both CTAs): each thread owns one accumulator row,
//               reads it from TMEM (tcgen05.ld) and applies the problem's
//               epilogue; the warps then free the accumulator on the even
//               CTA's "empty" mbarrier.
// Every wait is bounded; a timeout raises RL_ERR_TIMEOUT and the kernel
// stops waiting, so it always finishes.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "proj.cuh"
#include "ptx.cuh"

namespace rlk {

namespace {

constexpr int BK = 64;              // K per stage (one 128-byte swizzle row of bf16)
constexpr int kThreads = 192;
constexpr int kTileN = 256;         // accumulator columns = N of one MMA
constexpr int kRowsCta = 128;       // accumulator rows per CTA (TMEM lanes)
constexpr int kTileM = 2 * kRowsCta;
constexpr int kBnCta = kTileN / 2;  // B columns staged per CTA
constexpr uint32_t kStageA = kRowsCta * BK * 2;  // 16 KB
constexpr uint32_t kStageB = kBnCta * BK * 2;    // 16 KB
constexpr uint32_t kMnBlock = 64 * BK * 2;       // one 64 (M/N) x 64 (K) MN-major box: 8 KB
constexpr int NSTAGE = 6;
constexpr uint32_t kTmemCols = 2 * kTileN;       // two fp32 accumulators of 128 x 256 per CTA
constexpr uint32_t kLboMn = kMnBlock;            // MN-major: distance between 64-element M/N blocks
constexpr uint32_t kSbo = 1024;                  // distance between 8-row (K-major) / 8-k (MN-major) atoms

struct Smem {
    static constexpr uint32_t a_off = 0;
    static constexpr uint32_t b_off = NSTAGE * kStageA;
    static constexpr uint32_t bar_off = b_off + NSTAGE * kStageB;
    // full[NSTAGE], empty[NSTAGE], accf[2], acce[2], done
    static constexpr uint32_t tmem_off = bar_off + 8 * (2 * NSTAGE + 5);
    static constexpr uint32_t total = tmem_off + 16;
};

enum { kEpiStats = 0, kEpiBf16 = 1, kEpiF32 = 2 };

struct TcProblem {
    int M, N, K;
    int a_mn, b_mn;     // operand stored MN-major (else K-major)
    int epi;            // kEpiStats / kEpiBf16 / kEpiF32
    int accumulate;     // kEpiF32: D += A B (else D = A B)
    int n_fastest;      // tile order: consecutive tiles walk N (else M)
    int tiles_m, tiles_n, k_blocks;
    int tiles_nc, tiles;  // cluster tiles: tiles_m x tiles_nc, each kTileM x (CP x kTileN)
    void *d;            // output, row stride ldd elements (fp32 or bf16 by epi)
    int64_t ldd;
    float4 *stats;      // kEpiStats: [M x tiles_n] partial row statistics (optional)
};

struct TcParams {
    TcProblem prob[2];
    int nprob;
    // problem 1 is dealt out in rounds of consecutive tiles: the clusters with
    // one more tile of problem 0 (the first tiles0 % clusters) join `p1_delay`
    // rounds after the others, the time their extra tile takes
    int p1_delay;
    uint32_t *status;
};

struct TcMaps {
    CUtensorMap a[2], b[2];
};

// The tiles of a cluster, in order: its strided share of problem 0, then its
// share of problem 1. Clusters running at the same time work on neighbouring
// tiles of the same problem, so their operands are shared through L2 (a
// contiguous range per cluster would spread them over the whole problem).
// Every CTA of the cluster walks the same list.
struct ClusterTiles {
    int cl, ncl, n0, r, t1, delay;
    __device__ ClusterTiles(const TcParams &p, int cl_, int ncl_) : cl(cl_), ncl(ncl_) {
        const int t0 = p.prob[0].tiles;
        n0 = cl < t0 ? (t0 - 1 - cl) / ncl + 1 : 0;
        r = t0 % ncl;
        t1 = p.nprob > 1 ? p.prob[1].tiles : 0;
        delay = p.p1_delay;
    }
    // problem index and cluster-tile index of the i-th tile of the cluster;
    // false past its last tile
    __device__ bool at(int i, int &prob, int &tile) const {
        if (i < n0) {
            prob = 0;
            tile = cl + i * ncl;
            return true;
        }
        const int j = i - n0;
        int t;
        if (cl < r)  // one tile of problem 0 more: starts `delay` rounds late
            t = delay * (ncl - r) + j * ncl + cl;
        else if (j < delay)  // rounds shared by the other clusters only
            t = j * (ncl - r) + (cl - r);
        else
            t = delay * (ncl - r) + (j - delay) * ncl + cl;
        if (t >= t1) return false;
        prob = 1;
        tile = t;
        return true;
    }
};

// Origin of pair `pr`'s 256 x 256 tile within cluster tile `tile` (the pairs
// of a cluster share the rows m0 and take consecutive 256-column tiles), and
// that tile's 256-column index `nt`.
template <int CP>
__device__ __forceinline__ void tile_origin(const TcProblem &q, int tile, int pr, int &m0, int &n0, int &nt) {
    int mt, ntc;
    if (q.n_fastest) {
        mt = tile / q.tiles_nc;
        ntc = tile % q.tiles_nc;
    } else {
        mt = tile % q.tiles_m;
        ntc = tile / q.tiles_m;
    }
    m0 = mt * kTileM;
    nt = ntc * CP + pr;
    n0 = nt * kTileN;
}

// ---------------------------------------------------------------- epilogues (one accumulator row per thread)

__device__ __forceinline__ void epi_stats(const TcProblem &q, uint32_t tbase, int row, int n0, int nt) {
    RowStats2 st = empty_stats();
    float *zrow = (q.d && row < q.M) ? reinterpret_cast<float *>(q.d) + (size_t)row * (size_t)q.ldd : nullptr;
#pragma unroll 1
    for (int c = 0; c < kTileN / 32; ++c) {
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(tbase + c * 32, r);
        ptx::tmem_ld_wait();
        const int col0 = n0 + c * 32;
        const int nvalid = min(32, q.N - col0);
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
            if (nvalid == 32 && (q.ldd & 3) == 0) {
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
    if (q.stats && row < q.M) q.stats[(size_t)row * q.tiles_n + nt] = make_float4(st.m2, st.s, st.u2, 0.f);
}

__device__ __forceinline__ void epi_bf16(const TcProblem &q, uint32_t tbase, int row, int n0) {
    __nv_bfloat16 *drow =
        row < q.M ? reinterpret_cast<__nv_bfloat16 *>(q.d) + (size_t)row * (size_t)q.ldd : nullptr;
#pragma unroll 1
    for (int c = 0; c < kTileN / 32; ++c) {
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(tbase + c * 32, r);
        ptx::tmem_ld_wait();
        const int col0 = n0 + c * 32;
        const int nvalid = min(32, q.N - col0);
        if (nvalid <= 0 || !drow) continue;
        if (nvalid == 32 && (q.ldd & 7) == 0) {
            uint4 *dst = reinterpret_cast<uint4 *>(drow + col0);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                dst[j] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * j]), __uint_as_float(r[8 * j + 1])),
                                    pack_bf16x2(__uint_as_float(r[8 * j + 2]), __uint_as_float(r[8 * j + 3])),
                                    pack_bf16x2(__uint_as_float(r[8 * j + 4]), __uint_as_float(r[8 * j + 5])),
                                    pack_bf16x2(__uint_as_float(r[8 * j + 6]), __uint_as_float(r[8 * j + 7])));
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < nvalid) drow[col0 + j] = __float2bfloat16_rn(__uint_as_float(r[j]));
        }
    }
}

__device__ __forceinline__ void epi_f32(const TcProblem &q, uint32_t tbase, int row, int n0) {
    float *drow = row < q.M ? reinterpret_cast<float *>(q.d) + (size_t)row * (size_t)q.ldd : nullptr;
#pragma unroll 1
    for (int c = 0; c < kTileN / 32; ++c) {
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(tbase + c * 32, r);
        const int col0 = n0 + c * 32;
        const int nvalid = min(32, q.N - col0);
        const bool vec = nvalid == 32 && (q.ldd & 3) == 0;
        float4 old[8];
        if (drow && vec && q.accumulate) {  // issued before the TMEM load completes
            const float4 *src = reinterpret_cast<const float4 *>(drow + col0);
#pragma unroll
            for (int j = 0; j < 8; ++j) old[j] = __ldcs(src + j);
        }
        ptx::tmem_ld_wait();
        if (nvalid <= 0 || !drow) continue;
        if (vec) {
            float4 *dst = reinterpret_cast<float4 *>(drow + col0);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float4 v = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                       __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                if (q.accumulate) {
                    v.x = old[j].x + v.x;
                    v.y = old[j].y + v.y;
                    v.z = old[j].z + v.z;
                    v.w = old[j].w + v.w;
                }
                __stcs(dst + j, v);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < nvalid) drow[col0 + j] = (q.accumulate ? drow[col0 + j] : 0.f) + __uint_as_float(r[j]);
        }
    }
}

// ---------------------------------------------------------------- the kernel

// CP: CTA pairs per cluster. With CP = 2 the two pairs of a cluster compute
// horizontally adjacent tiles that share A: each CTA loads half of its A rows
// and multicasts them to the matching CTA of the other pair, so every stage's
// A arrives once from L2 for both pairs.
template <int CP>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ TcMaps maps, const __grid_constant__ TcParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // the swizzled tiles need 1024-byte alignment (the same offset in every CTA of the cluster)
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    unsigned char *smem = smem_raw + (sbase - raw);

    const uint32_t full0 = sbase + Smem::bar_off;
    const uint32_t empty0 = full0 + 8 * NSTAGE;
    const uint32_t accf0 = empty0 + 8 * NSTAGE;
    const uint32_t acce0 = accf0 + 16;
    const uint32_t done_bar = acce0 + 16;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Smem::tmem_off);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const uint32_t half = rank & 1u;        // 0: the pair's MMA issuer
    const int pr = (int)(rank >> 1);         // pair within the cluster
    const uint32_t leader = rank & ~1u;      // the even CTA of this pair
    const uint16_t pair_mask = (uint16_t)(3u << (2 * pr));
    const uint16_t cluster_mask = (uint16_t)((1u << (2 * CP)) - 1u);
    const int cl = blockIdx.x / (2 * CP), ncl = gridDim.x / (2 * CP);
    const ClusterTiles tiles(p, cl, ncl);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            ptx::mbar_init(full0 + 8 * s, 1);
            ptx::mbar_init(empty0 + 8 * s, CP);  // one commit per pair of the cluster
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(accf0 + 8 * a, 1);
            ptx::mbar_init(acce0 + 8 * a, 8);  // one arrival per epilogue warp of the pair
        }
        ptx::mbar_init(done_bar, 1);
        ptx::fence_mbar_init();
        for (int i = 0; i < p.nprob; ++i) {
            ptx::prefetch_tmap(&maps.a[i]);
            ptx::prefetch_tmap(&maps.b[i]);
        }
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), kTmemCols);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();  // every CTA's barriers are initialised before any other signals them
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    bool timed_out = false;
    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            const uint32_t full_leader0 = ptx::mapa_shared(full0, leader);
            const uint16_t a_mask = (uint16_t)((1u << rank) | (1u << (rank ^ 2u)));
            uint32_t it = 0;
            int prob, tile;
            for (int i = 0; tiles.at(i, prob, tile); ++i) {
                int m0, n0, nt;
                const TcProblem &q = p.prob[prob];
                tile_origin<CP>(q, tile, pr, m0, n0, nt);
                const void *am = &maps.a[prob];
                const void *bm = &maps.b[prob];
                const int ma = m0 + (int)half * kRowsCta, nb = n0 + (int)half * kBnCta;
                for (int kb = 0; kb < q.k_blocks; ++kb, ++it) {
                    const uint32_t s = it % NSTAGE, ph = (it / NSTAGE) & 1u;
                    if (!timed_out && !ptx::mbar_wait(empty0 + 8 * s, ph ^ 1u)) timed_out = true;
                    const uint32_t fb = full_leader0 + 8 * s;
                    if (half == 0) ptx::mbar_arrive_expect_tx(full0 + 8 * s, 2 * (kStageA + kStageB));
                    const uint32_t a_dst = sbase + Smem::a_off + s * kStageA;
                    const uint32_t b_dst = sbase + Smem::b_off + s * kStageB;
                    const int k0 = kb * BK;
                    if (CP == 1) {
                        if (q.a_mn) {
                            ptx::tma_load_2d_pair(a_dst, am, ma, k0, fb);
                            ptx::tma_load_2d_pair(a_dst + kMnBlock, am, ma + 64, k0, fb);
                        } else {
                            ptx::tma_load_2d_pair(a_dst, am, k0, ma, fb);
                        }
                    } else {
                        // this CTA's 64-row (or 64-column) half of the A block, into both pairs
                        const uint32_t dst = a_dst + (uint32_t)pr * kMnBlock;
                        if (q.a_mn)
                            ptx::tma_load_2d_pair_mc(dst, am, ma + 64 * pr, k0, fb, a_mask);
                        else
                            ptx::tma_load_2d_pair_mc(dst, am, k0, ma + 64 * pr, fb, a_mask);
                    }
                    if (q.b_mn) {
                        ptx::tma_load_2d_pair(b_dst, bm, nb, k0, fb);
                        ptx::tma_load_2d_pair(b_dst + kMnBlock, bm, nb + 64, k0, fb);
                    } else {
                        ptx::tma_load_2d_pair(b_dst, bm, k0, nb, fb);
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer (even CTA of each pair)
        if (half == 0 && lane == 0) {
            uint32_t it = 0;
            int prob, tile;
            for (int i = 0; tiles.at(i, prob, tile); ++i) {
                const TcProblem &q = p.prob[prob];
                const uint32_t idesc = ptx::idesc_bf16_f32_major(kTileM, kTileN, q.a_mn, q.b_mn);
                const uint32_t a_step = q.a_mn ? 16 * 128 : 32, b_step = q.b_mn ? 16 * 128 : 32;
                const uint32_t a_lbo = q.a_mn ? kLboMn : 16, b_lbo = q.b_mn ? kLboMn : 16;
                const uint32_t acc = (uint32_t)i & 1u, aph = ((uint32_t)i >> 1) & 1u;
                if (!timed_out && !ptx::mbar_wait(acce0 + 8 * acc, aph ^ 1u)) timed_out = true;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * kTileN;
                for (int kb = 0; kb < q.k_blocks; ++kb, ++it) {
                    const uint32_t s = it % NSTAGE, ph = (it / NSTAGE) & 1u;
                    if (!timed_out && !ptx::mbar_wait(full0 + 8 * s, ph)) timed_out = true;
                    ptx::tc_fence_after();
                    const uint32_t a_addr = sbase + Smem::a_off + s * kStageA;
                    const uint32_t b_addr = sbase + Smem::b_off + s * kStageB;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t ad = ptx::smem_desc_sw128(a_addr + kk * a_step, a_lbo, kSbo);
                        const uint64_t bd = ptx::smem_desc_sw128(b_addr + kk * b_step, b_lbo, kSbo);
                        ptx::mma_bf16_ss_pair(d_tmem, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                    }
                    // the stage is free in every CTA of the cluster once both pairs have read it
                    ptx::mma_commit_pair(empty0 + 8 * s, cluster_mask);
                }
                ptx::mma_commit_pair(accf0 + 8 * acc, pair_mask);  // accumulator complete in both CTAs
            }
            ptx::mma_commit_pair(done_bar, pair_mask);  // every MMA of this pair has completed
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- epilogue (every CTA)
        const int qd = warp & 3;  // TMEM lane quarter this warp may access
        const int r_local = qd * 32 + lane;
        const uint32_t acce_leader0 = ptx::mapa_shared(acce0, leader);
        int prob, tile;
        for (int i = 0; tiles.at(i, prob, tile); ++i) {
            int m0, n0, nt;
            const TcProblem &q = p.prob[prob];
            tile_origin<CP>(q, tile, pr, m0, n0, nt);
            const int row = m0 + (int)half * kRowsCta + r_local;
            const uint32_t acc = (uint32_t)i & 1u, aph = ((uint32_t)i >> 1) & 1u;
            if (!timed_out && !ptx::mbar_wait(accf0 + 8 * acc, aph)) timed_out = true;
            ptx::tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(qd * 32) << 16) + acc * kTileN;
            if (n0 >= q.N) {
                // the second pair's tile past the last column of an odd column count: nothing to write
            } else if (q.epi == kEpiStats)
                epi_stats(q, tbase, row, n0, nt);
            else if (q.epi == kEpiBf16)
                epi_bf16(q, tbase, row, n0);
            else
                epi_f32(q, tbase, row, n0);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster(acce_leader0 + 8 * acc);
        }
    }

    ptx::tc_fence_before();
    ptx::cluster_sync();  // no CTA leaves while another may still signal it or write its shared memory
    ptx::tc_fence_after();
    if (warp == 1) {
        // every MMA of the pair has completed before the accumulators are released
        if (!ptx::mbar_wait(done_bar, 0, timed_out ? 100000000ull : 2000000000ull)) timed_out = true;
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
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
// `ld` elements: boxes of box_rows x 64 columns, 128-byte swizzle. Out-of-range
// parts of a box read as zero.
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

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tensor maps of one operand: K-major [outer x K] (boxes of `k_rows` outer
// rows x 64 K) or MN-major [K x outer] (boxes of 64 k rows x 64 outer elements).
bool operand_map(CUtensorMap *m, const GemmOperand &o, int64_t outer, int64_t K, uint32_t k_rows) {
    if (!o.base || !aligned16(o.base) || (o.ld * 2) % 16 != 0) return false;
    if (o.mn_major) {
        if (o.ld < outer) return false;
        return make_tmap(m, o.base, K, outer, o.ld, 64);
    }
    if (o.ld < K) return false;
    return make_tmap(m, o.base, outer, K, o.ld, k_rows);
}

// Cluster shape: CTA pairs per cluster (2: the pairs share A by multicast).
// Measured on the case-4 chunk GEMMs: a cluster of 4 CTAs leaves 8 of the 152
// SMs idle (36 clusters resident) and the multicast saves little, since each
// SM's shared-memory fill rate, not L2, limits the loads; one pair it is.
constexpr int kPairsPerCluster = 1;
constexpr int kClusterCtas = 2 * kPairsPerCluster;
const auto kKernel = tc_gemm_kernel<kPairsPerCluster>;

std::mutex g_mu;
int g_clusters[64] = {};
bool g_attr[64] = {};

cudaLaunchConfig_t cluster_config(int clusters, int smem, cudaStream_t stream, cudaLaunchAttribute *attr) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kClusterCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kClusterCtas * clusters, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

cudaError_t launch(const GemmProblem *probs, int nprob, uint32_t *status, cudaStream_t stream) {
    constexpr int CP = kPairsPerCluster;
    TcMaps maps;
    TcParams p{};
    p.nprob = nprob;
    p.status = status;
    for (int i = 0; i < nprob; ++i) {
        const GemmProblem &g = probs[i];
        if (g.M <= 0 || g.N <= 0 || g.K <= 0) return cudaErrorInvalidValue;
        // with CP = 2 each CTA loads 64 of its 128 A rows (the other pair loads the rest)
        if (!operand_map(&maps.a[i], g.a, g.M, g.K, CP == 1 ? kRowsCta : 64) ||
            !operand_map(&maps.b[i], g.b, g.N, g.K, kBnCta))
            return cudaErrorInvalidValue;
        if (!g.d && g.epi != GemmProblem::kZStats) return cudaErrorInvalidValue;
        TcProblem &q = p.prob[i];
        q.M = g.M;
        q.N = g.N;
        q.K = g.K;
        q.a_mn = g.a.mn_major;
        q.b_mn = g.b.mn_major;
        q.epi = g.epi == GemmProblem::kZStats ? kEpiStats : (g.epi == GemmProblem::kBf16 ? kEpiBf16 : kEpiF32);
        q.accumulate = g.accumulate;
        q.n_fastest = g.n_fastest;
        q.tiles_m = (g.M + kTileM - 1) / kTileM;
        q.tiles_n = (g.N + kTileN - 1) / kTileN;
        q.k_blocks = (g.K + BK - 1) / BK;
        q.tiles_nc = (q.tiles_n + CP - 1) / CP;
        q.tiles = q.tiles_m * q.tiles_nc;
        q.d = g.d;
        q.ldd = g.ldd;
        q.stats = g.stats;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int smem = (int)Smem::total + 1024;
    int max_clusters = 0;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (dev < 64 && !g_attr[dev]) {
            e = cudaFuncSetAttribute(kKernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            cudaLaunchAttribute oa[1];
            cudaLaunchConfig_t oc = cluster_config(1, smem, 0, oa);
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, kKernel, &oc) != cudaSuccess || clusters <= 0) {
                cudaGetLastError();
                int sms = 0;
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
                clusters = sms / kClusterCtas;
            }
            g_clusters[dev] = clusters;
            g_attr[dev] = true;
        }
        max_clusters = dev < 64 ? g_clusters[dev] : 0;
    }
    if (max_clusters <= 0) {
        int sms = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        max_clusters = std::max(1, sms / kClusterCtas);
    }
    int64_t all_tiles = 0;
    for (int i = 0; i < nprob; ++i) all_tiles += p.prob[i].tiles;
    const int ncl = (int)std::min<int64_t>(all_tiles, max_clusters);
    if (nprob > 1)  // one problem-0 tile, in problem-1 tiles
        p.p1_delay = (p.prob[0].k_blocks + p.prob[1].k_blocks / 2) / p.prob[1].k_blocks;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = cluster_config(ncl, smem, stream, attr);
    e = cudaLaunchKernelEx(&cfg, kKernel, maps, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

int proj_gemm_tile_cols() { return kTileN; }

cudaError_t launch_proj_gemm(const void *A, int64_t lda, const void *B, int64_t ldb, const ProjGemmParams &p,
                             cudaStream_t stream) {
    if (p.M <= 0 || p.N <= 0) return cudaSuccess;
    GemmProblem g{};
    g.M = p.M;
    g.N = p.N;
    g.K = p.K;
    g.a = GemmOperand{A, lda, 0};
    g.b = GemmOperand{B, ldb, 0};
    g.epi = GemmProblem::kZStats;
    g.n_fastest = 0;  // pairs running at once share the LM-head tiles through L2
    g.d = p.z;
    g.ldd = p.ldz;
    g.stats = p.stats;
    return launch(&g, 1, p.status, stream);
}

cudaError_t launch_gemm_problems(const GemmProblem *probs, int nprob, uint32_t *status, cudaStream_t stream) {
    if (nprob < 1 || nprob > 2) return cudaErrorInvalidValue;
    return launch(probs, nprob, status, stream);
}

}  // namespace rlk
