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
// and the short dW tiles (K = m) follow in strided rounds that the pairs with
// one more dH tile join later, so every pair gets about the same number of
// k-blocks and the pairs running at once share operands through L2. Every
// output tile is owned by one pair and accumulated over K in a fixed order,
// and dW is added into chunk after chunk in chunk order (one addend per
// element per launch): the results do not depend on scheduling and repeat
// bit for bit.
//
// Kernel structure (persistent; clusters of 2 CTAs, one CTA per SM, 192
// threads). A pair of CTAs computes a 256 x 512 tile as two 256-column
// halves of tcgen05.mma cta_group::2 (M = 256, N = 256, K = 16, kind::f16,
// bf16 -> fp32): each CTA stages 128 rows of A and 2 x 128 columns of B per
// k-block, and holds 128 rows x 512 columns of the accumulator (all of its
// TMEM).
//   warp 0      TMA producer (both CTAs): 128-byte-swizzled tiles into a
//               4-stage ring; the loads of both CTAs complete on the even
//               CTA's "full" mbarrier.
//   warp 1      MMA issuer (one thread of the even CTA): 8 MMAs per k-block;
//               each stage's release and the accumulator's completion are
//               committed to the mbarriers of both CTAs. A new tile's MMAs
//               on a half wait until the epilogue has drained that half.
//   warps 2..5  epilogue (both CTAs): each thread owns one accumulator row and
//               reads it from TMEM (tcgen05.ld); each warp stages 32-row
//               blocks in shared memory and one thread writes them out with a
//               bulk tensor store (or reduce-add, for dW), so the epilogue
//               issues no global loads.
// Every wait is bounded; a timeout raises RL_ERR_TIMEOUT and the kernel
// stops waiting, so it always finishes.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "proj.cuh"
#include "ptx.cuh"
#include "tmap.cuh"

namespace rlk {

namespace {

constexpr int BK = 64;              // K per stage (one 128-byte swizzle row of bf16)
constexpr int kThreads = 192;
constexpr int kTileN = 256;         // N of one MMA = columns of one accumulator half
constexpr int kRowsCta = 128;       // accumulator rows per CTA (TMEM lanes)
constexpr int kTileM = 2 * kRowsCta;
constexpr int kBnCta = kTileN / 2;  // B columns of one half staged per CTA
constexpr uint32_t kStageA = kRowsCta * BK * 2;  // 16 KB
constexpr uint32_t kHalfB = kBnCta * BK * 2;     // 16 KB per half
constexpr uint32_t kMnBlock = 64 * BK * 2;       // one 64 (M/N) x 64 (K) MN-major box: 8 KB
constexpr uint32_t kTmemCols = 512;              // all of TMEM: 128 lanes x 512 fp32 columns
constexpr uint32_t kLboMn = kMnBlock;            // MN-major: distance between 64-element M/N blocks
constexpr uint32_t kSbo = 1024;                  // distance between 8-row (K-major) / 8-k (MN-major) atoms
constexpr uint32_t kOutBuf = 32 * 128;            // one staged 32-row x 128-byte output block
constexpr uint32_t kOutStaging = 4 * 2 * kOutBuf; // two blocks per epilogue warp: 32 KB

// NH: 256-column halves per pair tile. NH = 1: 256 x 256 tiles, two TMEM
// accumulators (the epilogue of one tile overlaps the MMAs of the next), a
// 6-stage ring of 32 KB per CTA. NH = 2: 256 x 512 tiles, one accumulator
// filling TMEM, a 4-stage ring of 48 KB: a quarter fewer bytes staged per MMA.
template <int NH>
struct Cfg {
    static constexpr int NACC = 2 / NH;                 // accumulators in TMEM
    static constexpr int NSTAGE = NH == 1 ? 6 : 4;
    static constexpr uint32_t kStageB = NH * kHalfB;
    static constexpr uint32_t a_off = 0;
    static constexpr uint32_t b_off = NSTAGE * kStageA;
    static constexpr uint32_t out_off = b_off + NSTAGE * kStageB;  // epilogue staging
    static constexpr uint32_t bar_off = out_off + kOutStaging;
    // full[NSTAGE], empty[NSTAGE], accf[2], acce[2], done
    static constexpr uint32_t tmem_off = bar_off + 8 * (2 * NSTAGE + 5);
    static constexpr uint32_t total = tmem_off + 16;
};

enum { kEpiStats = 0, kEpiBf16 = 1, kEpiF32 = 2, kEpiProbs = 3 };

struct TcProblem {
    int M, N, K;
    int a_mn, b_mn;     // operand stored MN-major (else K-major)
    int epi;            // kEpiStats / kEpiBf16 / kEpiF32 / kEpiProbs
    int accumulate;     // kEpiF32: D += A B (else D = A B)
    int n_fastest;      // tile order: consecutive tiles walk N (else M)
    int tiles_m, tiles_n, k_blocks;  // tiles_n counts 256-column tiles
    int tiles_np, tiles;             // pair tiles: tiles_m x tiles_np, each kTileM x (NH x kTileN)
    void *d;            // output, row stride ldd elements (fp32 or bf16 by epi)
    int64_t ldd;
    float4 *stats;      // kEpiStats, kEpiProbs: [M x tiles_n] partial row statistics (optional for kEpiStats)
    float4 *refs;       // kEpiProbs: [M x tiles_n] base-2 reference of each 64-column block
    const int32_t *targets;  // kEpiProbs: [M] target column of each row (any value: only in-range ones are kept)
    float *target_logit;     // kEpiProbs: [M] the target's logit, fp32, for rows whose target is in [0, N)
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
    CUtensorMap a[2], b[2], d[2];  // operands and output of each problem
};

// The tiles of a CTA pair, in order: its strided share of problem 0, then its
// share of problem 1. Pairs running at the same time work on neighbouring
// tiles of the same problem, so their operands are shared through L2 (a
// contiguous range per pair would spread them over the whole problem). Both
// CTAs of the pair walk the same list.
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

// Origin of pair tile `tile` and the index of its first 256-column tile.
template <int NH>
__device__ __forceinline__ void tile_origin(const TcProblem &q, int tile, int &m0, int &n0, int &nt) {
    int mt, ntp;
    if (q.n_fastest) {
        mt = tile / q.tiles_np;
        ntp = tile % q.tiles_np;
    } else {
        mt = tile % q.tiles_m;
        ntp = tile / q.tiles_m;
    }
    m0 = mt * kTileM;
    nt = ntp * NH;
    n0 = nt * kTileN;
}

// ---------------------------------------------------------------- epilogues (one accumulator row per thread)
//
// A warp owns 32 accumulator rows. Each 32-column (fp32) or 64-column (bf16)
// block of them goes through one of the warp's two 4-KB staging buffers in
// the 128-byte-swizzled layout of the output's tensor map, and one thread
// issues a bulk tensor store (or reduce-add) of the block; parts past the
// output's edge are clipped by the copy.

struct EpiStage {
    uint32_t buf0;  // this warp's two staging buffers
    int issued;     // blocks issued so far (the buffer alternates)
};

// The next staging buffer, once the copy that last read it is done.
__device__ __forceinline__ uint32_t stage_acquire(EpiStage &e, int lane) {
    const uint32_t b = e.buf0 + (uint32_t)(e.issued & 1) * kOutBuf;
    if (e.issued >= 2 && lane == 0) ptx::bulk_wait_group_read<1>();
    __syncwarp();
    return b;
}

// One 128-byte row of the block (this thread's): 16-byte unit j at j ^ (row % 8).
__device__ __forceinline__ void stage_row(uint32_t buf, int lane, const uint32_t (&v)[32]) {
    const uint32_t row = buf + (uint32_t)lane * 128u;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        ptx::st_shared_v4(row + ((uint32_t)(j ^ (lane & 7)) << 4), v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
}

__device__ __forceinline__ void stage_issue(EpiStage &e, int lane, const void *tmap, int x, int y, uint32_t buf,
                                            bool reduce) {
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (reduce)
            ptx::tma_reduce_add_2d(tmap, x, y, buf);
        else
            ptx::tma_store_2d(tmap, x, y, buf);
        ptx::bulk_commit_group();
    }
    ++e.issued;
}

// fp32 logits + per-row softmax statistics of the 256 columns at n0.
__device__ __forceinline__ void epi_stats(const TcProblem &q, const void *dmap, EpiStage &es, int lane,
                                          uint32_t tbase, int row, int wrow0, int n0, int nt) {
    RowStats2 st = empty_stats();
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
        if (st.m2 == -INFINITY) {  // every value so far is -inf (adds nothing) or NaN (must show)
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < nvalid && !(__uint_as_float(r[j]) == __uint_as_float(r[j]))) st.s = __uint_as_float(r[j]);
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (j < nvalid) {  // a -inf logit adds nothing (0 log 0 = 0): see the row kernel
                    const float d2 = fmaf(__uint_as_float(r[j]), kLog2e, -st.m2);
                    const float e = ex2_approx(d2);
                    st.s += e;
                    st.u2 = fmaf(e, fmaxf(d2, -256.f), st.u2);
                }
            }
        }
        if (q.d) {
            const uint32_t buf = stage_acquire(es, lane);
            stage_row(buf, lane, r);
            stage_issue(es, lane, dmap, col0, wrow0, buf, false);
        }
    }
    if (q.stats && row < q.M) q.stats[(size_t)row * q.tiles_n + nt] = make_float4(st.m2, st.s, st.u2, 0.f);
}

// Scaled probabilities + per-row softmax statistics of the 256 columns at n0
// (the fused loss path). Each 64-column block is stored in bf16 as
// e_v = 2^{z_v log2e - m}, m the row's running base-2 maximum after the block,
// and m is kept per block in `refs`: every stored value is in [0, 1] and keeps
// bf16's relative precision whatever its size, so p_v = e_v 2^{m - logZ2}
// once the row's logZ is known. The target's own logit is kept exactly
// (fp32) for the log-probability.
__device__ __forceinline__ void epi_probs(const TcProblem &q, const void *dmap, EpiStage &es, int lane,
                                          uint32_t tbase, int row, int wrow0, int n0, int nt, int y) {
    RowStats2 st = empty_stats();
    float4 ref = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
#pragma unroll 1
    for (int c = 0; c < kTileN / 64; ++c) {
        uint32_t r[2][32];
        ptx::tmem_ld_32x32b_x32(tbase + c * 64, r[0]);
        ptx::tmem_ld_32x32b_x32(tbase + c * 64 + 32, r[1]);
        ptx::tmem_ld_wait();
        const int col0 = n0 + c * 64;
        const int nvalid = min(64, q.N - col0);
        if (nvalid <= 0) break;
        float mv = -INFINITY;
#pragma unroll
        for (int j = 0; j < 64; ++j)
            if (j < nvalid) mv = fmaxf(mv, __uint_as_float(r[j >> 5][j & 31]));
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
        float e[64];
        if (st.m2 == -INFINITY) {  // every value so far is -inf (probability 0) or NaN (must show)
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                const float x = __uint_as_float(r[j >> 5][j & 31]);
                const bool nan = j < nvalid && !(x == x);
                if (nan) st.s = x;
                e[j] = nan ? x : 0.f;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                const float d2 = fmaf(__uint_as_float(r[j >> 5][j & 31]), kLog2e, -st.m2);
                const float ej = ex2_approx(d2);
                if (j < nvalid) {  // a -inf logit adds nothing (0 log 0 = 0): see the row kernel
                    st.s += ej;
                    st.u2 = fmaf(ej, fmaxf(d2, -256.f), st.u2);
                }
                e[j] = j < nvalid ? ej : 0.f;
            }
        }
        if ((unsigned)(y - col0) < (unsigned)nvalid) {  // this row's target: its logit exactly
            float zy = 0.f;
#pragma unroll
            for (int j = 0; j < 64; ++j) zy = (j == y - col0) ? __uint_as_float(r[j >> 5][j & 31]) : zy;
            q.target_logit[row] = zy;
        }
        ref.x = c == 0 ? st.m2 : ref.x;
        ref.y = c == 1 ? st.m2 : ref.y;
        ref.z = c == 2 ? st.m2 : ref.z;
        ref.w = c == 3 ? st.m2 : ref.w;
        uint32_t pk[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) pk[j] = pack_bf16x2(e[2 * j], e[2 * j + 1]);
        const uint32_t buf = stage_acquire(es, lane);
        stage_row(buf, lane, pk);
        stage_issue(es, lane, dmap, col0, wrow0, buf, false);
    }
    if (row < q.M) {
        const size_t i = (size_t)row * q.tiles_n + nt;
        q.stats[i] = make_float4(st.m2, st.s, st.u2, 0.f);
        q.refs[i] = ref;
    }
}

// bf16 output of the 256 columns at n0, 64 columns per staged block.
__device__ __forceinline__ void epi_bf16(const TcProblem &q, const void *dmap, EpiStage &es, int lane,
                                         uint32_t tbase, int wrow0, int n0) {
#pragma unroll 1
    for (int c = 0; c < kTileN / 64; ++c) {
        const int col0 = n0 + c * 64;
        if (col0 >= q.N) break;
        uint32_t pk[32];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x32(tbase + c * 64 + hh * 32, r);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j)
                pk[hh * 16 + j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
        }
        const uint32_t buf = stage_acquire(es, lane);
        stage_row(buf, lane, pk);
        stage_issue(es, lane, dmap, col0, wrow0, buf, false);
    }
}

// fp32 output of the 256 columns at n0: stored, or added into the output.
__device__ __forceinline__ void epi_f32(const TcProblem &q, const void *dmap, EpiStage &es, int lane,
                                        uint32_t tbase, int wrow0, int n0) {
#pragma unroll 1
    for (int c = 0; c < kTileN / 32; ++c) {
        const int col0 = n0 + c * 32;
        if (col0 >= q.N) break;
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(tbase + c * 32, r);
        ptx::tmem_ld_wait();
        const uint32_t buf = stage_acquire(es, lane);
        stage_row(buf, lane, r);
        stage_issue(es, lane, dmap, col0, wrow0, buf, q.accumulate != 0);
    }
}

// ---------------------------------------------------------------- the kernel

template <int NH>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ TcMaps maps, const __grid_constant__ TcParams p) {
    using C = Cfg<NH>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // the swizzled tiles need 1024-byte alignment (the same offset in both CTAs of a pair)
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    unsigned char *smem = smem_raw + (sbase - raw);

    const uint32_t full0 = sbase + C::bar_off;
    const uint32_t empty0 = full0 + 8 * C::NSTAGE;
    const uint32_t accf0 = empty0 + 8 * C::NSTAGE;
    const uint32_t acce0 = accf0 + 16;
    const uint32_t done_bar = acce0 + 16;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::tmem_off);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();  // 0: the pair's MMA issuer
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const ClusterTiles tiles(p, pair, npairs);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NSTAGE; ++s) {
            ptx::mbar_init(full0 + 8 * s, 1);
            ptx::mbar_init(empty0 + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(accf0 + 8 * a, 1);
            ptx::mbar_init(acce0 + 8 * a, 8);  // one arrival per epilogue warp of both CTAs
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
    ptx::cluster_sync();  // both CTAs' barriers are initialised before either signals the other's
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    bool timed_out = false;
    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer (both CTAs)
        if (lane == 0) {
            const uint32_t full_leader0 = ptx::mapa_shared(full0, 0);
            uint32_t it = 0;
            int prob, tile;
            for (int i = 0; tiles.at(i, prob, tile); ++i) {
                int m0, n0, nt;
                const TcProblem &q = p.prob[prob];
                tile_origin<NH>(q, tile, m0, n0, nt);
                const void *am = &maps.a[prob];
                const void *bm = &maps.b[prob];
                const int ma = m0 + (int)rank * kRowsCta;
                for (int kb = 0; kb < q.k_blocks; ++kb, ++it) {
                    const uint32_t s = it % C::NSTAGE, ph = (it / C::NSTAGE) & 1u;
                    if (!timed_out && !ptx::mbar_wait(empty0 + 8 * s, ph ^ 1u)) timed_out = true;
                    const uint32_t fb = full_leader0 + 8 * s;
                    if (rank == 0) ptx::mbar_arrive_expect_tx(full0 + 8 * s, 2 * (kStageA + C::kStageB));
                    const uint32_t a_dst = sbase + C::a_off + s * kStageA;
                    const uint32_t b_dst = sbase + C::b_off + s * C::kStageB;
                    const int k0 = kb * BK;
                    if (q.a_mn) {
                        ptx::tma_load_2d_pair(a_dst, am, ma, k0, fb);
                        ptx::tma_load_2d_pair(a_dst + kMnBlock, am, ma + 64, k0, fb);
                    } else {
                        ptx::tma_load_2d_pair(a_dst, am, k0, ma, fb);
                    }
#pragma unroll
                    for (int h = 0; h < NH; ++h) {
                        // this CTA's 128 columns of half h: [n0 + 256 h + 128 rank, + 128)
                        const int nb = n0 + h * kTileN + (int)rank * kBnCta;
                        const uint32_t bd = b_dst + h * kHalfB;
                        if (q.b_mn) {
                            ptx::tma_load_2d_pair(bd, bm, nb, k0, fb);
                            ptx::tma_load_2d_pair(bd + kMnBlock, bm, nb + 64, k0, fb);
                        } else {
                            ptx::tma_load_2d_pair(bd, bm, k0, nb, fb);
                        }
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer (even CTA)
        if (rank == 0 && lane == 0) {
            uint32_t it = 0;
            int prob, tile;
            for (int i = 0; tiles.at(i, prob, tile); ++i) {
                const TcProblem &q = p.prob[prob];
                const uint32_t idesc = ptx::idesc_bf16_f32_major(kTileM, kTileN, q.a_mn, q.b_mn);
                const uint32_t a_step = q.a_mn ? 16 * 128 : 32, b_step = q.b_mn ? 16 * 128 : 32;
                const uint32_t a_lbo = q.a_mn ? kLboMn : 16, b_lbo = q.b_mn ? kLboMn : 16;
                const uint32_t acc = (uint32_t)i % C::NACC, aph = ((uint32_t)i / C::NACC) & 1u;
                if (NH == 1) {  // this accumulator's previous tile has been drained
                    if (!timed_out && !ptx::mbar_wait(acce0 + 8 * acc, aph ^ 1u)) timed_out = true;
                    ptx::tc_fence_after();
                }
                for (int kb = 0; kb < q.k_blocks; ++kb, ++it) {
                    const uint32_t s = it % C::NSTAGE, ph = (it / C::NSTAGE) & 1u;
                    if (!timed_out && !ptx::mbar_wait(full0 + 8 * s, ph)) timed_out = true;
                    ptx::tc_fence_after();
                    const uint32_t a_addr = sbase + C::a_off + s * kStageA;
                    const uint32_t b_addr = sbase + C::b_off + s * C::kStageB;
#pragma unroll
                    for (int h = 0; h < NH; ++h) {
                        if (NH > 1 && kb == 0) {  // half h of the previous tile has been drained
                            if (!timed_out && !ptx::mbar_wait(acce0 + 8 * h, aph ^ 1u)) timed_out = true;
                            ptx::tc_fence_after();
                        }
                        const uint32_t d_tmem = tmem_base + (acc * NH + h) * kTileN;
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk) {
                            const uint64_t ad = ptx::smem_desc_sw128(a_addr + kk * a_step, a_lbo, kSbo);
                            const uint64_t bd = ptx::smem_desc_sw128(b_addr + h * kHalfB + kk * b_step, b_lbo, kSbo);
                            ptx::mma_bf16_ss_pair(d_tmem, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    ptx::mma_commit_pair(empty0 + 8 * s, 0x3);  // the stage is free in both CTAs
                }
                ptx::mma_commit_pair(accf0 + 8 * acc, 0x3);  // accumulator complete in both CTAs
            }
            ptx::mma_commit_pair(done_bar, 0x3);  // every MMA of this pair has completed
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- epilogue (both CTAs)
        const int qd = warp & 3;  // TMEM lane quarter this warp may access
        const uint32_t acce_leader0 = ptx::mapa_shared(acce0, 0);
        EpiStage es{sbase + C::out_off + (uint32_t)(warp - 2) * 2u * kOutBuf, 0};
        int prob, tile;
        for (int i = 0; tiles.at(i, prob, tile); ++i) {
            int m0, n0, nt;
            const TcProblem &q = p.prob[prob];
            const void *dmap = &maps.d[prob];
            tile_origin<NH>(q, tile, m0, n0, nt);
            const int wrow0 = m0 + (int)rank * kRowsCta + qd * 32;  // this warp's first row
            const int row = wrow0 + lane;
            const uint32_t acc = (uint32_t)i % C::NACC, aph = ((uint32_t)i / C::NACC) & 1u;
            const int y = (q.epi == kEpiProbs && row < q.M) ? __ldg(q.targets + row) : -1;
            if (!timed_out && !ptx::mbar_wait(accf0 + 8 * acc, aph)) timed_out = true;
            ptx::tc_fence_after();
#pragma unroll 1
            for (int h = 0; h < NH; ++h) {
                const int n0h = n0 + h * kTileN;
                const uint32_t tbase = tmem_base + ((uint32_t)(qd * 32) << 16) + (acc * NH + h) * kTileN;
                if (n0h >= q.N || wrow0 >= q.M) {
                    // past the last column (an odd count of 256-column tiles) or below the last row
                } else if (q.epi == kEpiProbs) {
                    epi_probs(q, dmap, es, lane, tbase, row, wrow0, n0h, nt + h, y);
                } else if (q.epi == kEpiStats) {
                    epi_stats(q, dmap, es, lane, tbase, row, wrow0, n0h, nt + h);
                } else if (q.epi == kEpiBf16) {
                    epi_bf16(q, dmap, es, lane, tbase, wrow0, n0h);
                } else {
                    epi_f32(q, dmap, es, lane, tbase, wrow0, n0h);
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive_cluster(acce_leader0 + 8 * (NH == 1 ? acc : (uint32_t)h));
            }
        }
        if (lane == 0) ptx::bulk_wait_group<0>();  // the staged blocks are written out
        __syncwarp();
    }

    ptx::tc_fence_before();
    ptx::cluster_sync();  // no CTA leaves while the other may still signal it
    ptx::tc_fence_after();
    if (warp == 1) {
        // every MMA of the pair has completed before TMEM is released
        if (!ptx::mbar_wait(done_bar, 0, timed_out ? 100000000ull : 2000000000ull)) timed_out = true;
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
    }
    if (timed_out) raise_status(p.status, RL_ERR_TIMEOUT);
}

// ------------------------------------------------------------------ host side

bool make_tmap_bf16(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int64_t ld, uint32_t box_rows) {
    return make_tmap_sw128(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, rows, cols, ld, BK, box_rows);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tensor maps of one operand: K-major [outer x K] (boxes of `k_rows` outer
// rows x 64 K) or MN-major [K x outer] (boxes of 64 k rows x 64 outer elements).
bool operand_map(CUtensorMap *m, const GemmOperand &o, int64_t outer, int64_t K, uint32_t k_rows) {
    if (!o.base || !aligned16(o.base) || (o.ld * 2) % 16 != 0) return false;
    if (o.mn_major) {
        if (o.ld < outer) return false;
        return make_tmap_bf16(m, o.base, K, outer, o.ld, 64);
    }
    if (o.ld < K) return false;
    return make_tmap_bf16(m, o.base, outer, K, o.ld, k_rows);
}

// 256-column halves per pair tile (see Cfg).
constexpr int kHalves = 2;
using KCfg = Cfg<kHalves>;
const auto kKernel = tc_gemm_kernel<kHalves>;

std::mutex g_mu;
int g_pairs[64] = {};
bool g_attr[64] = {};

cudaLaunchConfig_t pair_config(int pairs, int smem, cudaStream_t stream, cudaLaunchAttribute *attr) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

cudaError_t launch(const GemmProblem *probs, int nprob, uint32_t *status, cudaStream_t stream) {
    TcMaps maps;
    TcParams p{};
    p.nprob = nprob;
    p.status = status;
    for (int i = 0; i < nprob; ++i) {
        const GemmProblem &g = probs[i];
        if (g.M <= 0 || g.N <= 0 || g.K <= 0) return cudaErrorInvalidValue;
        if (!operand_map(&maps.a[i], g.a, g.M, g.K, kRowsCta) || !operand_map(&maps.b[i], g.b, g.N, g.K, kBnCta))
            return cudaErrorInvalidValue;
        if (!g.d && g.epi != GemmProblem::kZStats) return cudaErrorInvalidValue;
        if (g.epi == GemmProblem::kProbStats && (!g.stats || !g.refs || !g.targets || !g.target_logit))
            return cudaErrorInvalidValue;
        if (g.d) {  // the output, written in staged 32-row blocks of 128 bytes per row
            const bool f32 = g.epi == GemmProblem::kZStats || g.epi == GemmProblem::kF32;
            const uint32_t es = f32 ? 4 : 2;
            if (!aligned16(g.d) || g.ldd < g.N || (g.ldd * es) % 16 != 0 ||
                !make_tmap_sw128(&maps.d[i], f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, es,
                           g.d, g.M, g.N, g.ldd, 128 / es, 32))
                return cudaErrorInvalidValue;
        }
        TcProblem &q = p.prob[i];
        q.M = g.M;
        q.N = g.N;
        q.K = g.K;
        q.a_mn = g.a.mn_major;
        q.b_mn = g.b.mn_major;
        q.epi = g.epi == GemmProblem::kZStats      ? kEpiStats
                : g.epi == GemmProblem::kProbStats ? kEpiProbs
                : g.epi == GemmProblem::kBf16      ? kEpiBf16
                                                   : kEpiF32;
        q.accumulate = g.accumulate;
        q.n_fastest = g.n_fastest;
        q.tiles_m = (g.M + kTileM - 1) / kTileM;
        q.tiles_n = (g.N + kTileN - 1) / kTileN;
        q.k_blocks = (g.K + BK - 1) / BK;
        q.tiles_np = (q.tiles_n + kHalves - 1) / kHalves;
        q.tiles = q.tiles_m * q.tiles_np;
        q.d = g.d;
        q.ldd = g.ldd;
        q.stats = g.stats;
        q.refs = g.refs;
        q.targets = g.targets;
        q.target_logit = g.target_logit;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int smem = (int)KCfg::total + 1024;
    int max_pairs = 0;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (dev < 64 && !g_attr[dev]) {
            e = cudaFuncSetAttribute(kKernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            cudaLaunchAttribute oa[1];
            cudaLaunchConfig_t oc = pair_config(1, smem, 0, oa);
            int pairs = 0;
            if (cudaOccupancyMaxActiveClusters(&pairs, kKernel, &oc) != cudaSuccess || pairs <= 0) {
                cudaGetLastError();
                int sms = 0;
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
                pairs = sms / 2;
            }
            g_pairs[dev] = pairs;
            g_attr[dev] = true;
        }
        max_pairs = dev < 64 ? g_pairs[dev] : 0;
    }
    if (max_pairs <= 0) {
        int sms = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        max_pairs = std::max(1, sms / 2);
    }
    int64_t all_tiles = 0;
    for (int i = 0; i < nprob; ++i) all_tiles += p.prob[i].tiles;
    const int npairs = (int)std::min<int64_t>(all_tiles, max_pairs);
    if (nprob > 1)  // one problem-0 tile, in problem-1 tiles
        p.p1_delay = (p.prob[0].k_blocks + p.prob[1].k_blocks / 2) / p.prob[1].k_blocks;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pair_config(npairs, smem, stream, attr);
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
