// Generalized advantage estimation with skipped observation tokens and the
// cross-trajectory discount ("Zhipu AI / GLM: From Blank Infilling to
// Compaction-Aware Agentic Reinforcement Learning", section 11: skip-
// observation GAE of the single-rollout critic, and CompactionRL's
// "cross-trajectory GAE" over the segments of one rollout), as a deterministic
// segmented reverse scan.
//
// Per response, walking backwards over its action (mask=1) tokens t with next
// action token t':  A_t = r_t + gamma V_{t'} - V_t + gamma lambda A_{t'}
// (V_{t'} = A_{t'} = 0 after the last one); observation tokens get A = 0.
// The map a run of tokens applies to the state (A, V) entering it from the
// right is affine and, once it holds an action token, of the form
//   A <- p A + q V + c,  V <- v_first   with p = (gamma lambda)^k,
//   q = gamma (gamma lambda)^(k-1) for k action tokens, v_first the value of the
//   leftmost one
// (observation-only runs are the identity). Such maps compose associatively,
// so a block handles one response as a sequence of tiles of 8192 tokens taken
// right to left: each tile is staged in shared memory with coalesced loads,
// every thread folds its 8 tokens into a map (fp32), a fixed-tree suffix scan
// over the 1024 threads' maps (warp shuffles, then across warps) gives each
// thread the state entering its tokens, the thread re-walks them, and the
// state leaving the tile is carried in double to the next tile on the left.
// The tree depends only on the response length: results are bit-identical
// from run to run. One block per response (responses are independent).
#include "common.cuh"

namespace rlk {

namespace {

constexpr int kGaeThreads = 1024;
constexpr int kPerThread = 8;
constexpr int kTile = kGaeThreads * kPerThread;

// A <- p A + q V + c, V <- vf when `has` (at least one action token); identity otherwise.
struct GaeMap {
    float p, q, c, vf;
    int has;
};

__device__ __forceinline__ GaeMap gae_identity() { return GaeMap{1.f, 0.f, 0.f, 0.f, 0}; }

// (F o G): G (the tokens to the right) acts first.
__device__ __forceinline__ GaeMap gae_compose(const GaeMap &F, const GaeMap &G) {
    if (!G.has) return F;
    if (!F.has) return G;
    return GaeMap{F.p * G.p, F.p * G.q, fmaf(F.q, G.vf, fmaf(F.p, G.c, F.c)), F.vf, 1};
}

__device__ __forceinline__ GaeMap gae_shfl_down(const GaeMap &a, int off) {
    return GaeMap{__shfl_down_sync(0xffffffffu, a.p, off), __shfl_down_sync(0xffffffffu, a.q, off),
                  __shfl_down_sync(0xffffffffu, a.c, off), __shfl_down_sync(0xffffffffu, a.vf, off),
                  __shfl_down_sync(0xffffffffu, a.has, off)};
}

// Inclusive suffix scan within a warp: lane l gets F_l o ... o F_31.
__device__ __forceinline__ GaeMap gae_warp_suffix(GaeMap x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const GaeMap o = gae_shfl_down(x, off);
        if (lane + off < 32) x = gae_compose(x, o);
    }
    return x;
}

__global__ void __launch_bounds__(kGaeThreads) gae_kernel(GaeParams p) {
    __shared__ float s_r[kTile];
    __shared__ float s_v[kTile];
    __shared__ uint8_t s_m[kTile];
    __shared__ GaeMap warp_tot[kGaeThreads / 32];
    __shared__ GaeMap warp_after[kGaeThreads / 32];
    __shared__ int iscratch[32];
    const int s = blockIdx.x;
    const int T = p.num_tokens;
    int b = __ldg(p.cu_seqlens + s), e = __ldg(p.cu_seqlens + s + 1);
    if (b < 0 || e < b || e > T) {
        if (threadIdx.x == 0 && p.status) raise_status(p.status, RL_ERR_SEQLENS);
        b = min(max(b, 0), T);
        e = min(max(e, b), T);
    }
    const float gamma = (float)p.gamma, gl = (float)(p.gamma * p.lambda);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    // cross-trajectory discount: trainable tokens in the later segments of this rollout
    double scale = 1.0;
    if (p.rollout_ids) {
        const int rid = __ldg(p.rollout_ids + s);
        int later = 0;
        for (int u = s + 1; u < p.num_seqs && __ldg(p.rollout_ids + u) == rid; ++u) {
            const int ub = min(max(__ldg(p.cu_seqlens + u), 0), T), ue = min(max(__ldg(p.cu_seqlens + u + 1), ub), T);
            int cnt = 0;
            for (int t = ub + threadIdx.x; t < ue; t += kGaeThreads) cnt += __ldg(p.mask + t) ? 1 : 0;
            later += block_sum_i32(cnt, iscratch);
        }
        scale = pow(p.gamma * p.lambda, (double)later);
    }

    double carry_A = 0.0, carry_V = 0.0;  // the state entering the current tile from the right
    const int n = e - b;
    const int ntiles = (n + kTile - 1) / kTile;
    for (int tile = ntiles - 1; tile >= 0; --tile) {
        const int t0 = b + tile * kTile, t1 = min(e, t0 + kTile);
        // stage the tile (coalesced); observation tokens become mask 0
#pragma unroll
        for (int i = 0; i < kPerThread; ++i) {
            const int j = i * kGaeThreads + threadIdx.x, t = t0 + j;
            const bool in = t < t1;
            s_r[j] = in ? __ldg(p.rewards + t) : 0.f;
            s_v[j] = in ? __ldg(p.values + t) : 0.f;
            s_m[j] = in && (!p.skip_observations || __ldg(p.mask + t)) ? 1 : 0;
        }
        __syncthreads();
        // this thread's 8 consecutive tokens, folded right to left
        const int j0 = threadIdx.x * kPerThread;
        GaeMap F = gae_identity();
#pragma unroll
        for (int i = kPerThread - 1; i >= 0; --i) {
            const int j = j0 + i;
            if (!s_m[j]) continue;
            const float r = s_r[j], v = s_v[j];
            if (!F.has)
                F = GaeMap{gl, gamma, r - v, v, 1};
            else
                F = GaeMap{gl * F.p, gl * F.q, fmaf(gl, F.c, fmaf(gamma, F.vf, r - v)), v, 1};
        }
        // exclusive suffix over the threads of the block
        const GaeMap incl = gae_warp_suffix(F);
        if (lane == 0) warp_tot[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const GaeMap wi = gae_warp_suffix(warp_tot[lane]);
            GaeMap after = gae_shfl_down(wi, 1);
            if (lane == 31) after = gae_identity();
            warp_after[lane] = after;
        }
        __syncthreads();
        GaeMap right = gae_shfl_down(incl, 1);
        if (lane == 31) right = gae_identity();
        const GaeMap ex = gae_compose(right, warp_after[warp]);
        // the state entering this thread's tokens: ex applied to the tile's carry
        float A_next, V_next;
        if (ex.has) {
            A_next = (float)((double)ex.c + (double)ex.q * carry_V + (double)ex.p * carry_A);
            V_next = ex.vf;
        } else {
            A_next = (float)carry_A;
            V_next = (float)carry_V;
        }
        // the state leaving the tile (thread 0's inclusive map), in double, for the next tile
        const GaeMap whole = gae_compose(incl, warp_after[warp]);
        __syncthreads();  // every thread has read warp_after before it is reused
        if (threadIdx.x == 0 && whole.has) {
            const double A = (double)whole.c + (double)whole.q * carry_V + (double)whole.p * carry_A;
            warp_tot[0] = GaeMap{(float)A, (float)(A - (double)(float)A), 0.f, whole.vf, 1};
        }
        // re-walk, results written back into s_r (coalesced store below)
#pragma unroll
        for (int i = kPerThread - 1; i >= 0; --i) {
            const int j = j0 + i;
            if (!s_m[j]) {
                s_r[j] = 0.f;
                continue;
            }
            const float v = s_v[j];
            const float A = fmaf(gl, A_next, fmaf(gamma, V_next, s_r[j] - v));
            s_r[j] = A;
            A_next = A;
            V_next = v;
        }
        __syncthreads();
        if (warp_tot[0].has && ntiles > 1) {  // the carry, hi + lo parts of the double
            carry_A = (double)warp_tot[0].p + (double)warp_tot[0].q;
            carry_V = (double)warp_tot[0].vf;
        }
#pragma unroll
        for (int i = 0; i < kPerThread; ++i) {
            const int j = i * kGaeThreads + threadIdx.x, t = t0 + j;
            if (t < t1) {
                const double A = (double)s_r[j] * scale;
                p.adv[t] = (float)A;
                if (p.returns) p.returns[t] = s_m[j] ? (float)(A + (double)s_v[j]) : 0.f;
            }
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_gae(const GaeParams &p, cudaStream_t stream) {
    if (p.num_seqs <= 0) return cudaSuccess;
    gae_kernel<<<p.num_seqs, kGaeThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace rlk
