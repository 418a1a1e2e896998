// The fused row kernel: log-softmax statistics, target log-prob, entropy, the
// token objective of Eq. (1) ("GLM-5: from Vibe Coding to Agentic
// Engineering", section 3.2) and dL/dlogits, one block per logits row.
//
// Per row t (z = logits row, V entries):
//   pass 1: statistics M, S, U (base 2, see RowStats2) with 16-byte loads, a
//           fixed element-to-thread map and a fixed merge tree;
//   finish: logZ, logp = z_y - logZ, H, and the token objective;
//   pass 2: dz_v = g (1[v == y] - 2^{z_v log2e - logZ2}), rounded once to the
//           logits dtype, re-reading the row (served by L1 / L2: DRAM traffic
//           stays one read and one write per element).
// Rows with g == 0 (masked, popped, clipped, zero advantage) are written as
// +0.0 without evaluating the softmax a second time.
#include <algorithm>
#include <cfloat>
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace rlk {

namespace {

// Rows of at most this many bytes use 256-thread blocks (eight rows per SM, eight
// 16-byte loads in flight per thread). Longer rows use 1024-thread blocks (two
// per SM) and keep their first kStageBytes in shared memory from the first pass
// to the second, which shrinks what must stay in L2: one thread issues bulk
// copies of that prefix into shared memory as the block starts, the threads
// fold the rest of the row meanwhile and then the prefix. Every row reads its
// second pass with an L1 evict-first hint, streams its dlogits out with
// evict-first stores (so they do not push rows still waiting for their second
// read out of L2), and walks each thread's groups in reverse in the second
// pass (most recently loaded first). Chosen from GB300 sweeps over
// 128/256/512/1024 threads, staging sizes, unrolling and the cache hints.
constexpr size_t kShortRowBytes = 128 * 1024;
constexpr int kStageBytes = 96 * 1024;

template <typename T>
struct VecTraits;

template <>
struct VecTraits<float> {
    static constexpr int kElems = 4;
    __device__ __forceinline__ static void load(const void *p, float (&x)[4]) {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(p));
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    }

    __device__ __forceinline__ static float load1(const void *p, int64_t v) {
        return __ldg(reinterpret_cast<const float *>(p) + v);
    }
    // the second read, evict-first from L1: nothing reads it again, and it leaves L1 to the other rows
    __device__ __forceinline__ static void load_last(const void *p, float (&x)[4]) {
        float4 v;
        asm("ld.global.nc.L1::evict_first.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    }
    // streaming stores: dz is not read again here, and keeping it out of L2 leaves room for the rows
    // still waiting for their second read
    __device__ __forceinline__ static void store(void *p, const float (&x)[4]) {
        __stcs(reinterpret_cast<float4 *>(p), make_float4(x[0], x[1], x[2], x[3]));
    }
    __device__ __forceinline__ static void store1(void *p, int64_t v, float x) {
        reinterpret_cast<float *>(p)[v] = x;
    }
};

template <>
struct VecTraits<__nv_bfloat16> {
    static constexpr int kElems = 8;
    __device__ __forceinline__ static void load(const void *p, float (&x)[8]) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p));
        x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
        x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z); x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
    }

    __device__ __forceinline__ static float load1(const void *p, int64_t v) {
        const uint16_t b = __ldg(reinterpret_cast<const unsigned short *>(p) + v);
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
    // the second read, evict-first from L1 (as for fp32)
    __device__ __forceinline__ static void load_last(const void *p, float (&x)[8]) {
        uint4 v;
        asm("ld.global.nc.L1::evict_first.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
        x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
        x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z); x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
    }
    __device__ __forceinline__ static void store(void *p, const float (&x)[8]) {
        uint4 v;
        v.x = pack_bf16x2(x[0], x[1]); v.y = pack_bf16x2(x[2], x[3]);
        v.z = pack_bf16x2(x[4], x[5]); v.w = pack_bf16x2(x[6], x[7]);
        __stcs(reinterpret_cast<uint4 *>(p), v);  // streaming, as for fp32
    }
    __device__ __forceinline__ static void store1(void *p, int64_t v, float x) {
        reinterpret_cast<__nv_bfloat16 *>(p)[v] = __float2bfloat16_rn(x);
    }
};

// One 16-byte group of logits as floats.
template <typename T>
__device__ __forceinline__ void decode16(const uint4 &v, float (&x)[16 / sizeof(T)]);
template <>
__device__ __forceinline__ void decode16<float>(const uint4 &v, float (&x)[4]) {
    x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y); x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
}
template <>
__device__ __forceinline__ void decode16<__nv_bfloat16>(const uint4 &v, float (&x)[8]) {
    x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
    x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z); x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
}

// Fold a group of values into running base-2 statistics (one rescale per group).
template <int N>
__device__ __forceinline__ void accumulate(RowStats2 &st, const float (&x)[N]) {
    float mv = x[0];
#pragma unroll
    for (int k = 1; k < N; ++k) mv = fmaxf(mv, x[k]);
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
    for (int k = 0; k < N; ++k) {
        const float d2 = fmaf(x[k], kLog2e, -st.m2);
        const float e = ex2_approx(d2);
        st.s += e;
        st.u2 = fmaf(e, d2, st.u2);  // NaN for a -inf logit (0 * -inf): see kRowStart
    }
}

// Start of a thread's statistics: a finite reference point, so that a -inf logit gives e = 0
// (it adds nothing to s) even before the thread has seen a finite one. Only u2 then turns NaN
// (0 * -inf): a row whose s is finite but whose u2 is NaN holds -inf logits and no NaN or +inf,
// and its entropy is redone by entropy_fix_kernel. Merging a start that saw nothing scales it
// by 2^(-FLT_MAX - M) = 0: bit for bit the same as merging an empty part.
constexpr RowStats2 kRowStart{-FLT_MAX, 0.f, 0.f};

// kStage: the first stage_vecs 16-byte groups of the row arrive in shared memory by bulk copies
// and stay there between the passes; the bounded wait for them raises RL_ERR_TIMEOUT if it runs
// out (the row's results are then not valid).
template <typename T, int kRowThreads, bool kStage>
__global__ void __launch_bounds__(kRowThreads, 2048 / kRowThreads) row_loss_twopass_kernel(RowParams p, int stage_vecs) {
    using VT = VecTraits<T>;
    constexpr int VEC = VT::kElems;
    constexpr int kUnroll = kRowThreads <= 256 ? 8 : 4;  // 16-byte loads in flight per thread
    extern __shared__ uint4 s_row[];
    __shared__ RowStats2 warp_stats[kRowThreads / 32];
    __shared__ float s_logZ2, s_g;
    __shared__ uint32_t s_y;

    const int row = blockIdx.x;
    const int V = p.vocab;
    const int nvec = V / VEC;
    const int tail0 = nvec * VEC;
    const char *z = reinterpret_cast<const char *>(p.logits) + (size_t)row * p.ld_logits * sizeof(T);
    char *dz = reinterpret_cast<char *>(p.dlogits) + (size_t)row * p.ld_dlogits * sizeof(T);
    const float4 rec = __ldg(p.rec + row);
    const uint32_t meta = __ldg(p.meta + row);

    RowStats2 st = kRowStart;
    __shared__ __align__(8) uint64_t s_bar;
    if (kStage) {
        // the row's first stage_vecs groups arrive in shared memory by bulk copies while the
        // threads fold the rest of the row
        const uint32_t bar = ptx::smem_u32(&s_bar);
        if (threadIdx.x == 0) {
            ptx::mbar_init(bar, 1);
            ptx::fence_mbar_init();
            const uint32_t bytes = (uint32_t)stage_vecs * 16u;
            ptx::mbar_arrive_expect_tx(bar, bytes);
            const uint64_t pol = ptx::l2_evict_first_policy();  // read once: not needed in L2 again
            for (uint32_t off = 0; off < bytes; off += 16384u)
                ptx::bulk_g2s_hint(ptx::smem_u32(s_row) + off, z + off, min(16384u, bytes - off), bar, pol);
        }
        __syncthreads();
#pragma unroll kUnroll
        for (int k = stage_vecs + (int)threadIdx.x; k < nvec; k += kRowThreads) {
            float x[VEC];
            VT::load(z + (size_t)k * 16, x);
            accumulate(st, x);
        }
        if (tail0 + (int)threadIdx.x < V) {
            float x[1] = {VT::load1(z, tail0 + threadIdx.x)};
            accumulate(st, x);
        }
        if (!ptx::mbar_wait(bar, 0u)) {
            // the copies did not land in time: flag it (the row's results are not valid) and give
            // them one more bounded wait, so that none is still in flight when the block exits
            raise_status(p.status, RL_ERR_TIMEOUT);
            if (threadIdx.x == 0) ptx::mbar_wait(bar, 0u, 100000000ull);
        }
#pragma unroll kUnroll
        for (int k = threadIdx.x; k < stage_vecs; k += kRowThreads) {
            float x[VEC];
            decode16<T>(s_row[k], x);
            accumulate(st, x);
        }
    } else {
#pragma unroll kUnroll
        for (int k = threadIdx.x; k < nvec; k += kRowThreads) {
            float x[VEC];
            VT::load(z + (size_t)k * 16, x);
            accumulate(st, x);
        }
        if (tail0 + (int)threadIdx.x < V) {
            float x[1] = {VT::load1(z, tail0 + threadIdx.x)};
            accumulate(st, x);
        }
    }
    st = warp_merge_stats2(st);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) warp_stats[warp] = st;
    __syncthreads();
    if (warp == 0) {
        RowStats2 w = lane < kRowThreads / 32 ? warp_stats[lane] : empty_stats();
        w = warp_merge_stats2(w);
        if (lane == 0) {
            const RowOut o = finish_row(w, rec, meta, p.c, p.teacher ? __ldg(p.teacher + row) : 0.f);
            if (!isfinite(o.logZ2)) raise_status(p.status, RL_ERR_NONFINITE);  // NaN or +inf logit in the row
            // -inf logits (kRowStart): the entropy is redone by entropy_fix_kernel
            if (isfinite(w.s) && isnan(w.u2)) p.fix_rows[row] = 1;
            if (p.logp_out) p.logp_out[row] = o.logp;
            p.entropy_out[row] = o.H;
            p.flags_out[row] = static_cast<uint8_t>(o.flags);
            p.tok_obj[row] = o.obj;
            s_logZ2 = o.logZ2;
            s_g = o.g;
            s_y = o.y;
        }
    }
    __syncthreads();
    const float g = s_g;
    if (!RLK_CHECK(p.status, row < p.num_tokens && (g == 0.f || s_y < (uint32_t)V))) return;
    if (g == 0.f) {
        float zero[VEC];
#pragma unroll
        for (int k = 0; k < VEC; ++k) zero[k] = 0.f;
        for (int k = threadIdx.x; k < nvec; k += kRowThreads) VT::store(dz + (size_t)k * 16, zero);
        if (tail0 + (int)threadIdx.x < V) VT::store1(dz, tail0 + threadIdx.x, 0.f);
        return;
    }
    const float nlz2 = -s_logZ2;
    const float c = -g;
    const int y = (int)s_y;  // g != 0 implies a valid target
    // Pass 2 walks this thread's groups in reverse: the ones pass 1 loaded last are the likeliest
    // to still be in L1 / L2; with staging, the groups past the shared-memory prefix first.
    const int k0 = kStage ? stage_vecs : (int)threadIdx.x;
    const int k_last = (int)threadIdx.x < nvec ? (int)threadIdx.x + ((nvec - 1 - (int)threadIdx.x) / kRowThreads) * kRowThreads : -1;
#pragma unroll kUnroll
    for (int k = k_last; k >= k0; k -= kRowThreads) {
        float x[VEC];
        VT::load_last(z + (size_t)k * 16, x);
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const float pr = ex2_approx(fmaf(x[j], kLog2e, nlz2));
            x[j] = (k * VEC + j == y) ? g * (1.f - pr) : c * pr;
        }
        VT::store(dz + (size_t)k * 16, x);
    }
    if (kStage) {
        const int kp_last = (int)threadIdx.x < stage_vecs ? (int)threadIdx.x + ((stage_vecs - 1 - (int)threadIdx.x) / kRowThreads) * kRowThreads : -1;
#pragma unroll kUnroll
        for (int k = kp_last; k >= (int)threadIdx.x; k -= kRowThreads) {
            float x[VEC];
            decode16<T>(s_row[k], x);
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                const float pr = ex2_approx(fmaf(x[j], kLog2e, nlz2));
                x[j] = (k * VEC + j == y) ? g * (1.f - pr) : c * pr;
            }
            VT::store(dz + (size_t)k * 16, x);
        }
    }
    if (tail0 + (int)threadIdx.x < V) {
        const int v = tail0 + threadIdx.x;
        const float pr = ex2_approx(fmaf(VT::load1(z, v), kLog2e, nlz2));
        VT::store1(dz, v, v == y ? g * (1.f - pr) : c * pr);
    }
}

// The entropy of the rows the row kernel marked (rows that hold -inf logits): one pass over
// the row with every term of probability 0 left out (0 log 0 = 0), per-thread strided order
// and a fixed block tree; the mark is cleared. The blocks scan contiguous ranges of marks.
template <typename T>
__global__ void __launch_bounds__(256) entropy_fix_kernel(RowParams p) {
    using VT = VecTraits<T>;
    constexpr int VEC = VT::kElems;
    __shared__ uint8_t s_mark[256];
    __shared__ RowStats2 s_warp[8];
    const int T_ = p.num_tokens, V = p.vocab, nvec = V / VEC, tail0 = nvec * VEC;
    const int per = (T_ + (int)gridDim.x - 1) / (int)gridDim.x;
    const int r_begin = (int)blockIdx.x * per, r_end = min(T_, r_begin + per);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int base = r_begin; base < r_end; base += 256) {
        const int r = base + (int)threadIdx.x;
        const uint8_t m = r < r_end ? p.fix_rows[r] : 0;
        s_mark[threadIdx.x] = m;
        if (!__syncthreads_or(m)) continue;
        for (int i = 0; i < 256 && base + i < r_end; ++i) {
            if (!s_mark[i]) continue;  // block-uniform
            const int row = base + i;
            const char *z = reinterpret_cast<const char *>(p.logits) + (size_t)row * p.ld_logits * sizeof(T);
            RowStats2 st = empty_stats();
            auto add = [&](float x) {
                if (x == -INFINITY) return;
                const float x2 = x * kLog2e;
                if (x2 > st.m2) {
                    if (st.m2 != -INFINITY) {
                        const float dm = st.m2 - x2;
                        const float f = ex2_approx(dm);
                        st.u2 = f * fmaf(dm, st.s, st.u2);
                        st.s = f * st.s;
                    }
                    st.m2 = x2;
                }
                const float d2 = fmaf(x, kLog2e, -st.m2);
                const float e = ex2_approx(d2);
                st.s += e;
                if (e > 0.f) st.u2 = fmaf(e, d2, st.u2);
            };
            for (int k = threadIdx.x; k < nvec; k += 256) {
                float x[VEC];
                VT::load(z + (size_t)k * 16, x);
#pragma unroll
                for (int j = 0; j < VEC; ++j) add(x[j]);
            }
            if (tail0 + (int)threadIdx.x < V) add(VT::load1(z, tail0 + threadIdx.x));
            st = warp_merge_stats2(st);
            if (lane == 0) s_warp[warp] = st;
            __syncthreads();
            if (warp == 0) {
                RowStats2 w = lane < 8 ? s_warp[lane] : empty_stats();
                w = warp_merge_stats2(w);
                if (lane == 0) {
                    p.entropy_out[row] = (log2f(w.s) - w.u2 / w.s) * kLn2;
                    p.fix_rows[row] = 0;
                }
            }
            __syncthreads();
        }
        __syncthreads();
    }
}

template <typename T>
cudaError_t launch_fix_for(const RowParams &p, cudaStream_t stream) {
    const int grid = p.num_tokens < 608 ? p.num_tokens : 608;
    entropy_fix_kernel<T><<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_for(const RowParams &p, cudaStream_t stream) {
    if ((size_t)p.vocab * sizeof(T) <= kShortRowBytes) {
        row_loss_twopass_kernel<T, 256, false><<<p.num_tokens, 256, 0, stream>>>(p, 0);
        return cudaGetLastError();
    }
    // per device, once: the shared-memory opt-in (host threads may launch on different devices at
    // the same time)
    static std::mutex mu;
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= 64 || !configured[dev]) {
            e = cudaFuncSetAttribute(row_loss_twopass_kernel<T, 1024, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kStageBytes);
            if (e != cudaSuccess) return e;
            if (dev < 64) configured[dev] = true;
        }
    }
    const int nvec = p.vocab / (16 / (int)sizeof(T));
    const int stage_vecs = std::min(nvec, kStageBytes / 16);
    row_loss_twopass_kernel<T, 1024, true><<<p.num_tokens, 1024, (size_t)stage_vecs * 16, stream>>>(p, stage_vecs);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_row_loss(const RowParams &p, int dtype, cudaStream_t stream) {
    if (p.num_tokens == 0) return cudaSuccess;
    return dtype == RL_F32 ? launch_for<float>(p, stream) : launch_for<__nv_bfloat16>(p, stream);
}

cudaError_t launch_entropy_fix(const RowParams &p, int dtype, cudaStream_t stream) {
    if (p.num_tokens == 0) return cudaSuccess;
    return dtype == RL_F32 ? launch_fix_for<float>(p, stream) : launch_fix_for<__nv_bfloat16>(p, stream);
}

}  // namespace rlk
