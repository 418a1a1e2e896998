// The fused row kernel: log-softmax statistics, target gather, entropy, the
// token objective of Eq. (1) ("GLM-5: from Vibe Coding to Agentic
// Engineering", section 3.2) and dL/dlogits, one logits row per block.
//
// Per row t (z = logits row, V entries):
//   M = max z, S = sum e^{z-M}, U = sum e^{z-M} (z-M)
//   logZ = M + ln S, logp = z_y - logZ, H = ln S - U/S
//   g = dL/dlogp from the token objective (rho, pop, r, clip)
//   dz_v = g (1[v == y] - e^{z_v - logZ}), rounded once to the logits dtype
// Rows with g == 0 (masked, popped, clipped, zero advantage) are written as
// +0.0 without evaluating the softmax a second time.
//
// This version reads each row twice (statistics, then gradient; the second
// read is mostly served by L2) with 16-byte vector loads and stores.
#include "common.cuh"

namespace rlk {

namespace {

constexpr int kRowThreads = 512;

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
    __device__ __forceinline__ static void store(void *p, const float (&x)[4]) {
        *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
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
    __device__ __forceinline__ static void store(void *p, const float (&x)[8]) {
        uint4 v;
        v.x = pack_bf16x2(x[0], x[1]); v.y = pack_bf16x2(x[2], x[3]);
        v.z = pack_bf16x2(x[4], x[5]); v.w = pack_bf16x2(x[6], x[7]);
        *reinterpret_cast<uint4 *>(p) = v;
    }
    __device__ __forceinline__ static void store1(void *p, int64_t v, float x) {
        reinterpret_cast<__nv_bfloat16 *>(p)[v] = __float2bfloat16_rn(x);
    }
};

// Fold a group of values into running statistics (rescaling once per group).
template <int N>
__device__ __forceinline__ void accumulate(RowStats &st, const float (&x)[N]) {
    float mv = x[0];
#pragma unroll
    for (int k = 1; k < N; ++k) mv = fmaxf(mv, x[k]);
    if (mv > st.m) {
        if (st.m != -INFINITY) {
            const float dm = st.m - mv;
            const float f = ex2_approx(dm * kLog2e);
            st.u = f * fmaf(dm, st.s, st.u);
            st.s = f * st.s;
        }
        st.m = mv;
    }
#pragma unroll
    for (int k = 0; k < N; ++k) {
        const float d = x[k] - st.m;
        const float e = ex2_approx(d * kLog2e);
        st.s += e;
        st.u = fmaf(e, d, st.u);
    }
}

template <typename T>
__global__ void __launch_bounds__(kRowThreads) row_loss_twopass_kernel(RowParams p) {
    using VT = VecTraits<T>;
    constexpr int VEC = VT::kElems;
    __shared__ RowStats warp_stats[kRowThreads / 32];
    __shared__ float s_logZ, s_g;
    __shared__ int s_y;

    const int row = blockIdx.x;
    const int V = p.vocab;
    const int nvec = V / VEC;
    const int tail0 = nvec * VEC;
    const char *z = reinterpret_cast<const char *>(p.logits) + (size_t)row * p.ld_logits * sizeof(T);
    char *dz = reinterpret_cast<char *>(p.dlogits) + (size_t)row * p.ld_dlogits * sizeof(T);

    // ---- pass 1: softmax statistics (fixed element-to-thread map + fixed tree)
    RowStats st{-INFINITY, 0.f, 0.f};
    for (int k = threadIdx.x; k < nvec; k += kRowThreads) {
        float x[VEC];
        VT::load(z + (size_t)k * 16, x);
        accumulate(st, x);
    }
    if (tail0 + (int)threadIdx.x < V) {
        float x[1] = {VT::load1(z, tail0 + threadIdx.x)};
        accumulate(st, x);
    }
    st = warp_merge_stats(st);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) warp_stats[warp] = st;
    __syncthreads();
    if (warp == 0) {
        RowStats w = lane < kRowThreads / 32 ? warp_stats[lane] : RowStats{-INFINITY, 0.f, 0.f};
        w = warp_merge_stats(w);
        if (lane == 0) {
            const float lnS = logf(w.s);
            const float logZ = w.m + lnS;
            const float H = lnS - w.u / w.s;
            const int t = row;
            const int i = find_seq(p.cu_seqlens, p.num_seqs, t);
            if (i < 0) raise_status(p.status, RL_ERR_SEQLENS);
            const int y = __ldg(p.targets + t);
            const bool target_ok = (y >= 0) && (y < V);
            if (!target_ok) raise_status(p.status, RL_ERR_TARGET_RANGE);
            const float zy = target_ok ? VT::load1(z, y) : 0.f;
            const bool m = (i >= 0) && (__ldg(p.mask + t) != 0);
            const float A = i >= 0 ? p.seq_adv[i] : 0.f;
            const float wt = i >= 0 ? p.seq_w[i] : 0.f;
            const TokenResult r =
                token_objective(zy, logZ, target_ok, __ldg(p.logp_old + t), __ldg(p.logp_infer + t), m, A, wt, p.c);
            if (p.logp_out) p.logp_out[t] = r.logp;
            p.entropy_out[t] = H;
            p.flags_out[t] = static_cast<uint8_t>(r.flags);
            p.tok_obj[t] = r.obj;
            s_logZ = logZ;
            s_g = r.g;
            s_y = target_ok ? y : -1;
        }
    }
    __syncthreads();
    const float g = s_g;

    // ---- pass 2: dz = g (onehot - softmax), rounded once to T
    if (g == 0.f) {
        float zero[VEC];
#pragma unroll
        for (int k = 0; k < VEC; ++k) zero[k] = 0.f;
        for (int k = threadIdx.x; k < nvec; k += kRowThreads) VT::store(dz + (size_t)k * 16, zero);
        if (tail0 + (int)threadIdx.x < V) VT::store1(dz, tail0 + threadIdx.x, 0.f);
        return;
    }
    const float nlz2 = -s_logZ * kLog2e;
    const float c = -g;
    const int y = s_y;
    for (int k = threadIdx.x; k < nvec; k += kRowThreads) {
        float x[VEC];
        VT::load(z + (size_t)k * 16, x);
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const float pr = ex2_approx(fmaf(x[j], kLog2e, nlz2));
            x[j] = (k * VEC + j == y) ? g * (1.f - pr) : c * pr;
        }
        VT::store(dz + (size_t)k * 16, x);
    }
    if (tail0 + (int)threadIdx.x < V) {
        const int v = tail0 + threadIdx.x;
        const float pr = ex2_approx(fmaf(VT::load1(z, v), kLog2e, nlz2));
        VT::store1(dz, v, v == y ? g * (1.f - pr) : c * pr);
    }
}

}  // namespace

cudaError_t launch_row_loss(const RowParams &p, int dtype, cudaStream_t stream) {
    if (p.num_tokens == 0) return cudaSuccess;
    if (dtype == RL_F32)
        row_loss_twopass_kernel<float><<<p.num_tokens, kRowThreads, 0, stream>>>(p);
    else
        row_loss_twopass_kernel<__nv_bfloat16><<<p.num_tokens, kRowThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace rlk
