// Row step of the fused projection path: for every row of a chunk, merge the
// per-tile softmax statistics written by the projection GEMM (in tile order,
// so the result does not depend on scheduling), finish the token objective of
// Eq. (1) ("GLM-5: from Vibe Coding to Agentic Engineering", section 3.2) and
// turn the chunk's scaled probabilities e_v = 2^{z_v log2e - m_b} (bf16, m_b
// the reference of v's 64-column block) into dZ = g (1[v == y] - softmax(z)_v)
// in bf16, in place: softmax(z)_v = e_v 2^{m_b - logZ2}. The target's entry
// uses its exact fp32 logit. One read and one write of a bf16 chunk.
#include "common.cuh"
#include "proj.cuh"

namespace rlk {

namespace {

constexpr int kThreads = 1024;

__global__ void __launch_bounds__(kThreads) proj_rows_kernel(ProjRowParams p) {
    __shared__ RowStats2 warp_stats[kThreads / 32];
    __shared__ float s_logZ2, s_g, s_dzy;
    __shared__ uint32_t s_y;
    const int r = blockIdx.x;
    const int t = p.row0 + r;
    if (!RLK_CHECK(p.status, r < p.rows)) return;
    const float4 *st_row = p.stats + (size_t)r * p.n_tiles;

    RowStats2 st = empty_stats();
    for (int j = threadIdx.x; j < p.n_tiles; j += kThreads) {
        const float4 v = st_row[j];
        st = merge_stats2(st, RowStats2{v.x, v.y, v.z});
    }
    st = warp_merge_stats2(st);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) warp_stats[warp] = st;
    __syncthreads();
    if (warp == 0) {
        RowStats2 w = lane < kThreads / 32 ? warp_stats[lane] : empty_stats();
        w = warp_merge_stats2(w);
        if (lane == 0) {
            const RowOut o = finish_row(w, __ldg(p.rec + t), __ldg(p.meta + t), p.c, p.teacher ? __ldg(p.teacher + t) : 0.f);
            if (!isfinite(o.logZ2)) raise_status(p.status, RL_ERR_NONFINITE);
            if (p.logp_out) p.logp_out[t] = o.logp;
            p.entropy_out[t] = o.H;
            p.flags_out[t] = static_cast<uint8_t>(o.flags);
            p.tok_obj[t] = o.obj;
            s_logZ2 = o.logZ2;
            s_g = o.g;
            s_y = o.y;
            // the target's entry from its exact logit: g (1 - p_y)
            s_dzy = o.g * (1.f - ex2_approx(fmaf(__ldg(p.rec + t).x, kLog2e, -o.logZ2)));
        }
    }
    __syncthreads();
    const float g = s_g;
    const int V = p.vocab;
    __nv_bfloat16 *pz = reinterpret_cast<__nv_bfloat16 *>(p.probs) + (size_t)r * p.ldp;
    const int ngrp = V / 8;  // 16-byte groups of 8 values; a group lies in one 64-column block
    if (g == 0.f) {
        for (int k = threadIdx.x; k < ngrp; k += kThreads) __stcs(reinterpret_cast<uint4 *>(pz + 8 * k), make_uint4(0u, 0u, 0u, 0u));
        for (int v = ngrp * 8 + threadIdx.x; v < V; v += kThreads) pz[v] = __float2bfloat16_rn(0.f);
        return;
    }
    const float lz2 = s_logZ2, c = -g, dzy = s_dzy;
    const int y = (int)s_y;
    const float *ref = reinterpret_cast<const float *>(p.refs + (size_t)r * p.n_tiles);
    for (int k = threadIdx.x; k < ngrp; k += kThreads) {
        const uint4 v = __ldcs(reinterpret_cast<const uint4 *>(pz + 8 * k));
        const float sc = c * ex2_approx(__ldg(ref + (k >> 3)) - lz2);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float a = sc * __uint_as_float(w[j] << 16), b = sc * __uint_as_float(w[j] & 0xffff0000u);
            a = (8 * k + 2 * j == y) ? dzy : a;
            b = (8 * k + 2 * j + 1 == y) ? dzy : b;
            o[j] = pack_bf16x2(a, b);
        }
        __stcs(reinterpret_cast<uint4 *>(pz + 8 * k), make_uint4(o[0], o[1], o[2], o[3]));
    }
    for (int v = ngrp * 8 + threadIdx.x; v < V; v += kThreads) {
        const float pr = __bfloat162float(pz[v]) * ex2_approx(__ldg(ref + (v >> 6)) - lz2);
        pz[v] = __float2bfloat16_rn(v == y ? dzy : c * pr);
    }
}

}  // namespace

cudaError_t launch_proj_rows(const ProjRowParams &p, cudaStream_t stream) {
    if (p.rows <= 0) return cudaSuccess;
    proj_rows_kernel<<<p.rows, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace rlk
