// Row step of the fused projection path: for every row of a chunk, merge the
// per-tile softmax statistics written by the projection GEMM (in tile order,
// so the result does not depend on scheduling), finish the token objective of
// Eq. (1) ("GLM-5: from Vibe Coding to Agentic Engineering", section 3.2) and
// write dZ = g (1[v == y] - softmax(z)_v) in bf16 -- one read of the fp32
// logits chunk, one write of dZ.
#include "common.cuh"
#include "proj.cuh"

namespace rlk {

namespace {

constexpr int kThreads = 1024;

__global__ void __launch_bounds__(kThreads) proj_rows_kernel(ProjRowParams p) {
    __shared__ RowStats2 warp_stats[kThreads / 32];
    __shared__ float s_logZ2, s_g;
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
        }
    }
    __syncthreads();
    const float g = s_g;
    const int V = p.vocab;
    const float *z = p.z + (size_t)r * p.ldz;
    __nv_bfloat16 *dz = reinterpret_cast<__nv_bfloat16 *>(p.dz) + (size_t)r * p.lddz;
    const int nvec = V / 4;
    if (g == 0.f) {
        for (int k = threadIdx.x; k < nvec; k += kThreads)
            __stcs(reinterpret_cast<uint2 *>(dz + 4 * k), make_uint2(0u, 0u));
        for (int v = nvec * 4 + threadIdx.x; v < V; v += kThreads) dz[v] = __float2bfloat16_rn(0.f);
        return;
    }
    const float nlz2 = -s_logZ2, c = -g;
    const int y = (int)s_y;
    for (int k = threadIdx.x; k < nvec; k += kThreads) {
        const float4 v = __ldcs(reinterpret_cast<const float4 *>(z + 4 * k));
        float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float pr = ex2_approx(fmaf(x[j], kLog2e, nlz2));
            x[j] = (4 * k + j == y) ? g * (1.f - pr) : c * pr;
        }
        __stcs(reinterpret_cast<uint2 *>(dz + 4 * k), make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3])));
    }
    for (int v = nvec * 4 + threadIdx.x; v < V; v += kThreads) {
        const float pr = ex2_approx(fmaf(z[v], kLog2e, nlz2));
        dz[v] = __float2bfloat16_rn(v == y ? g * (1.f - pr) : c * pr);
    }
}

}  // namespace

cudaError_t launch_proj_rows(const ProjRowParams &p, cudaStream_t stream) {
    if (p.rows <= 0) return cudaSuccess;
    proj_rows_kernel<<<p.rows, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace rlk
