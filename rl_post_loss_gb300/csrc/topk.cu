// Deterministic top-k over DSA indexer scores ("GLM-5: from Vibe Coding to
// Agentic Engineering", section 3.2, "DSA RL insights": the indexer keeps the
// k = 2048 best-scoring key positions of every query, and the top-k used in RL
// must be deterministic; a non-deterministic CUDA top-k collapsed RL).
//
// The selection is the first k positions of a row under one total order: NaN
// above every number, then larger score, then lower position; -0 and +0 tie.
// Scores map to 32-bit keys whose unsigned order is that order's score part.
//
// Design: one CTA per row, one pass over the row in HBM. Any prefix of the
// row bounds the final selection: an element that is not among the k best of
// the prefix seen so far (in the total order) cannot be among the k best of
// the row. So the CTA streams the row in tiles of 4096 scores and appends to
// a shared-memory buffer only the scores whose key reaches a lower bound L;
// when the buffer fills, a radix select over the buffer (11, 11 and 10 bits of
// the key, then the position for ties) raises L and drops what can no longer
// be selected. At the end the same select, run to the exact k-th element, keeps
// exactly min(k, n) entries, and a bitonic sort in shared memory orders them
// (by score, ties by position, or by position). The buffer's order of arrival
// (shared-memory atomics) never decides anything: the kept set is defined by
// the total order and the output order by the sort, so the result is
// bit-identical from run to run. All counts are integers.
#include "common.cuh"

namespace rlk {

namespace {

constexpr int kThreads = 512;
constexpr int kPer = 8;                 // scores per thread per tile (two float4)
constexpr int kTile = kThreads * kPer;  // 4096
constexpr int kCap = 8192;              // buffer entries
constexpr int kBins = 2048;
constexpr unsigned kFull = 0xffffffffu;

// Unsigned order = score order; NaN above +inf; -0 folded onto +0. Every number maps to >= 0x007fffff,
// so key 0 is free for padding.
__device__ __forceinline__ uint32_t order_key(float x) {
    uint32_t b = __float_as_uint(x);
    if ((b & 0x7fffffffu) > 0x7f800000u) return 0xffffffffu;
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

struct TopkSmem {
    uint32_t key[kCap];
    uint32_t idx[kCap];
    uint32_t hist[kBins];
    uint32_t warp_tot[kThreads / 32];
    int count;      // entries in the buffer
    int found_bin;  // result of the last histogram search
    int found_before;
};

// Finds, over hist[0..kBins), the bin b at which the running count (from the top bin down when
// `from_top`, from bin 0 up otherwise) first reaches `target`; stores b and the count of the bins
// passed before it. Needs target <= total. Block-wide; ends with a barrier.
__device__ void find_bin(TopkSmem &s, uint32_t target, bool from_top) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int per = kBins / kThreads;  // 4 bins per thread
    // thread t owns a run of 4 bins; in scan order, the runs go t = 0, 1, ... (from_top: highest bins first)
    const int base = from_top ? (kBins - per * (tid + 1)) : per * tid;
    uint32_t h[per], local = 0u;
#pragma unroll
    for (int i = 0; i < per; ++i) {
        h[i] = s.hist[from_top ? base + per - 1 - i : base + i];  // h[0] first in scan order
        local += h[i];
    }
    // exclusive prefix of `local` over threads in scan order
    uint32_t incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) s.warp_tot[warp] = incl;
    __syncthreads();
    uint32_t before = 0u;
    for (int w = 0; w < warp; ++w) before += s.warp_tot[w];
    uint32_t run = before + incl - local;
#pragma unroll
    for (int i = 0; i < per; ++i) {
        if (run < target && run + h[i] >= target) {
            s.found_bin = from_top ? base + per - 1 - i : base + i;
            s.found_before = (int)run;
        }
        run += h[i];
    }
    __syncthreads();
}

// Reduces the buffer to its best entries. With `exact`, keeps exactly `target` entries (the first
// `target` in the total order); otherwise keeps the entries whose key reaches a lower bound, at
// least `target` of them and at most `limit`. Returns the new lower bound for incoming scores
// (as a 64-bit value: 2^32 admits nothing). Block-wide.
__device__ uint64_t compact(TopkSmem &s, int target, int limit, bool exact) {
    const int tid = threadIdx.x;
    const int cnt = s.count;
    // the key prefix fixed so far, and how many buffer entries lie strictly above it
    uint32_t prefix = 0u;
    int above = 0;
    int shift = 32;  // bits of the key still open: the prefix covers key >> shift
    int kept = cnt;
    uint64_t bound = 0u;
    bool resolved = false;
    for (int level = 0; level < 3 && !resolved; ++level) {
        const int w = level == 2 ? 10 : 11;
        const int sh = shift - w;
        for (int b = tid; b < kBins; b += kThreads) s.hist[b] = 0u;
        __syncthreads();
        for (int i = tid; i < cnt; i += kThreads) {
            const uint32_t k = s.key[i];
            if (shift == 32 || (k >> shift) == prefix) atomicAdd(&s.hist[(k >> sh) & ((1u << w) - 1u)], 1u);
        }
        __syncthreads();
        find_bin(s, (uint32_t)(target - above), true);
        const uint32_t d = (uint32_t)s.found_bin;
        const int before = s.found_before;  // entries in the open range above the chosen digit
        const int in_bin = (int)s.hist[d];
        __syncthreads();
        prefix = (shift == 32 ? 0u : (prefix << w)) | d;
        above += before;
        shift = sh;
        kept = above + in_bin;  // everything at or above this prefix
        bound = (uint64_t)prefix << shift;
        if (!exact && kept <= limit) resolved = true;
        if (exact && kept == target) resolved = true;
    }
    uint32_t key_star = prefix;  // when every level ran, the exact threshold key
    uint32_t idx_star = 0u;
    if (!resolved) {
        // all 32 bits fixed: key_star is the key of the target-th entry; `above` entries are larger
        if (exact || kept > limit) {
            // keep only the (target - above) equal entries with the lowest positions
            const int need = target - above;
            uint32_t ipre = 0u;
            int ishift = 32, ibelow = 0;
            for (int level = 0; level < 3; ++level) {
                const int w = level == 2 ? 10 : 11;
                const int sh = ishift - w;
                for (int b = tid; b < kBins; b += kThreads) s.hist[b] = 0u;
                __syncthreads();
                for (int i = tid; i < cnt; i += kThreads) {
                    if (s.key[i] != key_star) continue;
                    const uint32_t ix = s.idx[i];
                    if (ishift == 32 || (ix >> ishift) == ipre) atomicAdd(&s.hist[(ix >> sh) & ((1u << w) - 1u)], 1u);
                }
                __syncthreads();
                find_bin(s, (uint32_t)(need - ibelow), false);
                ipre = (ishift == 32 ? 0u : (ipre << w)) | (uint32_t)s.found_bin;
                ibelow += s.found_before;
                ishift = sh;
                __syncthreads();
            }
            idx_star = ipre;
            kept = target;
        }
        bound = (uint64_t)key_star + 1u;  // incoming scores have later positions: equal keys rank below
    }
    // compaction: every thread takes its entries into registers, then writes back the kept ones
    constexpr int kMine = kCap / kThreads;
    uint32_t mk[kMine], mi[kMine];
    uint32_t keepm = 0u;
#pragma unroll
    for (int j = 0; j < kMine; ++j) {
        const int i = j * kThreads + tid;
        mk[j] = i < cnt ? s.key[i] : 0u;
        mi[j] = i < cnt ? s.idx[i] : 0u;
        bool keep;
        if (resolved)
            keep = (uint64_t)mk[j] >= bound;
        else
            keep = mk[j] > key_star || (mk[j] == key_star && mi[j] <= idx_star);
        keepm |= (uint32_t)(i < cnt && keep) << j;
    }
    __syncthreads();
    if (tid == 0) s.count = 0;
    __syncthreads();
    int pos = atomicAdd(&s.count, __popc(keepm));
#pragma unroll
    for (int j = 0; j < kMine; ++j) {
        if ((keepm >> j) & 1u) {
            s.key[pos] = mk[j];
            s.idx[pos] = mi[j];
            ++pos;
        }
    }
    __syncthreads();
    return resolved ? bound : (uint64_t)key_star + 1u;
}

// Bitonic sort of s.key/s.idx[0..n2) (n2 a power of two): by (key desc, idx asc) or by idx asc.
__device__ void bitonic(TopkSmem &s, int n2, bool by_score) {
    const int tid = threadIdx.x;
    for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t = tid; t < n2 / 2; t += kThreads) {
                const int i = 2 * t - (t & (stride - 1));
                const int j = i + stride;
                const bool up = (i & size) == 0;  // this run ascends in the output order
                const uint32_t ka = s.key[i], kb = s.key[j], ia = s.idx[i], ib = s.idx[j];
                const bool a_first = by_score ? (ka > kb || (ka == kb && ia < ib)) : (ia < ib);
                if (a_first != up) {
                    s.key[i] = kb;
                    s.key[j] = ka;
                    s.idx[i] = ib;
                    s.idx[j] = ia;
                }
            }
            __syncthreads();
        }
    }
}

__global__ void __launch_bounds__(kThreads, 2) topk_kernel(TopkParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    TopkSmem &s = *reinterpret_cast<TopkSmem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31;
    const int row = blockIdx.x;
    const float *x = p.scores + (size_t)row * (size_t)p.ld;
    int n = p.lengths ? __ldg(p.lengths + row) : (int)p.ld;
    if (n < 0 || n > p.ld) {
        if (tid == 0 && p.status) raise_status(p.status, RL_ERR_SEQLENS);
        n = min(max(n, 0), (int)p.ld);
    }
    const int k = p.k, kk = min(k, n);
    if (tid == 0) s.count = 0;
    __syncthreads();

    uint64_t bound = 0u;  // incoming scores are kept when key >= bound
    const int ntiles = (n + kTile - 1) / kTile;
    float4 cur[2], nxt[2];
    auto load_tile = [&](int t, float4 (&v)[2]) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int e = t * kTile + 4 * (j * kThreads + tid);
            v[j] = e < n ? __ldcs(reinterpret_cast<const float4 *>(x + e)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    if (ntiles > 0) load_tile(0, cur);
    for (int t = 0; t < ntiles; ++t) {
        if (t + 1 < ntiles) load_tile(t + 1, nxt);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int e = t * kTile + 4 * (j * kThreads + tid);
            const float v4[4] = {cur[j].x, cur[j].y, cur[j].z, cur[j].w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t key = order_key(v4[u]);
                const bool keep = e + u < n && (uint64_t)key >= bound;
                const unsigned m = __ballot_sync(kFull, keep);
                if (m) {
                    int base = 0;
                    if (lane == __ffs(m) - 1) base = atomicAdd(&s.count, __popc(m));
                    base = __shfl_sync(kFull, base, __ffs(m) - 1);
                    if (keep) {
                        const int pos = base + __popc(m & ((1u << lane) - 1u));
                        s.key[pos] = key;
                        s.idx[pos] = (uint32_t)(e + u);
                    }
                }
            }
        }
        __syncthreads();
        if (s.count > kCap - kTile) bound = compact(s, k, kCap - kTile, false);
        if (t + 1 < ntiles) {
            cur[0] = nxt[0];
            cur[1] = nxt[1];
        }
    }
    // exactly the best min(k, n)
    if (s.count > kk) compact(s, kk, kk, true);
    // order them: pad to a power of two with entries that sort last
    int n2 = 1;
    while (n2 < kk) n2 <<= 1;
    for (int i = kk + tid; i < n2; i += kThreads) {
        s.key[i] = 0u;
        s.idx[i] = 0xffffffffu;
    }
    __syncthreads();
    if (kk > 1) bitonic(s, n2, p.order_by_score != 0);
    int32_t *oi = p.out_idx + (size_t)row * (size_t)p.ldo;
    float *ov = p.out_val ? p.out_val + (size_t)row * (size_t)p.ldo : nullptr;
    for (int i = tid; i < k; i += kThreads) {
        if (i < kk) {
            const uint32_t ix = s.idx[i];
            oi[i] = (int32_t)ix;
            if (ov) ov[i] = __ldg(x + ix);
        } else {
            oi[i] = -1;
            if (ov) ov[i] = -INFINITY;
        }
    }
}

}  // namespace

int topk_max_k() { return kCap - kTile; }

cudaError_t launch_topk(const TopkParams &p, cudaStream_t stream) {
    if (p.rows <= 0) return cudaSuccess;
    static int configured_dev = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_dev != dev) {
        e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(TopkSmem));
        if (e != cudaSuccess) return e;
        configured_dev = dev;
    }
    topk_kernel<<<p.rows, kThreads, sizeof(TopkSmem), stream>>>(p);
    return cudaGetLastError();
}

}  // namespace rlk
