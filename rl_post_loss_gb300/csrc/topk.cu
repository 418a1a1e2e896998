// Deterministic top-k over DSA indexer scores ("GLM-5: from Vibe Coding to
// Agentic Engineering", section 3.2, "DSA RL insights": the indexer keeps the
// k = 2048 best-scoring key positions of every query, and the top-k used in RL
// must be deterministic; a non-deterministic CUDA top-k collapsed RL).
//
// The selection is the first k positions of a row under one total order: NaN
// above every number, then larger score, then lower position; -0 and +0 tie.
// Scores map to 32-bit keys whose unsigned order is that order's score part.
//
// Design: one CTA per row at a time, one pass over the row in HBM. Any prefix of the
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
// bit-identical from run to run. All counts are integers. The CTAs are
// persistent (two per SM); thread 0 keeps two 16 KB tiles in flight with bulk
// copies (TMA) into a shared-memory ring, completing on mbarriers whose waits
// are bounded, and runs ahead into the next row while this one is finished.
#include <algorithm>

#include "common.cuh"
#include "scan_select.cuh"
#include "ptx.cuh"

namespace rlk {

namespace {

constexpr int kThreads = 512;
constexpr int kPer = 8;                 // scores per thread per tile (two float4)
constexpr int kTile = kThreads * kPer;  // 4096
constexpr int kCap = 8192;              // buffer entries
constexpr int kBins = 2048;
constexpr int kStages = 2;              // tiles in flight per CTA (16 KB each)
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
    float ring[kStages][kTile];  // tiles of scores, filled by bulk copies
    uint32_t key[kCap];
    uint32_t idx[kCap];
    uint32_t hist[kBins];
    unsigned long long full[kStages];  // mbarriers: a tile has landed
    uint32_t warp_tot[kThreads / 32];
    int count;      // entries in the buffer
    int found_bin;  // result of the last histogram search
    int found_before;
    int failed;     // a bounded wait ran out
    int broken;     // an internal check failed (the row's result is invalid; no access left its array)
};

// hist[digit] += 1 for every lane with `valid`, one atomic per distinct digit of the warp (the
// scores tie often, so many lanes share a digit). All 32 lanes must call it.
__device__ __forceinline__ void hist_add_warp(uint32_t *hist, uint32_t digit, bool valid) {
    const unsigned peers = __match_any_sync(kFull, valid ? digit : 0xffffffffu);
    if (valid && (threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[digit], (uint32_t)__popc(peers));
}

// Finds, over hist[0..kBins), the bin b at which the running count (from the top bin down when
// `from_top`, from bin 0 up otherwise) first reaches `target`; stores b and the count of the bins
// passed before it. Needs target <= total. Block-wide; ends with a barrier.
__device__ void find_bin(TopkSmem &s, uint32_t target, bool from_top) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s.found_bin = -1;  // stays -1 if no bin reaches the target (a broken invariant)
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
__device__ uint64_t compact(TopkSmem &s, int target, int limit, bool exact, int idx_bits) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cnt = s.count;
    // Every key shares the bits above the highest bit where the smallest and the largest differ
    // (after the first compaction they all lie above the bound), so the radix starts below them.
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    for (int i = tid; i < cnt; i += kThreads) {
        const uint32_t k = s.key[i];
        kmin = min(kmin, k);
        kmax = max(kmax, k);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        kmin = min(kmin, __shfl_xor_sync(kFull, kmin, off));
        kmax = max(kmax, __shfl_xor_sync(kFull, kmax, off));
    }
    if (lane == 0) {
        s.hist[warp] = kmin;
        s.hist[kThreads / 32 + warp] = kmax;
    }
    __syncthreads();
    for (int w = 0; w < kThreads / 32; ++w) {
        kmin = min(kmin, s.hist[w]);
        kmax = max(kmax, s.hist[kThreads / 32 + w]);
    }
    __syncthreads();
    const uint32_t diff = kmin ^ kmax;
    // the key prefix fixed so far, and how many buffer entries lie strictly above it
    int shift = diff ? 32 - __clz(diff) : 0;  // bits of the key still open: the prefix covers key >> shift
    uint32_t prefix = shift >= 32 ? 0u : (kmax >> shift);
    int above = 0;
    int kept = cnt;
    uint64_t bound = shift >= 32 ? 0u : ((uint64_t)prefix << shift);
    bool resolved = false;
    while (shift > 0 && !resolved) {
        const int w = min(11, shift);
        const int sh = shift - w;
        for (int b = tid; b < kBins; b += kThreads) s.hist[b] = 0u;
        __syncthreads();
        for (int i0 = tid & ~31; i0 < cnt; i0 += kThreads) {  // warp-uniform trip count
            const int i = i0 + (tid & 31);
            const uint32_t k = i < cnt ? s.key[i] : 0u;
            const bool in = i < cnt && (shift >= 32 || (k >> shift) == prefix);
            hist_add_warp(s.hist, (k >> sh) & ((1u << w) - 1u), in);
        }
        __syncthreads();
        find_bin(s, (uint32_t)(target - above), true);
        if (s.found_bin < 0 && tid == 0) s.broken = 1;
        const uint32_t d = (uint32_t)max(s.found_bin, 0);
        const int before = s.found_before;  // entries in the open range above the chosen digit
        const int in_bin = (int)s.hist[d];
        __syncthreads();
        prefix = (shift >= 32 ? 0u : (prefix << w)) | d;
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
            int ishift = idx_bits, ibelow = 0;  // positions are below 2^idx_bits
            while (ishift > 0) {
                const int w = min(11, ishift);
                const int sh = ishift - w;
                for (int b = tid; b < kBins; b += kThreads) s.hist[b] = 0u;
                __syncthreads();
                for (int i0 = tid & ~31; i0 < cnt; i0 += kThreads) {
                    const int i = i0 + (tid & 31);
                    const bool eq = i < cnt && s.key[i] == key_star;
                    const uint32_t ix = eq ? s.idx[i] : 0u;
                    const bool in = eq && (ishift >= 32 || (ix >> ishift) == ipre);
                    hist_add_warp(s.hist, (ix >> sh) & ((1u << w) - 1u), in);
                }
                __syncthreads();
                find_bin(s, (uint32_t)(need - ibelow), false);
                if (s.found_bin < 0 && tid == 0) s.broken = 1;
                ipre = (ishift >= 32 ? 0u : (ipre << w)) | (uint32_t)max(s.found_bin, 0);
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
        if (((keepm >> j) & 1u) && pos < kCap) {
            s.key[pos] = mk[j];
            s.idx[pos] = mi[j];
            ++pos;
        }
    }
    __syncthreads();
    return resolved ? bound : (uint64_t)key_star + 1u;
}

// a comes before b in the output order
__device__ __forceinline__ bool out_first(uint32_t ka, uint32_t ia, uint32_t kb, uint32_t ib, bool by_score) {
    return by_score ? (ka > kb || (ka == kb && ia < ib)) : (ia < ib);
}

// The same bitonic network for n2 = kThreads * E entries with E per thread in registers: strides
// below E inside a thread, below 32 E by warp shuffles, and only the wider strides through shared
// memory (one barrier each). Thread t holds entries [E t, E t + E).
template <int E>
__device__ void bitonic_regs(TopkSmem &s, bool by_score) {
    constexpr int n2 = kThreads * E;
    const int tid = threadIdx.x;
    uint32_t k[E], ix[E];
#pragma unroll
    for (int j = 0; j < E; ++j) {
        k[j] = s.key[E * tid + j];
        ix[j] = s.idx[E * tid + j];
    }
    bool in_regs = true;
#pragma unroll
    for (int size = 2; size <= n2; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (stride >= 32 * E) {  // across warps: through shared memory
                if (in_regs) {
#pragma unroll
                    for (int j = 0; j < E; ++j) {
                        s.key[E * tid + j] = k[j];
                        s.idx[E * tid + j] = ix[j];
                    }
                    in_regs = false;
                }
                __syncthreads();
                for (int t = tid; t < n2 / 2; t += kThreads) {
                    const int i = 2 * t - (t & (stride - 1));
                    const int jj = i + stride;
                    const bool up = (i & size) == 0;
                    const uint32_t ka = s.key[i], kb = s.key[jj], ia = s.idx[i], ib = s.idx[jj];
                    if (out_first(ka, ia, kb, ib, by_score) != up) {
                        s.key[i] = kb;
                        s.key[jj] = ka;
                        s.idx[i] = ib;
                        s.idx[jj] = ia;
                    }
                }
                continue;
            }
            if (!in_regs) {
                __syncthreads();
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    k[j] = s.key[E * tid + j];
                    ix[j] = s.idx[E * tid + j];
                }
                in_regs = true;
            }
            if (stride >= E) {  // across lanes of the warp
                const int lmask = stride / E;
                const bool lower = ((tid & 31) & lmask) == 0;
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    const uint32_t ok = __shfl_xor_sync(kFull, k[j], lmask);
                    const uint32_t oi = __shfl_xor_sync(kFull, ix[j], lmask);
                    const int i = E * tid + j;
                    const bool up = (i & size) == 0;
                    // the lower position keeps the entry that comes first in a rising run
                    const bool mine_first = out_first(k[j], ix[j], ok, oi, by_score);
                    const bool keep_mine = (lower == up) ? mine_first : !mine_first;
                    if (!keep_mine) {
                        k[j] = ok;
                        ix[j] = oi;
                    }
                }
            } else {  // inside the thread
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    const int jp = j ^ stride;
                    if (jp > j) {
                        const int i = E * tid + j;
                        const bool up = (i & size) == 0;
                        if (out_first(k[j], ix[j], k[jp], ix[jp], by_score) != up) {
                            const uint32_t tk = k[j], ti = ix[j];
                            k[j] = k[jp];
                            ix[j] = ix[jp];
                            k[jp] = tk;
                            ix[jp] = ti;
                        }
                    }
                }
            }
        }
    }
    if (!in_regs) __syncthreads();
    else {
#pragma unroll
        for (int j = 0; j < E; ++j) {
            s.key[E * tid + j] = k[j];
            s.idx[E * tid + j] = ix[j];
        }
    }
    __syncthreads();
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

// The score test equivalent to key >= bound. mode 0: !(x < thr), thr the smallest score whose key
// reaches the bound (NaN passes it, and -0 and +0 compare equal, as their keys do); mode 1 (bound
// above the key of +inf): NaN only; mode 2 (bound above every key): nothing.
__device__ __forceinline__ void set_threshold(uint64_t bound, float &thr, int &mode) {
    mode = bound > 0xffffffffull ? 2 : (bound > 0xff800000ull ? 1 : 0);
    const uint32_t b = bound > 0xff800000ull ? 0xff800000u : (uint32_t)bound;
    if (b < 0x007fffffu) {  // at or below the key of -inf: every number
        thr = -INFINITY;
    } else {
        thr = __uint_as_float((b & 0x80000000u) ? (b & 0x7fffffffu) : ~b);
    }
}

// The valid length of row r (clamped to [0, ld]).
__device__ __forceinline__ int row_length(const TopkParams &p, int r) {
    const int n = p.lengths ? __ldg(p.lengths + r) : (int)p.ld;
    return min(max(n, 0), (int)p.ld);
}

// Persistent CTAs, each taking rows blockIdx.x, blockIdx.x + gridDim.x, ... Thread 0 keeps
// kStages tiles of 4096 scores in flight (bulk copies into a shared-memory ring, one mbarrier
// per stage), running ahead across row boundaries, and waits for each tile just before the
// barrier that ends the previous one; every thread filters the landed tile into the candidate
// buffer.
__global__ void __launch_bounds__(kThreads, 2) topk_kernel(TopkParams p) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    TopkSmem &s = *reinterpret_cast<TopkSmem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31;
    const int k = p.k;
    const int idx_bits = p.ld <= (1 << 22) ? 22 : 32;
    // producer cursor (thread 0): the next tile to copy
    int prow = blockIdx.x, ptile = 0, pn = prow < p.rows ? row_length(p, prow) : 0;
    uint32_t issued = 0u, landed = 0u;  // thread 0: tiles copied so far / known to have landed
    const uint64_t policy = ptx::policy_evict_first();
    auto issue_next = [&](int stage) {
        while (prow < p.rows && ptile * kTile >= pn) {
            prow += gridDim.x;
            ptile = 0;
            pn = prow < p.rows ? row_length(p, prow) : 0;
        }
        if (prow >= p.rows) return;
        ++issued;
        const int cnt = min(kTile, pn - ptile * kTile);
        const uint32_t bytes = (uint32_t)((cnt + 3) & ~3) * 4u;  // whole 16-byte groups: ld % 4 == 0 keeps it in the row
        const uint32_t bar = ptx::smem_u32(&s.full[stage]);
        ptx::mbar_arrive_expect_tx(bar, bytes);
        ptx::bulk_g2s(ptx::smem_u32(s.ring[stage]), p.scores + (size_t)prow * (size_t)p.ld + (size_t)ptile * kTile,
                      bytes, bar, policy);
        ++ptile;
    };
    if (tid == 0) {
        for (int st = 0; st < kStages; ++st) ptx::mbar_init(ptx::smem_u32(&s.full[st]), 1);
        ptx::fence_mbar_init();
        s.failed = 0;
        s.broken = 0;
    }
    __syncthreads();
    // Only thread 0 waits for a tile, just before a barrier: the barrier then releases everybody with
    // the tile in shared memory (no other thread spins on the mbarrier).
    auto wait_tile = [&](uint32_t gi) {
        if (gi >= issued) return;
        if (!s.failed && !ptx::mbar_wait(ptx::smem_u32(&s.full[gi % kStages]), (gi / kStages) & 1u)) {
            s.failed = 1;
            if (p.status) raise_status(p.status, RL_ERR_TIMEOUT);
        }
        if (!s.failed) landed = gi + 1u;
    };
    if (tid == 0) {
        for (int st = 0; st < kStages; ++st) issue_next(st);
        wait_tile(0u);
    }

    uint32_t g = 0;  // tiles consumed by this CTA
    for (int row = blockIdx.x; row < p.rows; row += gridDim.x) {
        const float *x = p.scores + (size_t)row * (size_t)p.ld;
        const int nraw = p.lengths ? __ldg(p.lengths + row) : (int)p.ld;
        if (tid == 0 && p.status && (nraw < 0 || nraw > p.ld)) raise_status(p.status, RL_ERR_SEQLENS);
        const int n = row_length(p, row);
        const int kk = min(k, n);
        if (tid == 0) s.count = 0;
        __syncthreads();
        uint64_t bound = 0u;  // incoming scores are kept when key >= bound
        float thr = -INFINITY;  // the same test on the score itself
        int mode = 0;
        const int ntiles = (n + kTile - 1) / kTile;
        for (int t = 0; t < ntiles; ++t, ++g) {
            const int st = (int)(g % kStages);
            const float4 *tile4 = reinterpret_cast<const float4 *>(s.ring[st]);
            // keep a score when its key reaches the bound: one float compare (NaN passes !(x < thr))
            float vals[kPer];
            uint32_t keepm = 0u;
#pragma unroll
            for (int j = 0; j < kPer / 4; ++j) {
                const float4 v = tile4[j * kThreads + tid];
                vals[4 * j] = v.x, vals[4 * j + 1] = v.y, vals[4 * j + 2] = v.z, vals[4 * j + 3] = v.w;
            }
            if (mode == 0 && (t + 1) * kTile <= n) {  // a full tile and a plain threshold: one compare per score
#pragma unroll
                for (int q = 0; q < kPer; ++q) keepm |= (uint32_t)!(vals[q] < thr) << q;
            } else {
#pragma unroll
                for (int q = 0; q < kPer; ++q) {
                    const int e = t * kTile + 4 * ((q >> 2) * kThreads + tid) + (q & 3);
                    const bool keep = e < n && (mode == 0 ? !(vals[q] < thr) : (mode == 1 && isnan(vals[q])));
                    keepm |= (uint32_t)keep << q;
                }
            }
            int after_add = 0;  // the buffer count right after this warp's append
            if (__any_sync(kFull, keepm != 0u)) {
                // one atomic per warp: an exclusive scan of the lanes' counts
                const int c = __popc(keepm);
                int incl = c;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int o = __shfl_up_sync(kFull, incl, off);
                    if (lane >= off) incl += o;
                }
                int base = 0;
                if (lane == 31) base = atomicAdd(&s.count, incl);
                base = __shfl_sync(kFull, base, 31);
                after_add = base + __shfl_sync(kFull, incl, 31);
                int pos = base + incl - c;
#pragma unroll
                for (int q = 0; q < kPer; ++q) {
                    if (((keepm >> q) & 1u) && pos < kCap) {
                        s.key[pos] = order_key(vals[q]);
                        s.idx[pos] = (uint32_t)(t * kTile + 4 * ((q >> 2) * kThreads + tid) + (q & 3));
                        ++pos;
                    }
                }
            }
            if (tid == 0) wait_tile(g + 1u);
            // The stage is free again and the next tile has landed. Whether to compact is decided by
            // the barrier itself (the count passed the trigger iff some warp's append took it past):
            // a thread must not read s.count here, because a faster warp may already be appending
            // the next tile.
            const bool over = __syncthreads_or(after_add > kCap - kTile) != 0;
            if (tid == 0) issue_next(st);
            if (over) {
                // compact well below the trigger, so that many tiles fit before the next one
                bound = compact(s, k, k + (kCap - kTile - k) / 2, false, idx_bits);
                set_threshold(bound, thr, mode);
            }
        }
        // exactly the best min(k, n)
        if (s.count > kk) compact(s, kk, kk, true, idx_bits);
        // order them: pad to a power of two with entries that sort last
        int n2 = 1;
        while (n2 < kk) n2 <<= 1;
        for (int i = kk + tid; i < n2; i += kThreads) {
            s.key[i] = 0u;
            s.idx[i] = 0xffffffffu;
        }
        __syncthreads();
        if (n2 == 2 * kThreads)
            bitonic_regs<2>(s, p.order_by_score != 0);
        else if (n2 == 4 * kThreads)
            bitonic_regs<4>(s, p.order_by_score != 0);
        else if (kk > 1)
            bitonic(s, n2, p.order_by_score != 0);
        if (tid == 0 && (s.broken || s.count > kCap)) {
            if (p.status) raise_status(p.status, RL_ERR_INTERNAL);
            s.broken = 0;
        }
        int32_t *oi = p.out_idx + (size_t)row * (size_t)p.ldo;
        float *ov = p.out_val ? p.out_val + (size_t)row * (size_t)p.ldo : nullptr;
        for (int i = tid; i < k; i += kThreads) {
            if (i < kk) {
                const uint32_t key = s.key[i], ix = s.idx[i];
                oi[i] = (int32_t)ix;
                if (ov) {
                    // the score back from its key; -0 and NaN payloads were folded, so those are re-read
                    const uint32_t bits = (key & 0x80000000u) ? (key & 0x7fffffffu) : ~key;
                    ov[i] = ((bits == 0u || key == 0xffffffffu) && ix < (uint32_t)n) ? __ldg(x + ix) : __uint_as_float(bits);
                }
            } else {
                oi[i] = -1;
                if (ov) ov[i] = -INFINITY;
            }
        }
        __syncthreads();  // the buffer is reused by the next row
    }
    // after a timeout: let the copies that may still be in flight land before the CTA leaves (bounded)
    if (tid == 0 && s.failed) {
        for (uint32_t gi = landed; gi < issued; ++gi)
            ptx::mbar_wait(ptx::smem_u32(&s.full[gi % kStages]), (gi / kStages) & 1u, 100000000ull);
    }
}

}  // namespace

int topk_max_k() { return kCap - kTile; }

cudaError_t launch_topk(const TopkParams &p, cudaStream_t stream) {
    if (p.rows <= 0) return cudaSuccess;
    static int configured_dev = -1, sms = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_dev != dev) {
        e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(TopkSmem));
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        configured_dev = dev;
    }
    const int grid = std::min(p.rows, 2 * sms);  // persistent: two CTAs per SM
    topk_kernel<<<grid, kThreads, sizeof(TopkSmem), stream>>>(p);
    return cudaGetLastError();
}

}  // namespace rlk
