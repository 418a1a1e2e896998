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
// when the buffer fills, a radix select over the buffer (over the key bits
// that differ, then the position for ties) raises L and drops what can no
// longer be selected. Long rows start with L taken from a sample of the row
// rather than -inf, so most rows need no compaction at all; a row where fewer
// than k scores reach the sampled L is scanned again from -inf. At the end
// one pass of buckets over the keys' leading varying bits selects the
// min(k, n) best and orders them (by score, ties by position): each entry's
// output position is its bucket's start plus its rank within the bucket.
// Where the buckets are too uneven, or the order is by position, the radix
// select run to the exact k-th element keeps min(k, n) entries and a bucket
// ranking or a bitonic sort orders them. The buffer's order of arrival
// (shared-memory atomics) never decides anything: the kept set is defined by
// the total order and the output order by the sort, so the result is
// bit-identical from run to run. All counts are integers. The CTAs are
// persistent (two per SM) and warp-specialised: a producer warp keeps four
// 16 KB tiles in flight with bulk copies (TMA) into a shared-memory ring and
// runs ahead into the next row while this one is finished; sixteen filter
// warps do everything else, synchronising among themselves on a named
// barrier. Stages are handed over on "full" and "empty" mbarriers whose waits
// are bounded.
#include <algorithm>
#include <climits>
#include <mutex>

#include "common.cuh"
#include "scan_select.cuh"
#include "ptx.cuh"

namespace rlk {

namespace {

constexpr int kThreads = 512;           // filter threads (16 warps); one more warp issues the tile copies
constexpr int kBlock = kThreads + 32;
constexpr int kPer = 8;                 // scores per thread per tile (two float4)
constexpr int kTile = kThreads * kPer;  // 4096
constexpr int kCap = 5120;              // buffer entries
constexpr int kSlice = 512;             // positions per slice of a tile that overflowed the buffer
constexpr int kSoft = kCap - kSlice;    // a count above this compacts after the tile
constexpr int kCheck = 8;              // sampled rows: tiles between the checks of the count
constexpr int kSoftSampled = kCap - kCheck * 64;  // ... and the count that compacts at a check
constexpr int kBins = 2048;
constexpr int kStages = 4;              // tiles in flight per CTA (16 KB each)
constexpr unsigned kFull = 0xffffffffu;
// The sampled starting bound: 16 runs of 512 scores spread evenly over the row.
constexpr int kSampleRuns = 16;
constexpr int kSampleRun = 512;
constexpr int kSample = kSampleRuns * kSampleRun;  // 8192 keys, held in the (still empty) buffer's storage
constexpr int kSampleMinLen = 4 * kTile;           // shorter rows start from -inf
static_assert(kSample <= 2 * kCap, "the sample is held in the candidate buffer's storage");
static_assert(kTile == 8 * kSlice && kThreads == 4 * (kSlice / 4), "a slice is a quarter of the threads' first or second float4");

// Unsigned order = score order; NaN above +inf; -0 folded onto +0. Every number maps to >= 0x007fffff,
// so key 0 is free for padding.
__device__ __forceinline__ uint32_t order_key(float x) {
    uint32_t b = __float_as_uint(x);
    if ((b & 0x7fffffffu) > 0x7f800000u) return 0xffffffffu;
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Entries [0, keyed) hold order keys; entries appended since the last compaction hold the raw
// score bits until the next compaction (or the final selection) turns them into keys.
struct Candidates {
    uint32_t key[kCap];
    uint32_t idx[kCap];
};

// The filter warps' barriers: named barrier 1 over the kThreads filter threads (the producer warp
// never takes part).
__device__ __forceinline__ void fbar() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }
__device__ __forceinline__ int fbar_or(int pred) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\tbar.red.or.pred q, 1, %2, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred), "n"(kThreads)
        : "memory");
    return r;
}

struct TopkSmem {
    float ring[kStages][kTile];  // tiles of scores, filled by bulk copies
    union {
        Candidates cb;              // the candidate buffer
        uint32_t sample[kSample];   // at the start of a row: the sampled keys
        uint64_t packed[kCap];      // at the end of a row: the selection by bucket, then sorted (see pack_out)
    };
    uint32_t hist[kBins];
    unsigned long long full[kStages];   // mbarriers: a tile has landed
    unsigned long long empty[kStages];  // mbarriers: every filter warp is done with the stage
    uint32_t warp_tot[kThreads / 32];
    int warp_base[kThreads / 32];      // where each warp's append of the current tile started (INT_MAX: none)
    int count;      // entries in the buffer
    int keyed;      // leading entries that already hold order keys
    int found_bin;  // result of the last histogram search
    int found_before;
    int failed;     // a bounded wait ran out (read by several warps: volatile accesses)
    uint32_t issued;  // tiles the producer warp has issued
    int broken;     // an internal check failed (the row's result is invalid; no access left its array)
};

// hist[digit] += 1 when `valid`: one plain shared atomic per lane. Gathering the lanes of a warp
// that share a digit first (__match_any_sync, one atomic per distinct digit) measured slower on
// this kernel, although the scores tie often.
__device__ __forceinline__ void hist_add(uint32_t *hist, uint32_t digit, bool valid) {
    if (valid) atomicAdd(&hist[digit], 1u);
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
    fbar();
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
    fbar();
}

// Turns the raw scores appended since the last compaction into order keys. Block-wide; ends with
// a barrier, so every thread sees the new `keyed` before it can call this again.
__device__ void make_keys(TopkSmem &s) {
    const int cnt = s.count;
    for (int i = s.keyed + (int)threadIdx.x; i < cnt; i += kThreads) s.cb.key[i] = order_key(__uint_as_float(s.cb.key[i]));
    fbar();
    if (threadIdx.x == 0) s.keyed = cnt;
    fbar();
}

// The outcome of a radix descent over the first `cnt` buffer keys.
struct Descent {
    uint32_t prefix;  // the key bits fixed so far (key >> shift)
    int shift;        // key bits still open
    int above;        // entries whose key lies strictly above the prefix
    int kept;         // entries at or above the prefix
    bool resolved;    // the stopping rule was met before every bit was fixed
};

// Fixes the key from the top, up to 11 bits at a time, over the bits where the keys differ (below
// the common prefix of the smallest and the largest key, above the lowest bit that is not the same
// in every key), until at least `target` keys lie at or above the fixed prefix and, with `exact`,
// exactly `target`, otherwise at most `limit`; or until every bit is fixed (then `kept` may
// exceed the rule by keys equal to the prefix). Needs target <= cnt. Block-wide.
__device__ Descent radix_descent(TopkSmem &s, const uint32_t *keys, int cnt, int target, int limit, bool exact) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // Every key shares the bits above the highest bit where the smallest and the largest differ
    // (after the first compaction they all lie above the bound), so the radix starts below them.
    // the smallest and the largest key, and the bits in which any key differs from the first one
    const uint32_t k0 = cnt > 0 ? keys[0] : 0u;
    uint32_t kmin = 0xffffffffu, kmax = 0u, vary = 0u;
    for (int i = tid; i < cnt; i += kThreads) {
        const uint32_t k = keys[i];
        kmin = min(kmin, k);
        kmax = max(kmax, k);
        vary |= k ^ k0;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        kmin = min(kmin, __shfl_xor_sync(kFull, kmin, off));
        kmax = max(kmax, __shfl_xor_sync(kFull, kmax, off));
        vary |= __shfl_xor_sync(kFull, vary, off);
    }
    if (lane == 0) {
        s.hist[warp] = kmin;
        s.hist[kThreads / 32 + warp] = kmax;
        s.hist[2 * (kThreads / 32) + warp] = vary;
    }
    fbar();
    for (int w = 0; w < kThreads / 32; ++w) {
        kmin = min(kmin, s.hist[w]);
        kmax = max(kmax, s.hist[kThreads / 32 + w]);
        vary |= s.hist[2 * (kThreads / 32) + w];
    }
    fbar();
    const int low = vary ? __ffs(vary) - 1 : 32;  // bits below `low` are the same in every key
    const uint32_t diff = kmin ^ kmax;
    // the key prefix fixed so far, and how many buffer entries lie strictly above it
    int shift = diff ? 32 - __clz(diff) : 0;  // bits of the key still open: the prefix covers key >> shift
    uint32_t prefix = shift >= 32 ? 0u : (kmax >> shift);
    int above = 0;
    int kept = cnt;
    bool resolved = exact ? kept == target : kept <= limit;
    while (shift > low && !resolved) {
        const int w = min(11, shift - low);
        const int sh = shift - w;
        for (int b = tid; b < kBins; b += kThreads) s.hist[b] = 0u;
        fbar();
        for (int i0 = tid & ~31; i0 < cnt; i0 += kThreads) {
            const int i = i0 + (tid & 31);
            const uint32_t k = i < cnt ? keys[i] : 0u;
            const bool in = i < cnt && (shift >= 32 || (k >> shift) == prefix);
            hist_add(s.hist, (k >> sh) & ((1u << w) - 1u), in);
        }
        fbar();
        find_bin(s, (uint32_t)(target - above), true);
        if (s.found_bin < 0 && tid == 0) s.broken = 1;
        const uint32_t d = (uint32_t)max(s.found_bin, 0);
        const int before = s.found_before;  // entries in the open range above the chosen digit
        const int in_bin = (int)s.hist[d];
        fbar();
        prefix = (shift >= 32 ? 0u : (prefix << w)) | d;
        above += before;
        shift = sh;
        kept = above + in_bin;  // everything at or above this prefix
        if (!exact && kept <= limit) resolved = true;
        if (exact && kept == target) resolved = true;
    }
    if (!resolved && shift > 0) {  // only bits that every key shares are left: fix them too
        prefix = (prefix << shift) | (kmax & ((1u << shift) - 1u));
        shift = 0;
    }
    return Descent{prefix, shift, above, kept, resolved};
}

// Reduces the buffer to its best entries. With `exact`, keeps exactly `target` entries (the first
// `target` in the total order); otherwise keeps the entries whose key reaches a lower bound, at
// least `target` of them and at most `limit`. Returns the new lower bound for incoming scores
// (as a 64-bit value: 2^32 admits nothing). Block-wide.
__device__ uint64_t compact(TopkSmem &s, int target, int limit, bool exact, int idx_bits) {
    const int tid = threadIdx.x;
    make_keys(s);
    const int cnt = s.count;
    const Descent dsc = radix_descent(s, s.cb.key, cnt, target, limit, exact);
    const bool resolved = dsc.resolved;
    const int above = dsc.above;
    int kept = dsc.kept;
    uint64_t bound = (uint64_t)dsc.prefix << dsc.shift;
    uint32_t key_star = dsc.prefix;  // when every level ran, the exact threshold key
    uint32_t idx_star = 0u;
    if (!resolved) {
        // all 32 bits fixed: key_star is the key of the target-th entry; `above` entries are larger
        if (exact || kept > limit) {
            // keep only the (target - above) equal entries with the lowest positions
            const int need = target - above;
            const int ties = kept - above;  // the entries whose key is key_star
            uint32_t ipre = 0u;
            int ishift = idx_bits, ibelow = 0;  // positions are below 2^idx_bits
            if (ties <= kBins) {
                // few enough: gather their positions into the histogram's storage and take the
                // need-th smallest directly (positions are distinct, so exactly one has that rank)
                const int lane = tid & 31;
                if (tid == 0) {
                    s.found_bin = 0;
                    s.found_before = -1;  // stays -1 only if the invariant broke
                }
                fbar();
                for (int i0 = tid & ~31; i0 < cnt; i0 += kThreads) {  // warp-uniform trip count: the ballot
                    const int i = i0 + lane;
                    const bool eq = i < cnt && s.cb.key[i] == key_star;
                    const unsigned m = __ballot_sync(kFull, eq);
                    int b0 = 0;
                    if (lane == 0 && m) b0 = atomicAdd(&s.found_bin, __popc(m));
                    b0 = __shfl_sync(kFull, b0, 0);
                    if (eq) {
                        const int slot = b0 + __popc(m & ((1u << lane) - 1u));
                        if (slot < kBins) s.hist[slot] = s.cb.idx[i];
                    }
                }
                fbar();
                const int nt = min(s.found_bin, kBins);
                if (tid == 0 && nt != ties) s.broken = 1;
                for (int t = tid; t < nt; t += kThreads) {
                    const uint32_t x = s.hist[t];
                    int r = 0;
#pragma unroll 4
                    for (int j = 0; j < nt; ++j) r += s.hist[j] < x ? 1 : 0;
                    if (r == need - 1) s.found_before = (int)x;
                }
                fbar();
                if (tid == 0 && s.found_before < 0) s.broken = 1;
                ipre = (uint32_t)max(s.found_before, 0);
                ishift = 0;  // no radix passes
            }
            while (ishift > 0) {
                const int w = min(11, ishift);
                const int sh = ishift - w;
                for (int b = tid; b < kBins; b += kThreads) s.hist[b] = 0u;
                fbar();
                for (int i0 = tid & ~31; i0 < cnt; i0 += kThreads) {
                    const int i = i0 + (tid & 31);
                    const bool eq = i < cnt && s.cb.key[i] == key_star;
                    const uint32_t ix = eq ? s.cb.idx[i] : 0u;
                    const bool in = eq && (ishift >= 32 || (ix >> ishift) == ipre);
                    hist_add(s.hist, (ix >> sh) & ((1u << w) - 1u), in);
                }
                fbar();
                find_bin(s, (uint32_t)(need - ibelow), false);
                if (s.found_bin < 0 && tid == 0) s.broken = 1;
                ipre = (ishift >= 32 ? 0u : (ipre << w)) | (uint32_t)max(s.found_bin, 0);
                ibelow += s.found_before;
                ishift = sh;
                fbar();
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
        mk[j] = i < cnt ? s.cb.key[i] : 0u;
        mi[j] = i < cnt ? s.cb.idx[i] : 0u;
        bool keep;
        if (resolved)
            keep = (uint64_t)mk[j] >= bound;
        else
            keep = mk[j] > key_star || (mk[j] == key_star && mi[j] <= idx_star);
        keepm |= (uint32_t)(i < cnt && keep) << j;
    }
    fbar();
    if (tid == 0) s.count = 0;
    fbar();
    int pos = atomicAdd(&s.count, __popc(keepm));
#pragma unroll
    for (int j = 0; j < kMine; ++j) {
        if (((keepm >> j) & 1u) && pos < kCap) {
            s.cb.key[pos] = mk[j];
            s.cb.idx[pos] = mi[j];
            ++pos;
        }
    }
    fbar();
    if (tid == 0) s.keyed = s.count;
    return resolved ? bound : (uint64_t)key_star + 1u;
}

// The output order as one 64-bit value, larger first. By score: the key, then the complement of
// the position (ties to the lower position); by position: the complement of the position, then the
// key. Positions are distinct, so no two entries of a row pack to the same value.
__device__ __forceinline__ uint64_t pack_out(uint32_t key, uint32_t ix, bool by_score) {
    return by_score ? (((uint64_t)key << 32) | (uint64_t)(~ix)) : (((uint64_t)(~ix) << 32) | (uint64_t)key);
}
__device__ __forceinline__ void unpack_out(uint64_t c, bool by_score, uint32_t &key, uint32_t &ix) {
    const uint32_t hi = (uint32_t)(c >> 32), lo = (uint32_t)c;
    key = by_score ? hi : lo;
    ix = by_score ? ~lo : ~hi;
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
        k[j] = s.cb.key[E * tid + j];
        ix[j] = s.cb.idx[E * tid + j];
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
                        s.cb.key[E * tid + j] = k[j];
                        s.cb.idx[E * tid + j] = ix[j];
                    }
                    in_regs = false;
                }
                fbar();
                for (int t = tid; t < n2 / 2; t += kThreads) {
                    const int i = 2 * t - (t & (stride - 1));
                    const int jj = i + stride;
                    const bool up = (i & size) == 0;
                    const uint32_t ka = s.cb.key[i], kb = s.cb.key[jj], ia = s.cb.idx[i], ib = s.cb.idx[jj];
                    if (out_first(ka, ia, kb, ib, by_score) != up) {
                        s.cb.key[i] = kb;
                        s.cb.key[jj] = ka;
                        s.cb.idx[i] = ib;
                        s.cb.idx[jj] = ia;
                    }
                }
                continue;
            }
            if (!in_regs) {
                fbar();
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    k[j] = s.cb.key[E * tid + j];
                    ix[j] = s.cb.idx[E * tid + j];
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
    if (!in_regs) fbar();
    else {
#pragma unroll
        for (int j = 0; j < E; ++j) {
            s.cb.key[E * tid + j] = k[j];
            s.cb.idx[E * tid + j] = ix[j];
        }
    }
    fbar();
}

// Bitonic sort of s.key/s.cb.idx[0..n2) (n2 a power of two): by (key desc, idx asc) or by idx asc.
__device__ void bitonic(TopkSmem &s, int n2, bool by_score) {
    const int tid = threadIdx.x;
    for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t = tid; t < n2 / 2; t += kThreads) {
                const int i = 2 * t - (t & (stride - 1));
                const int j = i + stride;
                const bool up = (i & size) == 0;  // this run ascends in the output order
                const uint32_t ka = s.cb.key[i], kb = s.cb.key[j], ia = s.cb.idx[i], ib = s.cb.idx[j];
                const bool a_first = by_score ? (ka > kb || (ka == kb && ia < ib)) : (ia < ib);
                if (a_first != up) {
                    s.cb.key[i] = kb;
                    s.cb.key[j] = ka;
                    s.cb.idx[i] = ib;
                    s.cb.idx[j] = ia;
                }
            }
            fbar();
        }
    }
}

constexpr int kSortMax = kCap / 2;                             // entries bucket_sort takes
constexpr int kSortPer = (kSortMax + kThreads - 1) / kThreads;  // per thread
constexpr int kSortBudget = 128;  // allowed sum of squared bucket sizes, per entry

// Sorts the buffer's first n entries (n <= kSortMax) into output order through buckets of the
// leading bits in which the entries' high words (see pack_out) differ: the histogram of those
// bits gives each bucket's start (larger buckets first), the entries are scattered by bucket, and
// each entry's position is its bucket's start plus the number of entries of its bucket that come
// before it. The cost is the sum of the squared bucket sizes; when that exceeds kSortBudget n,
// nothing is written and false is returned (the caller sorts with the bitonic network). On
// success s.packed[n + i] holds the i-th entry in output order. Block-wide; ends with a barrier.
__device__ bool bucket_sort(TopkSmem &s, int n, bool by_score) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (n == 0) return true;
    // the entries, packed, and the bits in which their high words differ
    uint64_t c[kSortPer];
    const uint32_t h0 = (uint32_t)(pack_out(s.cb.key[0], s.cb.idx[0], by_score) >> 32);
    uint32_t hmin = 0xffffffffu, hmax = 0u, vary = 0u;
#pragma unroll
    for (int j = 0; j < kSortPer; ++j) {
        const int i = j * kThreads + tid;
        c[j] = i < n ? pack_out(s.cb.key[i], s.cb.idx[i], by_score) : 0ull;
        if (i < n) {
            const uint32_t h = (uint32_t)(c[j] >> 32);
            hmin = min(hmin, h);
            hmax = max(hmax, h);
            vary |= h ^ h0;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        hmin = min(hmin, __shfl_xor_sync(kFull, hmin, off));
        hmax = max(hmax, __shfl_xor_sync(kFull, hmax, off));
        vary |= __shfl_xor_sync(kFull, vary, off);
    }
    if (lane == 0) {
        s.hist[warp] = hmin;
        s.hist[kThreads / 32 + warp] = hmax;
        s.hist[2 * (kThreads / 32) + warp] = vary;
    }
    fbar();  // also: every entry of the buffer is in registers (s.packed overlays it)
    for (int w = 0; w < kThreads / 32; ++w) {
        hmin = min(hmin, s.hist[w]);
        hmax = max(hmax, s.hist[kThreads / 32 + w]);
        vary |= s.hist[2 * (kThreads / 32) + w];
    }
    fbar();
    // the digit: up to 11 bits below the common prefix, above the lowest bit that varies
    const uint32_t diff = hmin ^ hmax;
    const int shift = diff ? 32 - __clz(diff) : 0;
    const int low = vary ? __ffs(vary) - 1 : 0;
    const int w = min(11, max(shift - low, 0));
    const int sh = shift - w;
    const uint32_t dmask = w ? (1u << w) - 1u : 0u;
    auto digit = [&](uint64_t cc) { return ((uint32_t)(cc >> 32) >> sh) & dmask; };

    for (int b = tid; b < kBins; b += kThreads) s.hist[b] = 0u;
    fbar();
#pragma unroll
    for (int j = 0; j < kSortPer; ++j) hist_add(s.hist, digit(c[j]), j * kThreads + tid < n);
    fbar();

    // bucket starts from the top bin down, and the cost (sum of squared sizes)
    constexpr int per = kBins / kThreads;
    const int base = kBins - per * (tid + 1);  // this thread's bins, scanned from base + per - 1 down
    uint32_t h[per], local = 0u, sq = 0u;
#pragma unroll
    for (int i = 0; i < per; ++i) {
        h[i] = s.hist[base + per - 1 - i];
        local += h[i];
        sq += h[i] * h[i];
    }
    uint32_t incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += o;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(kFull, sq, off);
    if (lane == 31) s.warp_tot[warp] = incl;
    if (lane == 0) s.warp_base[warp] = (int)sq;
    fbar();
    uint32_t run = incl - local, cost = 0u;
    for (int v = 0; v < kThreads / 32; ++v) {
        if (v < warp) run += s.warp_tot[v];
        cost += (uint32_t)s.warp_base[v];
    }
    const bool ok = cost <= (uint32_t)kSortBudget * (uint32_t)n;
    if (ok) {
#pragma unroll
        for (int i = 0; i < per; ++i) {  // the bin's start, then the scatter's cursor
            s.hist[base + per - 1 - i] = run;
            run += h[i];
        }
    }
    fbar();
    if (!ok) return false;

    // scatter by bucket: each entry takes the next slot of its bucket (the order within a bucket is
    // free, since the ranking below compares the entries)
#pragma unroll
    for (int j = 0; j < kSortPer; ++j) {
        const bool valid = j * kThreads + tid < n;
        const uint32_t d = digit(c[j]);
        if (valid) s.packed[atomicAdd(&s.hist[d], 1u)] = c[j];
    }
    fbar();
    // hist[d] is now the end of bucket d, and hist[d + 1] its start (buckets run from the top bin down)
    for (int i = tid; i < n; i += kThreads) {
        const uint64_t cc = s.packed[i];
        const uint32_t d = digit(cc);
        const int st = d + 1 < (uint32_t)kBins ? (int)s.hist[d + 1] : 0;
        const int en = (int)s.hist[d];
        int rank = 0;
#pragma unroll 4
        for (int j = st; j < en; ++j) rank += s.packed[j] > cc ? 1 : 0;
        s.packed[n + st + rank] = cc;
    }
    fbar();
    return true;
}

// The score of an entry back from its key: -0 and NaN payloads were folded into the key, so those
// are read again from the row (x, n valid scores).
__device__ __forceinline__ float score_of(uint32_t key, uint32_t ix, const float *x, int n) {
    const uint32_t bits = (key & 0x80000000u) ? (key & 0x7fffffffu) : ~key;
    return ((bits == 0u || key == 0xffffffffu) && ix < (uint32_t)n) ? __ldg(x + ix) : __uint_as_float(bits);
}

// Output by score only: selects the kk best of the buffer's entries (all keyed) and writes them in
// output order to oi / ov (ov may be null), in one pass of buckets over the keys' leading varying
// bits: the histogram's scan gives every bucket's start, the buckets that start below kk are
// scattered, and each of their entries is ranked within its bucket as in bucket_sort; ranks below
// kk are written. Returns false with nothing written when the buckets are too uneven for the
// ranking to pay (the caller then selects and sorts separately). Block-wide; ends with a barrier.
__device__ bool select_sort_by_score(TopkSmem &s, int kk, int32_t *oi, float *ov, const float *x, int n) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cnt = s.count, keyed = s.keyed;
    if (kk == 0) return true;
    constexpr int kPerT = kCap / kThreads;
    // entries at or past `keyed` still hold raw score bits: keyed here, in registers
    auto key_at = [&](int i) {
        const uint32_t v = s.cb.key[i];
        return i < keyed ? v : order_key(__uint_as_float(v));
    };
    uint64_t c[kPerT];
    const uint32_t h0 = key_at(0);
    uint32_t hmin = 0xffffffffu, hmax = 0u, vary = 0u;
#pragma unroll
    for (int j = 0; j < kPerT; ++j) {
        c[j] = 0ull;
        if (j * kThreads < cnt) {  // the same for the whole block: slots past the count are skipped
            const int i = j * kThreads + tid;
            if (i < cnt) {
                c[j] = pack_out(key_at(i), s.cb.idx[i], true);
                const uint32_t h = (uint32_t)(c[j] >> 32);
                hmin = min(hmin, h);
                hmax = max(hmax, h);
                vary |= h ^ h0;
            }
        }
    }
    hmin = __reduce_min_sync(kFull, hmin);
    hmax = __reduce_max_sync(kFull, hmax);
    vary = __reduce_or_sync(kFull, vary);
    if (lane == 0) {
        s.hist[warp] = hmin;
        s.hist[kThreads / 32 + warp] = hmax;
        s.hist[2 * (kThreads / 32) + warp] = vary;
    }
    fbar();  // also: every entry of the buffer is in registers (s.packed overlays it)
    {
        const bool has = lane < kThreads / 32;
        hmin = __reduce_min_sync(kFull, has ? s.hist[lane] : 0xffffffffu);
        hmax = __reduce_max_sync(kFull, has ? s.hist[kThreads / 32 + lane] : 0u);
        vary = __reduce_or_sync(kFull, has ? s.hist[2 * (kThreads / 32) + lane] : 0u);
    }
    fbar();
    const uint32_t diff = hmin ^ hmax;
    const int shift = diff ? 32 - __clz(diff) : 0;
    const int low = vary ? __ffs(vary) - 1 : 0;
    const int w = min(11, max(shift - low, 0));
    const int sh = shift - w;
    const uint32_t dmask = w ? (1u << w) - 1u : 0u;
    // When the key bits take fewer than 11 bits of the digit and cover every bit in which the keys
    // differ, each key bucket holds a single key (low-precision scores tie often), and its entries
    // are ordered by position alone. The spare iw bits then split it further by position: the
    // entry at ix gets floor((n - 1 - ix) * (2^iw - 1) / n), which rises as ix falls, as the packed word
    // does. Float rounding keeps that map monotone, so every bucket is still a range of the order.
    // (The scale is (2^iw - 1) / n, so that the product stays below 2^iw without a clamp.)
    const int iw = (shift - low <= 11) ? 11 - w : 0;
    const float iscale = (float)((1u << iw) - 1u) / (float)max(n, 1);  // 0 when iw is 0
    auto digit = [&](uint64_t cc) {
        const uint32_t d = ((uint32_t)(cc >> 32) >> sh) & dmask;
        const int ix = (int)~(uint32_t)cc;
        return (d << iw) | (uint32_t)((float)max(n - 1 - ix, 0) * iscale);
    };

    for (int b = tid; b < kBins; b += kThreads) s.hist[b] = 0u;
    if (tid == 0) s.found_bin = -1;
    fbar();
#pragma unroll
    for (int j = 0; j < kPerT; ++j)
        if (j * kThreads < cnt && j * kThreads + tid < cnt) atomicAdd(&s.hist[digit(c[j])], 1u);
    fbar();

    // bucket starts from the top bin down, the cost (sum of squared sizes), and the bucket holding
    // the kk-th entry
    constexpr int per = kBins / kThreads;
    const int base = kBins - per * (tid + 1);
    uint32_t h[per], local = 0u, sq = 0u;
#pragma unroll
    for (int i = 0; i < per; ++i) {
        h[i] = s.hist[base + per - 1 - i];
        local += h[i];
        sq += h[i] * h[i];
    }
    uint32_t incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += o;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(kFull, sq, off);
    if (lane == 31) s.warp_tot[warp] = incl;
    if (lane == 0) s.warp_base[warp] = (int)sq;
    fbar();
    uint32_t run = incl - local;
    const bool has = lane < kThreads / 32;
    run += __reduce_add_sync(kFull, has && lane < warp ? s.warp_tot[lane] : 0u);
    const uint32_t cost = __reduce_add_sync(kFull, has ? (uint32_t)s.warp_base[lane] : 0u);
    const bool ok = cost <= (uint32_t)kSortBudget * (uint32_t)cnt;
    if (ok) {
#pragma unroll
        for (int i = 0; i < per; ++i) {
            const int b = base + per - 1 - i;
            if (run < (uint32_t)kk && run + h[i] >= (uint32_t)kk) s.found_bin = b;
            s.hist[b] = run;  // the bucket's start, then the scatter's cursor
            run += h[i];
        }
    }
    fbar();
    if (!ok) return false;
    const int cut = s.found_bin;
    if (cut < 0) {  // kk entries exist, so some bucket holds the kk-th (a broken invariant otherwise)
        if (tid == 0) s.broken = 1;
        fbar();
        return false;
    }

    // scatter the buckets at or above the cut
#pragma unroll
    for (int j = 0; j < kPerT; ++j) {
        if (j * kThreads < cnt) {
            const uint32_t d = digit(c[j]);
            const bool valid = j * kThreads + tid < cnt && d >= (uint32_t)cut;
            if (valid) s.packed[atomicAdd(&s.hist[d], 1u)] = c[j];  // the order within a bucket is free, as above
        }
    }
    fbar();
    // hist[d] is now the end of bucket d and hist[d + 1] its start; the cut bucket ends the scatter
    const int kept = (int)s.hist[cut];
    for (int i = tid; i < kept; i += kThreads) {
        const uint64_t cc = s.packed[i];
        const uint32_t d = digit(cc);
        const int st = d + 1 < (uint32_t)kBins ? (int)s.hist[d + 1] : 0;
        const int en = (int)s.hist[d];
        int rank = 0;
#pragma unroll 4
        for (int j = st; j < en; ++j) rank += s.packed[j] > cc ? 1 : 0;
        const int pos = st + rank;
        if (pos < kk) {
            uint32_t key, ix;
            unpack_out(cc, true, key, ix);
            oi[pos] = (int32_t)ix;
            if (ov) ov[pos] = score_of(key, ix, x, n);
        }
    }
    fbar();
    return true;
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

// A position in this CTA's sequence of tiles: tile `tile` of row `row`, a row of n valid scores.
struct TileCursor {
    int row, tile, n;
};

// Moves the cursor past finished rows; false once this CTA has no tile left.
__device__ __forceinline__ bool cursor_settle(const TopkParams &p, TileCursor &c) {
    while (c.row < p.rows && c.tile * kTile >= c.n) {
        c.row += gridDim.x;
        c.tile = 0;
        c.n = c.row < p.rows ? row_length(p, c.row) : 0;
    }
    return c.row < p.rows;
}

// The tile's first score and its length in bytes, rounded up to whole 16-byte groups (ld % 4 == 0
// keeps them inside the row).
__device__ __forceinline__ const float *cursor_src(const TopkParams &p, const TileCursor &c, uint32_t &bytes) {
    const int cnt = min(kTile, c.n - c.tile * kTile);
    bytes = (uint32_t)((cnt + 3) & ~3) * 4u;
    return p.scores + (size_t)c.row * (size_t)p.ld + (size_t)c.tile * kTile;
}

// First score of sample run j of a row of n scores (n >= kSampleMinLen): runs spread evenly,
// starting on a multiple of 4, inside the row and not overlapping.
__device__ __forceinline__ int sample_run_start(int j, int n) {
    return (int)(((long long)j * (n - kSampleRun) / (kSampleRuns - 1)) & ~3ll);
}

// Element of the row held by value q of this thread in tile t (two float4 per thread, 512 floats apart).
__device__ __forceinline__ int tile_elem(int t, int q) {
    return t * kTile + 4 * ((q >> 2) * kThreads + (int)threadIdx.x) + (q & 3);
}

// Appends this thread's scores of tile t whose key reaches the bound (the test on the score itself,
// see set_threshold) to the buffer, one shared atomic per warp; with slice >= 0, only the scores at
// the tile's positions [512 slice, 512 slice + 512). Entries that would land at kCap or beyond are
// not written. Records where the warp's append started in warp_base and returns the buffer count
// right after it (0 when the warp appends nothing).
// Bit q set: value q of this thread's part of tile t is kept (inside the row, key at or above the bound).
__device__ __forceinline__ uint32_t keep_mask(const float (&vals)[kPer], int t, int n, float thr, int mode) {
    uint32_t keepm = 0u;
    if (mode == 0 && (t + 1) * kTile <= n) {  // a full tile and a plain threshold: one compare per score
#pragma unroll
        for (int q = 0; q < kPer; ++q) keepm |= (uint32_t)!(vals[q] < thr) << q;
    } else {
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const bool keep = tile_elem(t, q) < n && (mode == 0 ? !(vals[q] < thr) : (mode == 1 && isnan(vals[q])));
            keepm |= (uint32_t)keep << q;
        }
    }
    return keepm;
}

__device__ __forceinline__ int filter_append(TopkSmem &s, const float (&vals)[kPer], int t, int n, float thr,
                                             int mode, int slice, int stage = -1) {
    const int lane = threadIdx.x & 31;
    uint32_t keepm = keep_mask(vals, t, n, thr, mode);
    if (slice >= 0)  // slice j: threads [128 (j % 4), +128), first (j < 4) or second float4
        keepm &= ((int)threadIdx.x >> 7) == (slice & 3) ? (0x0fu << (4 * (slice >> 2))) : 0u;
    const unsigned m = __ballot_sync(kFull, keepm != 0u);  // the lanes that keep something
    if (m == 0u) {
        if (lane == 0) s.warp_base[threadIdx.x >> 5] = INT_MAX;
        return 0;
    }
    const int c = __popc(keepm);
    if (!__any_sync(kFull, c > 1)) {
        // the common case: every lane keeps at most one score, so the ballot gives the positions
        const int total = __popc(m);
        int base = 0;
        if (lane == 0) base = atomicAdd(&s.count, total);
        base = __shfl_sync(kFull, base, 0);
        if (lane == 0) s.warp_base[threadIdx.x >> 5] = base;
        const int pos = base + __popc(m & ((1u << lane) - 1u));
        if (c != 0 && pos < kCap) {
            const int q = __ffs(keepm) - 1;
            const int o = 4 * (int)threadIdx.x + 4 * kThreads * (q >> 2) + (q & 3);  // offset within the tile
            float v;
            if (stage >= 0) {  // the tile is in the ring: read the one score back
                v = s.ring[stage][o];
            } else {
                v = vals[0];
#pragma unroll
                for (int qq = 1; qq < kPer; ++qq) v = q == qq ? vals[qq] : v;
            }
            s.cb.key[pos] = __float_as_uint(v);  // raw bits; the next compaction makes the key
            s.cb.idx[pos] = (uint32_t)(tile_elem(t, 0) + 4 * kThreads * (q >> 2) + (q & 3));
        }
        return base + total;
    }
    // an exclusive scan of the lanes' counts
    int incl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += o;
    }
    const int total = __shfl_sync(kFull, incl, 31);
    int base = 0;
    if (lane == 31) base = atomicAdd(&s.count, total);
    base = __shfl_sync(kFull, base, 31);
    if (lane == 0) s.warp_base[threadIdx.x >> 5] = base;
    int pos = base + incl - c;
    const uint32_t e0 = (uint32_t)tile_elem(t, 0);  // value q sits at e0 + 2048 (q / 4) + q % 4
    // raw score bits; the next compaction turns them into keys
    if (base + total <= kCap) {  // the whole warp's append fits
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            if ((keepm >> q) & 1u) {
                s.cb.key[pos] = __float_as_uint(vals[q]);
                s.cb.idx[pos] = e0 + (uint32_t)(4 * kThreads * (q >> 2) + (q & 3));
                ++pos;
            }
        }
    } else {
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            if (((keepm >> q) & 1u) && pos < kCap) {
                s.cb.key[pos] = __float_as_uint(vals[q]);
                s.cb.idx[pos] = e0 + (uint32_t)(4 * kThreads * (q >> 2) + (q & 3));
                ++pos;
            }
        }
    }
    return base + total;
}

// Warp-private appends for rows that start from the sampled bound: warp w owns entries
// [w kRegion, (w + 1) kRegion) of the buffer and keeps its fill in a register, so an append needs
// no shared atomic and no broadcast. The fills stay near 3.5K / 16 = 220 on low-precision indexer
// scores. A check that finds a fill above kRegionSoft gathers the regions and continues with the
// shared count; entries past a region's end are counted but not written (the row is then scanned
// again, as for a buffer overflow).
constexpr int kRegion = kCap / (kThreads / 32);  // 320
constexpr int kRegionSoft = kRegion - 4 * kCheck;  // 288
static_assert(kRegion * (kThreads / 32) == kCap, "the regions tile the buffer");

// Appends this thread's kept scores of tile t (held in ring stage `stage`) to its warp's region
// after `fill` entries; returns the warp's new fill (the same in every lane).
__device__ __forceinline__ int region_append(TopkSmem &s, const float (&vals)[kPer], int t, int n, float thr,
                                             int mode, int stage, int fill) {
    const int lane = threadIdx.x & 31;
    uint32_t keepm = keep_mask(vals, t, n, thr, mode);
    const unsigned m = __ballot_sync(kFull, keepm != 0u);
    if (m == 0u) return fill;
    uint32_t *rk = s.cb.key + (threadIdx.x >> 5) * kRegion;
    uint32_t *ri = s.cb.idx + (threadIdx.x >> 5) * kRegion;
    const int base = t * kTile + 4 * (int)threadIdx.x;  // the row position of value 0; value q adds off(q)
    auto put = [&](int pos, uint32_t bits) {
        const int q = __ffs(bits) - 1;
        const int off = 4 * kThreads * (q >> 2) + (q & 3);
        if (pos < kRegion) {
            rk[pos] = __float_as_uint(s.ring[stage][4 * (int)threadIdx.x + off]);  // raw bits, keyed later
            ri[pos] = (uint32_t)(base + off);
        }
    };
    {
        // every keeping lane's first score: its place among the keeping lanes. Straight-line code
        // for the whole warp (the read-back address is valid for any q) and predicated stores.
        const int q = __ffs(keepm) - 1;
        const int off = 4 * kThreads * ((q >> 2) & 1) + (q & 3);
        const int pos = fill + __popc(m & ((1u << lane) - 1u));
        const uint32_t bits = __float_as_uint(s.ring[stage][4 * (int)threadIdx.x + off]);
        if (keepm != 0u && pos < kRegion) {
            rk[pos] = bits;  // raw bits, keyed later
            ri[pos] = (uint32_t)(base + off);
        }
    }
    int next = fill + __popc(m);
    keepm &= keepm - 1u;
    if (__any_sync(kFull, keepm != 0u)) {
        const uint32_t more = keepm & (keepm - 1u);
        if (!__any_sync(kFull, more != 0u)) {
            // no lane keeps more than two: each second score after every first, in lane order
            const unsigned b = __ballot_sync(kFull, keepm != 0u);
            const int q = __ffs(keepm) - 1;
            const int off = 4 * kThreads * ((q >> 2) & 1) + (q & 3);
            const int pos = next + __popc(b & ((1u << lane) - 1u));
            const uint32_t bits = __float_as_uint(s.ring[stage][4 * (int)threadIdx.x + off]);
            if (keepm != 0u && pos < kRegion) {
                rk[pos] = bits;
                ri[pos] = (uint32_t)(base + off);
            }
            return next + __popc(b);
        }
        // lanes that keep several scores of the tile: the rest after every first, in lane order
        const int c = __popc(keepm);
        int incl = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(kFull, incl, off);
            if (lane >= off) incl += o;
        }
        int pos = next + incl - c;
        next += __shfl_sync(kFull, incl, 31);
        while (keepm) {
            put(pos++, keepm);
            keepm &= keepm - 1u;
        }
    }
    return next;
}

// Moves the regions' entries (fill = the calling warp's fill, at most kRegion) to the front of the
// buffer in warp order and sets the count to their total. Every append must be done. Block-wide;
// ends with a barrier.
__device__ void gather_regions(TopkSmem &s, int fill) {
    constexpr int kPerT = kCap / kThreads;
    const int tid = threadIdx.x, lane = tid & 31;
    if (lane == 0) s.warp_tot[tid >> 5] = (uint32_t)min(fill, kRegion);
    fbar();
    // lane v: warp v's fill and where its entries go
    const int f = lane < kThreads / 32 ? (int)s.warp_tot[lane] : 0;
    int incl = f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += o;
    }
    const int start = incl - f;
    const int total = __shfl_sync(kFull, incl, 31);
    uint32_t key[kPerT], idx[kPerT];
    int dst[kPerT];
#pragma unroll
    for (int j = 0; j < kPerT; ++j) {
        const int i = j * kThreads + tid;
        const int w = i / kRegion, r = i - w * kRegion;
        const int fw = __shfl_sync(kFull, f, w), sw = __shfl_sync(kFull, start, w);
        dst[j] = r < fw ? sw + r : -1;
        key[j] = s.cb.key[i];
        idx[j] = s.cb.idx[i];
    }
    fbar();
#pragma unroll
    for (int j = 0; j < kPerT; ++j) {
        if (dst[j] >= 0) {
            s.cb.key[dst[j]] = key[j];
            s.cb.idx[dst[j]] = idx[j];
        }
    }
    if (tid == 0) {
        s.count = total;
        s.keyed = 0;
    }
    fbar();
}

// This thread's kPer scores of tile t, read from `tile` (the tile's first score, in the ring or in
// global memory); float4 groups that start at or beyond n are not read.
__device__ __forceinline__ void load_tile_vals(const float *tile, int t, int n, float (&vals)[kPer]) {
    const float4 *t4 = reinterpret_cast<const float4 *>(tile);
#pragma unroll
    for (int j = 0; j < kPer / 4; ++j) {
        // a float4 that starts inside the row ends inside it too (ld is a multiple of 4)
        const float4 v = tile_elem(t, 4 * j) < n ? t4[j * kThreads + threadIdx.x] : make_float4(0.f, 0.f, 0.f, 0.f);
        vals[4 * j] = v.x, vals[4 * j + 1] = v.y, vals[4 * j + 2] = v.z, vals[4 * j + 3] = v.w;
    }
}

// The rare path of a tile whose appends took the buffer past kSoft (block-wide, right after the
// barrier that ends the tile's appends). If nothing was lost, the buffer is compacted. If some
// entries did not fit (count beyond kCap), the tile's appends are undone (they start at the lowest
// warp base) and the tile, read again from `tile`, is appended one slice of 512 positions at a time
// in position order, with a compaction before any slice that might not fit. Every entry then
// enters after all entries of lower position, as the compaction's tie rule assumes.
__device__ void settle_tile(TopkSmem &s, const float *tile, int t, int n, int k, int idx_bits, bool overflow,
                            float &thr, int &mode) {
    const int limit = k + (kSoft - k) / 2;  // compact well below kSoft, so that many tiles fit after it
    if (!overflow) {
        set_threshold(compact(s, k, limit, false, idx_bits), thr, mode);
        return;
    }
    int start = INT_MAX;
    for (int w = 0; w < kThreads / 32; ++w) start = min(start, s.warp_base[w]);
    fbar();  // every thread has read warp_base
    if (threadIdx.x == 0) s.count = start;
    fbar();
    int cnt = start;
    float vals[kPer];
    load_tile_vals(tile, t, n, vals);
    for (int j = 0; j < kTile / kSlice; ++j) {
        if (cnt > kCap - kSlice) {
            set_threshold(compact(s, k, limit, false, idx_bits), thr, mode);
        }
        filter_append(s, vals, t, n, thr, mode, j);
        fbar();
        cnt = s.count;
        fbar();  // every thread has read the count before it changes again
    }
}

// The sample rank r of the starting bound: with r0 = kk m / n the sample rank expected for the
// row's kk-th best score (m = sample size), r solves r - 5 sqrt(r) = r0, so a row whose scores
// are exchangeable holds fewer than kk keys at or above the bound only about 5 standard
// deviations below the mean. Any outcome is correct (a row that falls short is scanned again);
// r only trades that rescan against the number of compactions.
__device__ __forceinline__ int sample_rank(int kk, int n) {
    const float r0 = (float)kk * (float)kSample / (float)n;
    const float sq = 0.5f * (5.0f + sqrtf(25.0f + 4.0f * r0));
    return (int)ceilf(sq * sq);
}

// A starting lower bound for row x of n scores (n >= kSampleMinLen): a key with at least r of the
// sampled keys at or above it. The sample is 16 runs of 512 consecutive scores, run j starting at
// floor(j (n - 512) / 15) rounded down to a multiple of 4, so every run lies inside the row and
// the runs do not overlap. The bound is read off one histogram of the sampled keys in the window
// of 2^24 keys below the largest (two binades of positive scores, in 2048 bins of 2^13 keys): the
// lower edge of the bin holding the r-th largest. If fewer than r keys fall in the window, a radix
// descent over the whole sample finds it instead. Uses the buffer's storage and the histogram
// (the buffer must be empty).
__device__ uint64_t sampled_bound(TopkSmem &s, const float *x, int n, int r) {
    constexpr int kRunVec = kSampleRun / 4;
    constexpr int kWinBits = 24, kBinBits = kWinBits - 11;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int b = tid; b < kBins; b += kThreads) s.hist[b] = 0u;
    const float4 *x4 = reinterpret_cast<const float4 *>(x);
    float4 v[kSample / 4 / kThreads];
#pragma unroll
    for (int j = 0; j < kSample / 4 / kThreads; ++j) {
        const int w = j * kThreads + tid;  // float4 of the sample
        v[j] = __ldg(x4 + sample_run_start(w / kRunVec, n) / 4 + (w % kRunVec));
    }
    uint32_t kmax = 0u;
#pragma unroll
    for (int j = 0; j < kSample / 4 / kThreads; ++j) {
        const int w = j * kThreads + tid;
        const uint32_t a = order_key(v[j].x), b = order_key(v[j].y), c = order_key(v[j].z), d = order_key(v[j].w);
        s.sample[4 * w] = a;
        s.sample[4 * w + 1] = b;
        s.sample[4 * w + 2] = c;
        s.sample[4 * w + 3] = d;
        kmax = max(kmax, max(max(a, b), max(c, d)));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) kmax = max(kmax, __shfl_xor_sync(kFull, kmax, off));
    if (lane == 0) s.warp_tot[warp] = kmax;
    fbar();
    for (int w = 0; w < kThreads / 32; ++w) kmax = max(kmax, s.warp_tot[w]);
    const uint32_t wlo = kmax >= (1u << kWinBits) ? kmax - ((1u << kWinBits) - 1u) : 0u;
    for (int i0 = tid & ~31; i0 < kSample; i0 += kThreads) {
        const uint32_t key = s.sample[i0 + lane];
        hist_add(s.hist, (key - wlo) >> kBinBits, key >= wlo);
    }
    fbar();  // also: every thread has read warp_tot (find_bin rewrites it)
    find_bin(s, (uint32_t)r, true);
    if (s.found_bin >= 0) return (uint64_t)wlo + ((uint64_t)s.found_bin << kBinBits);
    const Descent d = radix_descent(s, s.sample, kSample, r, r + r / 4, false);
    return (uint64_t)d.prefix << d.shift;
}

// Persistent CTAs, each taking rows blockIdx.x, blockIdx.x + gridDim.x, ... A producer warp keeps
// kStages tiles of 4096 scores in flight (bulk copies into a shared-memory ring, one "full"
// mbarrier per stage), running ahead across row boundaries, and refills a stage as soon as every
// filter thread has released it (one "empty" mbarrier per stage, one arrival per thread, so no
// warp has to reconverge for one lane to arrive). The 16 filter warps wait for each tile
// themselves (every lane tests the mbarrier; one lane polls, bounded, when they do not all see it
// complete) and filter it into the candidate buffer; their own barriers only decide whether the
// buffer needs attention.
__global__ void __launch_bounds__(kBlock, 2) topk_kernel(TopkParams p) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    TopkSmem &s = *reinterpret_cast<TopkSmem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31;
    const int k = p.k;
    const int idx_bits = p.ld <= (1 << 22) ? 22 : 32;
    volatile int *failed = &s.failed;
    if (tid == 0) {
        for (int st = 0; st < kStages; ++st) {
            ptx::mbar_init(ptx::smem_u32(&s.full[st]), 1);
            ptx::mbar_init(ptx::smem_u32(&s.empty[st]), kThreads);
        }
        ptx::fence_mbar_init();
        s.failed = 0;
        s.broken = 0;
        s.issued = 0u;
    }
    __syncthreads();

    if (tid >= kThreads) {
        // ---------------------------------------------------------------- producer warp
        if (tid == kThreads) {
            TileCursor cur{(int)blockIdx.x, 0, blockIdx.x < p.rows ? row_length(p, blockIdx.x) : 0};
            uint32_t it = 0u;
            while (cursor_settle(p, cur)) {
                const uint32_t st = it % kStages;
                // the stage's previous tile has been released by every filter thread
                if (it >= kStages && !ptx::mbar_wait(ptx::smem_u32(&s.empty[st]), ((it / kStages) & 1u) ^ 1u)) {
                    *failed = 1;
                    if (p.status) raise_status(p.status, RL_ERR_TIMEOUT);
                    break;
                }
                if (*failed) break;
                uint32_t bytes;
                const float *src = cursor_src(p, cur, bytes);
                const uint32_t bar = ptx::smem_u32(&s.full[st]);
                ptx::mbar_arrive_expect_tx(bar, bytes);
                ptx::bulk_g2s(ptx::smem_u32(s.ring[st]), src, bytes, bar);  // default L2 policy: 1% faster than evict-first
                ++cur.tile;
                ++it;
                *reinterpret_cast<volatile uint32_t *>(&s.issued) = it;
            }
        }
        return;
    }

    // ---------------------------------------------------------------- filter warps
    // Waits for tile gi to land: every lane tests the stage's mbarrier once, and if they do not all
    // see it complete, one lane polls (bounded); after a timeout the tiles are no longer waited for
    // and the results are not valid (flagged).
    auto wait_tile = [&](uint32_t gi) {
        const uint32_t bar = ptx::smem_u32(&s.full[gi % kStages]), parity = (gi / kStages) & 1u;
        if (__all_sync(kFull, ptx::mbar_try_wait(bar, parity))) return;  // the common case: every lane sees it
        if (lane == 0 && !*failed && !ptx::mbar_wait(bar, parity)) {
            *failed = 1;
            if (p.status) raise_status(p.status, RL_ERR_TIMEOUT);
        }
        __syncwarp();
    };

    uint32_t g = 0;  // tiles consumed by this CTA
    for (int row = blockIdx.x; row < p.rows; row += gridDim.x) {
        const int nraw = p.lengths ? __ldg(p.lengths + row) : (int)p.ld;
        if (tid == 0 && p.status && (nraw < 0 || nraw > p.ld)) raise_status(p.status, RL_ERR_SEQLENS);
        const int n = row_length(p, row);
        const int kk = min(k, n);
        if (tid == 0) {
            s.count = 0;
            s.keyed = 0;
        }
        fbar();
        // incoming scores are kept when their key reaches a lower bound, tested on the score itself
        float thr = -INFINITY;
        int mode = 0;
        // Long rows start from a bound taken from a sample of the row instead of -inf. Whatever
        // the sample holds, the scores kept are all those whose key reaches the bound (compactions
        // drop only what the rows' kk best cannot contain), so if at least kk reach it they
        // contain the kk best; if fewer reach it, the row is scanned again from -inf below.
        const int r = n >= kSampleMinLen ? sample_rank(kk, n) : kSample;
        const bool sampled = r <= kSample / 4;
        if (sampled) {
            set_threshold(sampled_bound(s, p.scores + (size_t)row * (size_t)p.ld, n, r), thr, mode);
        }
        const int ntiles = (n + kTile - 1) / kTile;
        auto ring_vals = [&](int st, float (&vals)[kPer]) {
            const float4 *tile4 = reinterpret_cast<const float4 *>(s.ring[st]);
#pragma unroll
            for (int j = 0; j < kPer / 4; ++j) {
                const float4 v = tile4[j * kThreads + tid];
                vals[4 * j] = v.x, vals[4 * j + 1] = v.y, vals[4 * j + 2] = v.z, vals[4 * j + 3] = v.w;
            }
        };
        if (sampled) {
            // The sampled bound keeps about 3.5K scores of a 200K-score row, inside the buffer: the
            // warps stream the row with a block barrier only every kCheck tiles, each releasing a
            // stage as soon as it is done with it. At a barrier, a count past kSoftSampled compacts
            // the buffer (raising the bound); an append past the buffer is counted but not written,
            // and the row is then scanned again below.
            // The warps start in their own regions of the buffer (region_append). A check that finds
            // a region nearly full, with nothing dropped yet, gathers the regions and continues with
            // the shared count, compacting as above.
            int grp = 0;   // shared count: this warp's count after its last append since the last barrier
            int fill = 0;  // regions: this warp's fill
            bool regions = true;
            for (int t = 0; t < ntiles; ++t, ++g) {
                const int st = (int)(g % kStages);
                wait_tile(g);
                {
                    float vals[kPer];
                    ring_vals(st, vals);
                    if (regions)
                        fill = region_append(s, vals, t, n, thr, mode, st, fill);
                    else
                        grp = max(grp, filter_append(s, vals, t, n, thr, mode, -1, st));
                }
                ptx::mbar_arrive(ptx::smem_u32(&s.empty[st]));  // this thread is done with the stage
                if ((t % kCheck) == kCheck - 1 && t + 1 < ntiles) {
                    if (regions) {
                        if (fbar_or(fill > kRegionSoft) && !fbar_or(fill > kRegion)) {
                            gather_regions(s, fill);
                            regions = false;
                            if (s.count > kSoftSampled)
                                set_threshold(compact(s, k, k + (kSoft - k) / 2, false, idx_bits), thr, mode);
                        }
                    } else if (fbar_or(grp > kSoftSampled) && !fbar_or(grp > kCap)) {
                        set_threshold(compact(s, k, k + (kSoft - k) / 2, false, idx_bits), thr, mode);
                    }
                    grp = 0;
                }
            }
            if (regions) {
                if (fbar_or(fill > kRegion)) {
                    // a region dropped entries: scan the row again below, from -inf if fewer than kk
                    // scores reached the bound, else from the same bound
                    if (lane == 0) s.warp_tot[tid >> 5] = (uint32_t)fill;
                    fbar();
                    int total = 0;
                    for (int w = 0; w < kThreads / 32; ++w) total += (int)s.warp_tot[w];
                    if (tid == 0) s.count = total < kk ? total : kCap + 1;
                } else {
                    gather_regions(s, fill);
                }
            }
        } else {
            for (int t = 0; t < ntiles; ++t, ++g) {
                const int st = (int)(g % kStages);
                wait_tile(g);
                int after_add;
                {
                    float vals[kPer];
                    ring_vals(st, vals);
                    after_add = filter_append(s, vals, t, n, thr, mode, -1, st);
                }
                // Whether the buffer needs attention is decided by the barrier itself (the count
                // passed kSoft iff some warp's append took it past): a thread must not read s.count
                // here, because a faster warp may already be appending the next tile.
                if (fbar_or(after_add > kSoft)) {
                    const bool overflow = fbar_or(after_add > kCap) != 0;
                    settle_tile(s, s.ring[st], t, n, k, idx_bits, overflow, thr, mode);
                }
                ptx::mbar_arrive(ptx::smem_u32(&s.empty[st]));  // this thread is done with the stage
            }
        }
        fbar();  // every append of the row is done
        const int cnt = s.count;
        // A sampled row is scanned again with plain loads (the tile ring has moved on to the next
        // row), with a block barrier per tile and the compactions: from -inf if its bound was above
        // the row's kk-th best score (fewer than kk reached it), from the same bound if the scores
        // at or above it overflowed the buffer (ties at the bound) or a warp's region.
        const bool from_inf = sampled && cnt < kk, again = from_inf || (sampled && cnt > kCap);
        if (again) {
            fbar();  // every thread has read the count
            if (tid == 0) {
                s.count = 0;
                s.keyed = 0;
            }
            fbar();
            if (from_inf) {
                thr = -INFINITY;
                mode = 0;
            }
            for (int t = 0; t < ntiles; ++t) {
                const float *tile = p.scores + (size_t)row * (size_t)p.ld + (size_t)t * kTile;
                int after_add;
                {
                    float vals[kPer];
                    load_tile_vals(tile, t, n, vals);
                    after_add = filter_append(s, vals, t, n, thr, mode, -1);
                }
                if (fbar_or(after_add > kSoft)) {
                    const bool overflow = fbar_or(after_add > kCap) != 0;
                    settle_tile(s, tile, t, n, k, idx_bits, overflow, thr, mode);
                }
            }
        }
        const bool by_score = p.order_by_score != 0;
        const float *x = p.scores + (size_t)row * (size_t)p.ld;
        int32_t *oi = p.out_idx + (size_t)row * (size_t)p.ldo;
        float *ov = p.out_val ? p.out_val + (size_t)row * (size_t)p.ldo : nullptr;
        // by score: select the best min(k, n) and order them in one pass of buckets when the
        // buckets are even enough (keying the entries that still hold raw bits in registers)
        const bool direct = by_score && select_sort_by_score(s, kk, oi, ov, x, n);
        bool bucketed = false;
        if (!direct) {
            make_keys(s);
            // exactly the best min(k, n)
            if (s.count > kk) compact(s, kk, kk, true, idx_bits);
            // order them: by buckets of the key (or position) when they are even enough, else with
            // the bitonic network over the selection padded to a power of two with entries that sort last
            bucketed = kk <= kSortMax && bucket_sort(s, kk, by_score);
            if (!bucketed) {
                int n2 = 1;
                while (n2 < kk) n2 <<= 1;
                for (int i = kk + tid; i < n2; i += kThreads) {
                    s.cb.key[i] = 0u;
                    s.cb.idx[i] = 0xffffffffu;
                }
                fbar();
                if (n2 == 2 * kThreads)
                    bitonic_regs<2>(s, by_score);
                else if (n2 == 4 * kThreads)
                    bitonic_regs<4>(s, by_score);
                else if (kk > 1)
                    bitonic(s, n2, by_score);
            }
        }
        if (tid == 0 && (s.broken || s.count > kCap)) {
            if (p.status) raise_status(p.status, RL_ERR_INTERNAL);
            s.broken = 0;
        }
        for (int i = tid; i < k; i += kThreads) {
            if (i < kk) {
                if (direct) continue;  // written by the bucket pass
                uint32_t key, ix;
                if (bucketed) {
                    unpack_out(s.packed[kk + i], by_score, key, ix);
                } else {
                    key = s.cb.key[i];
                    ix = s.cb.idx[i];
                }
                oi[i] = (int32_t)ix;
                if (ov) ov[i] = score_of(key, ix, x, n);
            } else {
                oi[i] = -1;
                if (ov) ov[i] = -INFINITY;
            }
        }
        fbar();  // the buffer is reused by the next row
    }
    // after a timeout: let the copies that may still be in flight land before the CTA leaves (bounded)
    if (tid == 0 && *failed) {
        const uint32_t issued = *reinterpret_cast<volatile uint32_t *>(&s.issued);
        for (uint32_t gi = issued > (uint32_t)kStages ? issued - kStages : 0u; gi < issued; ++gi)  // the last ones
            ptx::mbar_wait(ptx::smem_u32(&s.full[gi % kStages]), (gi / kStages) & 1u, 100000000ull);
    }
}

}  // namespace

int topk_max_k() { return 4096; }  // the final sort pads to a power of two <= kCap
static_assert(4096 <= kSoft && 4096 <= kCap, "k up to 4096: compaction targets and the final sort fit");

cudaError_t launch_topk(const TopkParams &p, cudaStream_t stream) {
    if (p.rows <= 0) return cudaSuccess;
    // per device, once: the shared-memory opt-in and the SM count (host threads may launch on
    // different devices at the same time)
    static std::mutex mu;
    static int sms_of[64] = {};  // 0: this device is not configured yet
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int sms = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= 64 || sms_of[dev] == 0) {
            e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(TopkSmem));
            if (e != cudaSuccess) return e;
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return e;
            if (dev < 64) sms_of[dev] = sms;
        } else {
            sms = sms_of[dev];
        }
    }
    const int grid = std::min(p.rows, 2 * sms);  // persistent: two CTAs per SM
    topk_kernel<<<grid, kBlock, sizeof(TopkSmem), stream>>>(p);
    return cudaGetLastError();
}

}  // namespace rlk
