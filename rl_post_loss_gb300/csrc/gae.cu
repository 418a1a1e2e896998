// Generalized advantage estimation with skipped observation tokens and the
// cross-trajectory discount ("Zhipu AI / GLM: From Blank Infilling to
// Compaction-Aware Agentic Reinforcement Learning", section 11: skip-
// observation GAE of the single-rollout critic, and CompactionRL's
// "cross-trajectory GAE" over the segments of one rollout), as one pass over
// the token arrays.
//
// Per response, walking backwards over its action (mask=1) tokens t with next
// action token t':  A_t = r_t + gamma V_{t'} - V_t + gamma lambda A_{t'}
// (V_{t'} = A_{t'} = 0 after the last one); observation tokens get A = 0.
// With the cross-trajectory discount every advantage of segment s is further
// multiplied by (gamma lambda)^{N_{>s}}, N_{>s} the mask=1 tokens of the later
// segments of the same rollout.
//
// Design. The token range is cut into fixed chunks of 8192 tokens; one block
// per chunk, chunks handed out right to left by an atomic ticket. What a run
// of tokens does to the state (A, V) arriving from its right is affine,
//   A <- p A + q V + c,   V <- V (no action token, no response end) or vf,
// and a response end resets the state to zero; with the cross-trajectory
// discount two integer counts ride along (mask=1 tokens to the right within
// the response and within the rollout), whose difference is N_{>s}. Such maps
// compose associatively. A block stages its chunk in shared memory (two
// tensor copies of the rewards and values as [256 x 32] tiles with the
// 128-byte swizzle and one bulk copy of the mask bytes, issued by one thread;
// coalesced 16-byte asynchronous copies for a partial chunk or unaligned
// arrays), folds 32 tokens per thread into a map (fp32), scans the 256 maps
// with a fixed tree and publishes the chunk's map.
// Warp 0 then looks back: it composes the published maps of the chunks to its
// right, in a fixed order and tree, up to and including the first one that
// holds a response end (the state further right cannot reach it); the rollout
// count (an integer, so any order gives the same sum) uses the classic
// decoupled look-back with inclusive values. It waits only for the chunks up
// to those stopping points. Every floating-point result depends only on the
// inputs, never on timing: bit-identical from run to run. Waits are bounded
// (1 s of %globaltimer by default); one that runs out raises RL_ERR_TIMEOUT
// and treats the chunk as a response end. A map is published as 64-bit words
// that each pair a value with the launch's tag, so the look-back reads one in
// a single round trip. The advantages are written in place of the staged
// rewards and each warp's rows leave by a tensor store as soon as the warp is
// done, when the whole chunk lies inside the covered range. The last block
// past its look-back resets the ticket and the block count and advances the
// launch epoch (a record counts only under this launch's tag), so the
// workspace is ready for the next launch with nothing else to clear.
#include <cuda.h>

#include <atomic>

#include "common.cuh"
#include "ptx.cuh"
#include "scan_select.cuh"
#include "tmap.cuh"

namespace rlk {

namespace {

constexpr int kThreads = 256;
constexpr int kTok = 32;                 // consecutive tokens per thread
constexpr int kChunk = kThreads * kTok;  // tokens per chunk
constexpr int kVec = kTok / 4;           // float4 groups per thread
constexpr unsigned kFull = 0xffffffffu;
// Dynamic shared memory: rewards and values (one 128-byte row per thread,
// its eight 16-byte groups XOR-swizzled by the row index so that the 16-byte
// reads of a quarter warp hit distinct banks), then the mask bytes.
constexpr int kSmemR = 0;
constexpr int kSmemV = kChunk * 4;
constexpr int kSmemM = 2 * kChunk * 4;
constexpr int kSmemBytes = 2 * kChunk * 4 + kChunk;

// GaeMap::bits
constexpr uint32_t kPassV = 1;     // no action token and no response end: V passes
constexpr uint32_t kClosed = 2;    // holds a response end: ignores everything to its right
constexpr uint32_t kPassRoll = 4;  // no rollout end: the rollout count passes

// A <- p A + q V + c; V <- (bits & kPassV) ? V : vf; the response count
// n <- n_resp + (closed ? 0 : n), the rollout count m <- n_roll + (passroll ? m : 0).
struct GaeMap {
    float p, q, c, vf;
    uint32_t bits;
    int32_t n_resp, n_roll;
};

// One slot per chunk in the workspace, at an offset that depends only on the
// chunk index (so a later call with more chunks never reads an earlier call's
// records as its own). Every published 32-bit value travels in a 64-bit word
// together with the launch's tag (single-copy atomic), so a reader takes a map
// in one round trip, all its words at once, and accepts it when every tag is
// this launch's: no flag, no ordering between the words, and nothing to clear
// afterwards. Words 0-6: p, q, c, vf, bits, n_resp, n_roll (the map); word 7:
// the inclusive rollout count, published after the look-back.
struct ChunkRecord {
    uint64_t w[8];
};
static_assert(sizeof(ChunkRecord) == 64, "record size");
constexpr int kWsHeader = 256;
// Start offset between the first wave's blocks on an SM (measured on the 16.8M-token workload:
// 2.5-3.5 us gave 62.1-62.7 us per launch against 65.6 unstaggered; 1.5 us 63.8-64.2; 5 us 65.5).
constexpr uint32_t kStaggerNs = 3000;

// Tensor maps of the token arrays viewed as [T / 32 rows x 32 floats] (one 128-byte row per
// thread's 32 tokens), boxes of 256 rows (a chunk) with the 128-byte swizzle: the same XOR layout
// as tile_off, so the fold and the re-walk read the staged rows unchanged.
struct GaeMaps {
    CUtensorMap r, v, adv, ret;
    int32_t ok;  // 1: the maps are valid (every array 16-byte aligned, T >= one chunk)
};

struct GaeSmall {
    uint64_t bar;
    uint32_t last[kThreads];  // bit i of word w: token 32 w + i is the last of its response
    uint32_t cont[kThreads];  // ... and its rollout continues into the next response
    GaeMap wtot[kThreads / 32];
    GaeMap after[kThreads / 32];
    int k, sa, sb, lo, hi;
    float EA, EV;
    int EP, ER;
    uint32_t epoch;
    float pw[kTok + 1], qpw[kTok + 1];  // gl^k and gamma gl^(k-1), by repeated products
};
constexpr int kSmemTotal = kSmemBytes + (int)sizeof(GaeSmall);

struct WsHeader {
    uint32_t ticket, done;
    uint32_t epoch;  // launches so far (mod 2^32 - 1): the tag of this launch's records is epoch + 1
};

// The status word is optional for this entry point.
__device__ __forceinline__ void gae_raise(uint32_t *status, rl_status code) {
    if (status) raise_status(status, code);
}

__device__ __forceinline__ GaeMap map_identity() { return GaeMap{1.f, 0.f, 0.f, 0.f, kPassV | kPassRoll, 0, 0}; }
// the zero state beyond the last chunk
__device__ __forceinline__ GaeMap map_zero() { return GaeMap{0.f, 0.f, 0.f, 0.f, kClosed, 0, 0}; }

// F o G: G (the tokens to the right) acts first. kC: carry the two counts.
template <bool kC>
__device__ __forceinline__ GaeMap compose(const GaeMap &F, const GaeMap &G) {
    GaeMap r;
    r.p = F.p * G.p;
    r.q = fmaf(F.p, G.q, (G.bits & kPassV) ? F.q : 0.f);
    r.c = fmaf(F.q, G.vf, fmaf(F.p, G.c, F.c));
    r.vf = (F.bits & kPassV) ? G.vf : F.vf;
    r.bits = (F.bits & G.bits & (kPassV | kPassRoll)) | ((F.bits | G.bits) & kClosed);
    r.n_resp = kC ? F.n_resp + ((F.bits & kClosed) ? 0 : G.n_resp) : 0;
    r.n_roll = kC ? F.n_roll + ((F.bits & kPassRoll) ? G.n_roll : 0) : 0;
    return r;
}

template <bool kC>
__device__ __forceinline__ GaeMap shfl_down_map(const GaeMap &a, int off) {
    GaeMap r;
    r.p = __shfl_down_sync(kFull, a.p, off);
    r.q = __shfl_down_sync(kFull, a.q, off);
    r.c = __shfl_down_sync(kFull, a.c, off);
    r.vf = __shfl_down_sync(kFull, a.vf, off);
    r.bits = __shfl_down_sync(kFull, a.bits, off);
    r.n_resp = kC ? __shfl_down_sync(kFull, a.n_resp, off) : 0;
    r.n_roll = kC ? __shfl_down_sync(kFull, a.n_roll, off) : 0;
    return r;
}

template <bool kC>
__device__ __forceinline__ GaeMap shfl_map(const GaeMap &a, int src) {
    GaeMap r;
    r.p = __shfl_sync(kFull, a.p, src);
    r.q = __shfl_sync(kFull, a.q, src);
    r.c = __shfl_sync(kFull, a.c, src);
    r.vf = __shfl_sync(kFull, a.vf, src);
    r.bits = __shfl_sync(kFull, a.bits, src);
    r.n_resp = kC ? __shfl_sync(kFull, a.n_resp, src) : 0;
    r.n_roll = kC ? __shfl_sync(kFull, a.n_roll, src) : 0;
    return r;
}

// Inclusive suffix scan within a warp: lane l gets M_l o M_{l+1} o ... o M_31.
template <bool kC>
__device__ __forceinline__ GaeMap warp_suffix(GaeMap x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const GaeMap o = shfl_down_map<kC>(x, off);
        if (lane + off < 32) x = compose<kC>(x, o);
    }
    return x;
}

__device__ __forceinline__ uint64_t ld_word(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_word(uint64_t *p, uint32_t v, uint32_t tag) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(((uint64_t)tag << 32) | v) : "memory");
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// The map of a record, and whether all of its words carry `tag` (else it is not published yet).
__device__ __forceinline__ bool load_record(const ChunkRecord *rec, uint32_t tag, GaeMap &m) {
    uint64_t x[7];
#pragma unroll
    for (int i = 0; i < 7; ++i) x[i] = ld_word(&rec->w[i]);
    bool ok = true;
#pragma unroll
    for (int i = 0; i < 7; ++i) ok &= (uint32_t)(x[i] >> 32) == tag;
    m = GaeMap{__uint_as_float((uint32_t)x[0]), __uint_as_float((uint32_t)x[1]), __uint_as_float((uint32_t)x[2]),
               __uint_as_float((uint32_t)x[3]), (uint32_t)x[4], (int32_t)(uint32_t)x[5], (int32_t)(uint32_t)x[6]};
    return ok;
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Float offset, within a values or rewards tile, of token e of the chunk.
__device__ __forceinline__ int tile_off(int e) {
    const int row = e / kTok, col = e % kTok;
    return row * kTok + 4 * ((col >> 2) ^ (row & 7)) + (col & 3);
}

// First s in [0, S) with cu[s + 1] > x (S if none); one warp, 32-ary search.
// Terminates for any contents of cu (the span shrinks every round).
__device__ int warp_first_end_after(const int32_t *cu, int S, int x) {
    const int lane = threadIdx.x & 31;
    int lo = 0, hi = S;
    while (hi > lo) {
        const int step = (hi - lo + 31) / 32;
        const int pos = lo + lane * step;
        const bool pred = pos >= hi || __ldg(cu + pos + 1) > x;
        const unsigned b = __ballot_sync(kFull, pred);
        const int f = __ffs(b) - 1;
        if (f < 0) {
            lo = lo + 31 * step + 1;
        } else {
            hi = min(hi, lo + f * step);
            lo = f == 0 ? lo : lo + (f - 1) * step + 1;
        }
    }
    return lo;
}

// 2^k as a float, -149 <= k <= 127.
__device__ __forceinline__ float pow2i(int k) {
    return k >= -126 ? __int_as_float((k + 127) << 23) : __int_as_float(1 << (k + 149));
}

// (gamma lambda)^n as m * s1 * s2 * s3 (each s a power of two, so that a
// product with them rounds only once unless it falls below the normal range).
struct Scale {
    float m, s1, s2, s3;
};

struct ScaleArgs {
    int32_t gl_kind;
    float log2_gl_hi, log2_gl_lo;
    double log2_gl;
};

__device__ __noinline__ Scale cross_scale(int n, ScaleArgs p) {
    if (n <= 0 || p.gl_kind == 2) return Scale{1.f, 1.f, 1.f, 1.f};
    if (p.gl_kind == 1) return Scale{0.f, 1.f, 1.f, 1.f};
    // x = n log2(gamma lambda) = e + f with e an integer and |f| <= 1/2
    int e;
    float f;
    if (n < (1 << 24)) {
        const float nf = (float)n;  // exact
        const float ph = nf * p.log2_gl_hi;
        if (ph < -1000.f) return Scale{0.f, 1.f, 1.f, 1.f};
        const float pe = fmaf(nf, p.log2_gl_hi, -ph);  // the exact rounding error of ph
        const float ef = rintf(ph);
        f = (ph - ef) + fmaf(nf, p.log2_gl_lo, pe);
        e = (int)ef;
    } else {
        const double x = (double)n * p.log2_gl;
        if (x < -1000.0) return Scale{0.f, 1.f, 1.f, 1.f};
        const double ed = rint(x);
        f = (float)(x - ed);
        e = (int)ed;
    }
    if (e < -400) return Scale{0.f, 1.f, 1.f, 1.f};
    // 2^f = e^{f ln 2}: Taylor series to degree 7 (|f ln 2| <= 0.35: truncation < 1e-8)
    const float y = f * 0.69314718f;
    float m = 1.f / 5040.f;
    m = fmaf(m, y, 1.f / 720.f);
    m = fmaf(m, y, 1.f / 120.f);
    m = fmaf(m, y, 1.f / 24.f);
    m = fmaf(m, y, 1.f / 6.f);
    m = fmaf(m, y, 0.5f);
    m = fmaf(m, y, 1.f);
    m = fmaf(m, y, 1.f);
    const int e1 = max(e, -126), r1 = e - e1;
    const int e2 = max(r1, -126), e3 = r1 - e2;  // e3 >= -148
    return Scale{m, pow2i(e1), pow2i(e2), pow2i(e3)};
}

__device__ __forceinline__ float apply_scale(float a, const Scale &s) { return ((a * s.m) * s.s1) * s.s2 * s.s3; }

template <bool kCross>
__global__ void __launch_bounds__(kThreads, 3) gae_chunk_kernel(GaeParams p, const __grid_constant__ GaeMaps maps) {
    // All shared memory is dynamic, carved below: the staged rows first (1024-byte aligned for the
    // tensor copies' swizzle when the block's window allows it), then the small per-block state.
    extern __shared__ __align__(1024) unsigned char smem[];
    float *s_r = reinterpret_cast<float *>(smem + kSmemR);
    float *s_v = reinterpret_cast<float *>(smem + kSmemV);
    uint8_t *s_m = smem + kSmemM;
    GaeSmall &sm = *reinterpret_cast<GaeSmall *>(smem + kSmemBytes);
    uint32_t *s_last = sm.last;
    uint32_t *s_cont = sm.cont;
    GaeMap *s_wtot = sm.wtot;
    GaeMap *s_after = sm.after;
    int &s_k = sm.k, &s_sa = sm.sa, &s_sb = sm.sb, &s_lo = sm.lo, &s_hi = sm.hi;
    float &s_EA = sm.EA, &s_EV = sm.EV;
    int &s_EP = sm.EP, &s_ER = sm.ER;
    float *s_pow = sm.pw, *s_qpow = sm.qpw;
    uint64_t &s_bar = sm.bar;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = p.num_tokens, S = p.num_seqs;
    const int nchunks = (T + kChunk - 1) / kChunk;
    WsHeader *hdr = reinterpret_cast<WsHeader *>(p.workspace);
    ChunkRecord *recs = reinterpret_cast<ChunkRecord *>(static_cast<char *>(p.workspace) + kWsHeader);

    if (tid == 0) {
        // The blocks of a wave otherwise stay in step for the whole launch: all stage their chunks
        // at once (HBM saturated), then all fold, look back and re-walk (HBM idle). The first
        // wave's blocks on an SM start a few microseconds apart, before they take their tickets,
        // so the chunk order is unchanged and so is every result.
        if (p.stagger_ns != 0u && blockIdx.x < (unsigned)(p.stagger_sms * p.stagger_slots)) {
            const unsigned long long slot = blockIdx.x / (unsigned)p.stagger_sms;
            const unsigned long long t_start = global_ns(), dt = slot * p.stagger_ns;
            while (global_ns() - t_start < dt) __nanosleep(500);
        }
        const uint32_t ticket = atomicAdd(&hdr->ticket, 1u);
        s_k = nchunks - 1 - (int)ticket;
        sm.epoch = *reinterpret_cast<volatile uint32_t *>(&hdr->epoch);
    }
    s_last[tid] = 0u;
    s_cont[tid] = 0u;
    if (tid == 32) {
        float pw = 1.f, qw = 0.f;
        s_pow[0] = 1.f;
        s_qpow[0] = 0.f;
        for (int i = 1; i <= kTok; ++i) {
            pw = p.gl * pw;
            qw = fmaf(p.gl, qw, i == 1 ? p.gamma : 0.f);
            s_pow[i] = pw;
            s_qpow[i] = qw;
        }
    }
    __syncthreads();
    const int k = s_k;
    const uint32_t epoch = sm.epoch, tag = epoch % 0xffffffffu + 1u;  // never 0 (a zeroed workspace)
    if (!RLK_CHECK(p.status, k < nchunks)) return;
    if (k < 0) {  // a ticket counter left dirty (the workspace was not zeroed): flag and stop
        if (tid == 0) gae_raise(p.status, RL_ERR_INVALID_ARG);
        return;
    }
    const int cs = k * kChunk, ce = min(T, cs + kChunk);
    const int t0 = cs + tid * kTok;
    const bool tma = maps.ok && ce - cs == kChunk && (ptx::smem_u32(smem) & 1023u) == 0u;
    const uint32_t bar = ptx::smem_u32(&s_bar);

    // stage the chunk: tensor copies (128-byte swizzle) and one bulk copy of the mask bytes,
    // issued by one thread; else coalesced 16-byte copies
    if (tma) {
        if (tid == 0) {
            ptx::mbar_init(bar, 1);
            ptx::fence_mbar_init();
            ptx::mbar_arrive_expect_tx(bar, 2u * kChunk * 4u + kChunk);
            ptx::tma_load_2d(ptx::smem_u32(s_r), &maps.r, 0, k * kThreads, bar);
            ptx::tma_load_2d(ptx::smem_u32(s_v), &maps.v, 0, k * kThreads, bar);
            ptx::bulk_g2s(ptx::smem_u32(s_m), p.mask + cs, kChunk, bar);
        }
    } else if (p.vec && ce - cs == kChunk) {
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const int f = j * kThreads + tid;  // float4 index within the chunk
            const int off = tile_off(4 * f);
            cp_async16(s_r + off, p.rewards + cs + 4 * f);
            cp_async16(s_v + off, p.values + cs + 4 * f);
        }
#pragma unroll
        for (int j = 0; j < kChunk / 16 / kThreads; ++j) {
            const int f = j * kThreads + tid;
            cp_async16(s_m + 16 * f, p.mask + cs + 16 * f);
        }
    } else {
#pragma unroll 4
        for (int j = 0; j < kTok; ++j) {
            const int e = j * kThreads + tid, t = cs + e;
            const bool in = t < ce;
            const int off = tile_off(e);
            s_r[off] = in ? __ldg(p.rewards + t) : 0.f;
            s_v[off] = in ? __ldg(p.values + t) : 0.f;
            s_m[e] = in ? __ldg(p.mask + t) : (uint8_t)0;
        }
    }

    // the responses that end inside this chunk, the covered token range, and a slice of the offsets checked
    if (warp == 0) {
        const int sa = warp_first_end_after(p.cu_seqlens, S, cs);
        if (lane == 0) s_sa = sa;
    } else if (warp == 1) {
        const int sb = warp_first_end_after(p.cu_seqlens, S, ce) - 1;
        if (lane == 0) s_sb = sb;
    } else if (warp == 2) {
        if (lane == 0) {
            const int lo = min(max(__ldg(p.cu_seqlens), 0), T);
            s_lo = lo;
            s_hi = min(max(__ldg(p.cu_seqlens + S), lo), T);
        }
    } else {
        const int per = (S + nchunks) / nchunks;  // offsets 0..S split over the chunks
        const int a = k * per, b = min(S, a + per - 1);
        bool bad = false;
        for (int s = a + tid - 96; s <= b; s += kThreads - 96) {
            const int x = __ldg(p.cu_seqlens + s);
            bad |= x < 0 || x > T || (s < S && __ldg(p.cu_seqlens + s + 1) < x);
        }
        if (bad) gae_raise(p.status, RL_ERR_SEQLENS);
    }
    __syncthreads();
    for (int s = s_sa + tid; s <= s_sb; s += kThreads) {
        const int b = __ldg(p.cu_seqlens + s), e = __ldg(p.cu_seqlens + s + 1);
        const int j = e - 1 - cs;
        if (e > b && j >= 0 && j < kChunk) {
            atomicOr(&s_last[j >> 5], 1u << (j & 31));
            if (kCross) {
                // the rollout goes on if every following response up to the next non-empty one shares the id
                const int rid = __ldg(p.rollout_ids + s);
                bool cont = false;
                for (int u = s + 1; u < S; ++u) {
                    if (__ldg(p.rollout_ids + u) != rid) break;
                    if (__ldg(p.cu_seqlens + u + 1) > __ldg(p.cu_seqlens + u)) {
                        cont = true;
                        break;
                    }
                }
                if (cont) atomicOr(&s_cont[j >> 5], 1u << (j & 31));
            }
        }
    }
    if (tma) {
        // bounded: on a timeout the chunk's values are not valid (flagged), and the copies get one
        // more bounded wait so that none is in flight when the block exits
        if (!ptx::mbar_wait(bar, 0u)) {
            gae_raise(p.status, RL_ERR_TIMEOUT);
            if (tid == 0) ptx::mbar_wait(bar, 0u, 100000000ull);
        }
    } else {
        cp_async_wait_all();
    }
    __syncthreads();

    const uint32_t last = s_last[tid];
    const uint32_t cont = kCross ? s_cont[tid] : 0u;
    uint32_t inr, act, msk;
    {
        // bit i: token t0 + i lies in [lo, hi) / has a nonzero mask byte / is an action token
        const uint4 ma = *reinterpret_cast<const uint4 *>(s_m + kTok * tid);
        const uint4 mb4 = *reinterpret_cast<const uint4 *>(s_m + kTok * tid + 16);
        const uint32_t mw[8] = {ma.x, ma.y, ma.z, ma.w, mb4.x, mb4.y, mb4.z, mb4.w};
        uint32_t mb = 0u;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const uint32_t x = __vcmpne4(mw[w], 0u) & 0x01010101u;  // one bit per byte
            mb |= ((x * 0x10204080u) >> 28) << (4 * w);             // gathered into 4 bits
        }
        const int a = min(max(s_lo - t0, 0), kTok), b = min(max(s_hi - t0, 0), kTok);
        const uint32_t below_b = b >= 32 ? 0xffffffffu : ((1u << b) - 1u);
        inr = a < b ? (below_b & ~((1u << a) - 1u)) : 0u;
        msk = mb & inr;
        act = p.skip_observations ? msk : inr;
    }
    const float gamma = p.gamma, gl = p.gl;
    const ScaleArgs sargs{p.gl_kind, p.log2_gl_hi, p.log2_gl_lo, p.log2_gl};
    const float *row_r = s_r + tid * kTok;
    const float *row_v = s_v + tid * kTok;
    const int sw = tid & 7;  // this row's swizzle

    // fold the thread's tokens, right to left
    GaeMap F = map_identity();
    if (__popc(last) <= 1) {
        // at most one response end among them (at e): the map is the affine steps of the tokens from
        // e leftwards, from the zero state the end resets to; the tokens right of it only count
        const int e = last ? 31 - __clz(last) : -1;
        const uint32_t left = e < 0 || e == 31 ? 0xffffffffu : (2u << e) - 1u;  // tokens 0..e (all: no end)
        const uint32_t actl = act & left;
        float c = 0.f, vf = 0.f;
#pragma unroll
        for (int j = kVec - 1; j >= 0; --j) {
            const float4 r4 = *reinterpret_cast<const float4 *>(row_r + 4 * (j ^ sw));
            const float4 v4 = *reinterpret_cast<const float4 *>(row_v + 4 * (j ^ sw));
            const float rr[4] = {r4.x, r4.y, r4.z, r4.w}, vv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
            for (int u = 3; u >= 0; --u) {
                if ((actl >> (4 * j + u)) & 1u) {
                    c = fmaf(gl, c, fmaf(gamma, vf, rr[u] - vv[u]));
                    vf = vv[u];
                }
            }
        }
        const int na = __popc(actl);
        if (last == 0u) {
            const int n = kCross ? __popc(msk) : 0;
            F = GaeMap{s_pow[na], s_qpow[na], c, vf, (na ? 0u : kPassV) | kPassRoll, n, n};
        } else {
            // closed: nothing from the right reaches further left; the rollout count passes the end
            // only if the rollout goes on past it
            const bool ce = (cont >> e) & 1u;
            const int nl = kCross ? __popc(msk & left) : 0, nr = kCross ? __popc(msk & ~left) : 0;
            F = GaeMap{0.f, 0.f, c, vf, kClosed | (ce ? kPassRoll : 0u), nl, nl + (ce ? nr : 0)};
        }
    } else {
        // two or more responses end among them (responses shorter than 32 tokens): token by token
#pragma unroll 1
        for (int i = kTok - 1; i >= 0; --i) {
            const int o = 4 * ((i >> 2) ^ sw) + (i & 3);
            const float r = row_r[o], v = row_v[o];
            if ((last >> i) & 1u) {  // a response ends here: the state from the right is dropped
                const bool c = (cont >> i) & 1u;
                F.bits = kClosed | ((c && (F.bits & kPassRoll)) ? kPassRoll : 0u);
                F.p = F.q = F.c = F.vf = 0.f;
                F.n_resp = 0;
                F.n_roll = c ? F.n_roll : 0;
            }
            if ((act >> i) & 1u) {
                F.c = fmaf(gl, F.c, fmaf(gamma, F.vf, r - v));
                F.q = fmaf(gl, F.q, (F.bits & kPassV) ? gamma : 0.f);
                F.p = gl * F.p;
                F.vf = v;
                F.bits &= ~kPassV;
            }
            if (kCross && ((msk >> i) & 1u)) {
                F.n_resp += 1;
                F.n_roll += 1;
            }
        }
    }

    // exclusive suffix over the block's threads, and the chunk's map
    const GaeMap incl = warp_suffix<kCross>(F);
    if (lane == 0) s_wtot[warp] = incl;
    __syncthreads();
    GaeMap agg = map_identity();  // the chunk's map (held by warp 1)
    if (warp <= 1) {
        const GaeMap wi = warp_suffix<kCross>(lane < kThreads / 32 ? s_wtot[lane] : map_identity());
        agg = shfl_map<kCross>(wi, 0);
        if (warp == 1) {
            if (lane < 7 && k != p.withhold_chunk) {  // publish: one tagged word per lane
                const uint32_t v = lane == 0 ? __float_as_uint(agg.p)
                                 : lane == 1 ? __float_as_uint(agg.q)
                                 : lane == 2 ? __float_as_uint(agg.c)
                                 : lane == 3 ? __float_as_uint(agg.vf)
                                 : lane == 4 ? agg.bits
                                 : lane == 5 ? (uint32_t)agg.n_resp
                                             : (uint32_t)agg.n_roll;
                st_word(&recs[k].w[lane], v, tag);
            }
        } else {
            GaeMap after = shfl_down_map<kCross>(wi, 1);
            if (lane == 31) after = map_identity();
            if (lane < kThreads / 32) s_after[lane] = after;
            // Look back over the chunks to the right. The maps: composed in a
            // fixed tree up to the first chunk that holds a response end. The
            // rollout count (kCross): summed up to the first chunk with a
            // rollout end or a published inclusive count. Only the chunks up
            // to those stopping points are waited for.
            GaeMap acc = map_identity();
            int R = 0;
            bool need_map = true, need_roll = kCross;
            const unsigned long long t_begin = global_ns();
            for (int base = k + 1; need_map || need_roll; base += 32) {
                const int j = base + lane;
                bool ready = j >= nchunks;  // beyond the last chunk: the zero state
                GaeMap m = map_zero();
                bool incl = false;  // the inclusive rollout count is published too
                int incl_roll = 0;
                int fcm = -1, fcr = -1;
                while (true) {
                    if (!ready) {
                        GaeMap mj;
                        const uint64_t w7 = kCross ? ld_word(&recs[j].w[7]) : 0ull;
                        if (load_record(recs + j, tag, mj)) {
                            ready = true;
                            m = mj;
                            incl = kCross && (uint32_t)(w7 >> 32) == tag;
                            incl_roll = (int)(uint32_t)w7;
                        } else if (global_ns() - t_begin > p.wait_ns) {
                            gae_raise(p.status, RL_ERR_TIMEOUT);
                            ready = true;  // treated as a response end
                        }
                    }
                    const unsigned rdy = __ballot_sync(kFull, ready);
                    const unsigned stm = __ballot_sync(kFull, ready && (m.bits & kClosed));
                    const unsigned str = __ballot_sync(kFull, ready && (incl || !(m.bits & kPassRoll)));
                    const int pre = rdy == kFull ? 32 : __ffs(~rdy) - 1;  // lanes 0..pre-1 are ready
                    fcm = __ffs(stm) - 1;
                    fcr = __ffs(str) - 1;
                    const bool okm = !need_map || pre == 32 || (fcm >= 0 && fcm < pre);
                    const bool okr = !need_roll || pre == 32 || (fcr >= 0 && fcr < pre);
                    if (okm && okr) break;
                    __nanosleep(32);
                }
                if (need_map) {
                    const GaeMap mm = (fcm >= 0 && lane > fcm) ? map_identity() : m;
                    acc = compose<kCross>(acc, shfl_map<kCross>(warp_suffix<kCross>(mm), 0));
                    need_map = fcm < 0;
                }
                if (kCross && need_roll) {
                    int val = incl ? incl_roll : m.n_roll;
                    if (fcr >= 0 && lane > fcr) val = 0;
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) val += __shfl_xor_sync(kFull, val, off);
                    R += val;
                    need_roll = fcr < 0;
                }
            }
            if (lane == 0) {  // the state arriving at the chunk's right edge
                s_EA = acc.c;
                s_EV = acc.vf;
                s_EP = acc.n_resp;
                s_ER = R;
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        if (lane == 0) {
            if (kCross && k != p.withhold_chunk)
                st_word(&recs[k].w[7], (uint32_t)(agg.n_roll + ((agg.bits & kPassRoll) ? s_ER : 0)), tag);
        }
        // past the look-back: the last block to get here leaves the workspace ready for the next launch
        uint32_t d = 0u;
        if (lane == 0) asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(d) : "l"(&hdr->done) : "memory");
        d = __shfl_sync(kFull, d, 0);
        if (d == (uint32_t)nchunks - 1u && lane == 0) {
            // every block has read the epoch (before its look-back): the next launch's tag is new
            hdr->ticket = 0u;
            hdr->done = 0u;
            hdr->epoch = epoch + 1u;
        }
    }

    // the state arriving at this thread's tokens
    GaeMap right = shfl_down_map<kCross>(incl, 1);
    if (lane == 31) right = map_identity();
    const GaeMap X = compose<kCross>(right, s_after[warp]);
    float A = fmaf(X.p, s_EA, fmaf(X.q, s_EV, X.c));
    float V = (X.bits & kPassV) ? s_EV : X.vf;
    int P = X.n_resp + ((X.bits & kClosed) ? 0 : s_EP);
    int R = X.n_roll + ((X.bits & kPassRoll) ? s_ER : 0);

    // re-walk: advantages (and returns), scaled per response, written in place of the staged rows
    const bool want_ret = p.returns != nullptr;
    float *wrow_r = s_r + tid * kTok;
    float *wrow_v = s_v + tid * kTok;
    if (last == 0u) {
        // every token here belongs to one response: one discount factor
        Scale sc{1.f, 1.f, 1.f, 1.f};
        if (kCross) sc = cross_scale(R - P, sargs);
        // a factor whose product with m stays normal folds into one multiplication
        const bool single = sc.s2 == 1.f && sc.s3 == 1.f && (sc.m == 0.f || sc.s1 >= 0x1p-125f);
        const float f1 = sc.m * sc.s1;
#pragma unroll
        for (int j = kVec - 1; j >= 0; --j) {
            const float4 r4 = *reinterpret_cast<const float4 *>(row_r + 4 * (j ^ sw));
            const float4 v4 = *reinterpret_cast<const float4 *>(row_v + 4 * (j ^ sw));
            const float rr[4] = {r4.x, r4.y, r4.z, r4.w}, vv[4] = {v4.x, v4.y, v4.z, v4.w};
            float out[4], ret[4];
#pragma unroll
            for (int u = 3; u >= 0; --u) {
                out[u] = 0.f;
                ret[u] = 0.f;
                if ((act >> (4 * j + u)) & 1u) {
                    A = fmaf(gl, A, fmaf(gamma, V, rr[u] - vv[u]));
                    V = vv[u];
                    const float o = !kCross ? A : (single ? A * f1 : apply_scale(A, sc));
                    out[u] = o;
                    ret[u] = o + vv[u];
                }
            }
            *reinterpret_cast<float4 *>(wrow_r + 4 * (j ^ sw)) = make_float4(out[0], out[1], out[2], out[3]);
            if (want_ret)
                *reinterpret_cast<float4 *>(wrow_v + 4 * (j ^ sw)) = make_float4(ret[0], ret[1], ret[2], ret[3]);
        }
    } else if (__popc(last) == 1) {
        // one response end among them (at e): the tokens right of it with the arriving state and
        // their response's factor, then from e leftwards from the zero state with their own factor
        // (the same steps, in the same order, as the token-by-token walk below)
        const int e = 31 - __clz(last);
        Scale scR{1.f, 1.f, 1.f, 1.f}, scL{1.f, 1.f, 1.f, 1.f};
        if (kCross) {
            const uint32_t right = e == 31 ? 0u : ~((2u << e) - 1u);
            scR = cross_scale(R - P, sargs);
            scL = cross_scale(((cont >> e) & 1u) ? R + __popc(msk & right) : 0, sargs);
        }
#pragma unroll
        for (int j = kVec - 1; j >= 0; --j) {
            const float4 r4 = *reinterpret_cast<const float4 *>(row_r + 4 * (j ^ sw));
            const float4 v4 = *reinterpret_cast<const float4 *>(row_v + 4 * (j ^ sw));
            const float rr[4] = {r4.x, r4.y, r4.z, r4.w}, vv[4] = {v4.x, v4.y, v4.z, v4.w};
            float out[4], ret[4];
#pragma unroll
            for (int u = 3; u >= 0; --u) {
                const int i = 4 * j + u;
                out[u] = 0.f;
                ret[u] = 0.f;
                if (i == e) A = V = 0.f;
                if ((act >> i) & 1u) {
                    A = fmaf(gl, A, fmaf(gamma, V, rr[u] - vv[u]));
                    V = vv[u];
                    const float o = !kCross ? A : apply_scale(A, i <= e ? scL : scR);
                    out[u] = o;
                    ret[u] = o + vv[u];
                }
            }
            *reinterpret_cast<float4 *>(wrow_r + 4 * (j ^ sw)) = make_float4(out[0], out[1], out[2], out[3]);
            if (want_ret)
                *reinterpret_cast<float4 *>(wrow_v + 4 * (j ^ sw)) = make_float4(ret[0], ret[1], ret[2], ret[3]);
        }
    } else {
        int cached = -1;
        Scale sc{1.f, 1.f, 1.f, 1.f};
#pragma unroll 1
        for (int i = kTok - 1; i >= 0; --i) {
            const int o = 4 * ((i >> 2) ^ sw) + (i & 3);
            const float r = row_r[o], v = row_v[o];
            if ((last >> i) & 1u) {
                A = V = 0.f;
                P = 0;
                R = ((cont >> i) & 1u) ? R : 0;
            }
            if (kCross && ((msk >> i) & 1u)) {
                P += 1;
                R += 1;
            }
            float out = 0.f, ret = 0.f;
            if ((act >> i) & 1u) {
                A = fmaf(gl, A, fmaf(gamma, V, r - v));
                V = v;
                out = A;
                if (kCross) {
                    const int later = R - P;
                    if (later != cached) {
                        sc = cross_scale(later, sargs);
                        cached = later;
                    }
                    out = apply_scale(out, sc);
                }
                ret = out + v;
            }
            wrow_r[o] = out;
            if (want_ret) wrow_v[o] = ret;
        }
    }

    // store: each warp's 32 rows by tensor stores as soon as the warp is done, when the chunk
    // lies inside [lo, hi); else coalesced 16-byte stores of the rows inside [lo, hi), token by
    // token elsewhere
    const int a_in = min(max(s_lo - cs, 0), kChunk), b_in = min(max(min(s_hi, ce) - cs, 0), kChunk);
    if (tma && a_in == 0 && b_in == kChunk) {
        ptx::fence_proxy_async_smem();  // this thread's row, written above, is visible to the copy
        __syncwarp();
        if (lane == 0) {
            const int y = k * kThreads + warp * 32;
            ptx::tma_store_2d(&maps.adv, 0, y, ptx::smem_u32(s_r + warp * 32 * kTok));
            if (want_ret) ptx::tma_store_2d(&maps.ret, 0, y, ptx::smem_u32(s_v + warp * 32 * kTok));
            ptx::bulk_commit_group();
            ptx::bulk_wait_group_read<0>();  // shared memory is read before the warp (and block) exits
        }
        return;
    }
    __syncthreads();
    if (p.vec) {
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const int f = j * kThreads + tid;
            const int e0 = 4 * f, off = tile_off(e0);
            if (e0 >= a_in && e0 + 4 <= b_in) {
                __stcs(reinterpret_cast<float4 *>(p.adv + cs) + f, *reinterpret_cast<const float4 *>(s_r + off));
                if (want_ret)
                    __stcs(reinterpret_cast<float4 *>(p.returns + cs) + f, *reinterpret_cast<const float4 *>(s_v + off));
            } else {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (e0 + u < a_in || e0 + u >= b_in) continue;
                    p.adv[cs + e0 + u] = s_r[off + u];
                    if (want_ret) p.returns[cs + e0 + u] = s_v[off + u];
                }
            }
        }
    } else {
#pragma unroll 4
        for (int j = 0; j < kTok; ++j) {
            const int e = j * kThreads + tid;
            if (e < a_in || e >= b_in) continue;
            const int off = tile_off(e);
            p.adv[cs + e] = s_r[off];
            if (want_ret) p.returns[cs + e] = s_v[off];
        }
    }
}

// [rows x 32] fp32 view of a token array, boxes of box_rows rows, 128-byte swizzle.
bool token_map(CUtensorMap *m, const float *base, int64_t rows, uint32_t box_rows) {
    return make_tmap_sw128(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, rows, kTok, kTok, kTok, box_rows);
}

template <bool kCross>
cudaError_t launch_chunks(GaeParams p, unsigned nchunks, cudaStream_t stream) {
    static std::atomic<uint64_t> configured{0};  // one bit per device
    static int sms[64], slots[64];               // per device: SMs, and blocks resident per SM
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        e = cudaFuncSetAttribute(gae_chunk_kernel<kCross>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemTotal);
        if (e != cudaSuccess) return e;
        int n = 0, occ = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, gae_chunk_kernel<kCross>, kThreads, kSmemTotal);
        if (e != cudaSuccess) return e;
        sms[dev & 63] = n;
        slots[dev & 63] = occ;
        configured.fetch_or(bit);
    }
    // stagger only launches of several waves: the first wave's delay (up to 2 x 3 us with three
    // blocks per SM) is paid once
    p.stagger_sms = sms[dev & 63];
    p.stagger_slots = slots[dev & 63];
    p.stagger_ns = (p.stagger_slots > 1 && (int64_t)nchunks >= 4ll * p.stagger_sms * p.stagger_slots) ? kStaggerNs : 0u;
    GaeMaps maps{};
    const int64_t rows = p.num_tokens / kTok;
    if (p.vec && rows >= kThreads) {
        maps.ok = token_map(&maps.r, p.rewards, rows, kThreads) && token_map(&maps.v, p.values, rows, kThreads) &&
                  token_map(&maps.adv, p.adv, rows, 32) && (!p.returns || token_map(&maps.ret, p.returns, rows, 32));
        if (!p.returns) maps.ret = maps.adv;
    }
    gae_chunk_kernel<kCross><<<nchunks, kThreads, kSmemTotal, stream>>>(p, maps);
    return cudaGetLastError();
}

}  // namespace

size_t gae_workspace_bytes(int64_t num_tokens) {
    const int64_t nchunks = (num_tokens + kChunk - 1) / kChunk;
    return (size_t)(kWsHeader + nchunks * (int64_t)sizeof(ChunkRecord));
}

cudaError_t launch_gae(GaeParams p, cudaStream_t stream) {
    if (p.num_tokens <= 0 || p.num_seqs <= 0) return cudaSuccess;
    const int64_t nchunks = (p.num_tokens + kChunk - 1) / kChunk;
    const uintptr_t al = reinterpret_cast<uintptr_t>(p.rewards) | reinterpret_cast<uintptr_t>(p.values) |
                         reinterpret_cast<uintptr_t>(p.mask) | reinterpret_cast<uintptr_t>(p.adv) |
                         reinterpret_cast<uintptr_t>(p.returns);
    p.vec = (al & 15u) == 0u;
    return p.rollout_ids ? launch_chunks<true>(p, (unsigned)nchunks, stream)
                         : launch_chunks<false>(p, (unsigned)nchunks, stream);
}

}  // namespace rlk

