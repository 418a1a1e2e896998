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
// Design. The token range is cut into fixed chunks of 4096 tokens; one block
// per chunk, chunks handed out right to left by an atomic ticket. What a run
// of tokens does to the state (A, V) arriving from its right is affine,
//   A <- p A + q V + c,   V <- V (no action token, no response end) or vf,
// and a response end resets the state to zero; two integer counts ride along
// (mask=1 tokens to the right within the response and within the rollout),
// from which N_{>s} is their difference. Such maps compose associatively.
// A block folds its 16 tokens per thread into a map (fp32), scans the 256
// maps of the block with a fixed tree, publishes the chunk's map, and then
// looks back: it composes the published maps of the chunks to its right, in
// a fixed order and tree, up to and including the first one that holds a
// response end (the state further right cannot reach it). The rollout count
// (an integer, so any order gives the same sum) uses the classic decoupled
// look-back with inclusive values. Every floating-point result depends only on
// the inputs, never on timing: bit-identical from run to run.
// Waits on another chunk's record are bounded (1 s of %globaltimer); a wait
// that runs out raises RL_ERR_TIMEOUT and treats that chunk as a response end.
// The last block to finish its look-back clears the flags and the ticket (the
// records themselves are only read under a flag set by the same launch), so
// the workspace is ready for the next launch. The chunk is staged in
// shared memory by coalesced 16-byte asynchronous copies, so that no token
// value occupies a register across the scan and the look-back.
#include "common.cuh"

namespace rlk {

namespace {

constexpr int kThreads = 256;
constexpr int kTok = 16;                 // consecutive tokens per thread
constexpr int kChunk = kThreads * kTok;  // tokens per chunk
constexpr int kWords = kChunk / 32;
constexpr unsigned kFull = 0xffffffffu;
constexpr unsigned long long kWaitNs = 1000000000ull;

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
// records as flags). flag: 0 nothing yet, 1 the map is published, 2 the
// inclusive rollout count too.
struct ChunkRecord {
    float p, q, c, vf;
    uint32_t bits;
    int32_t n_resp, n_roll, roll_incl;
    uint32_t flag, pad[3];
};
static_assert(sizeof(ChunkRecord) == 48, "record size");
constexpr int kWsHeader = 256;

struct WsHeader {
    uint32_t ticket, done;
};

// The status word is optional for this entry point.
__device__ __forceinline__ void gae_raise(uint32_t *status, rl_status code) {
    if (status) raise_status(status, code);
}

__device__ __forceinline__ GaeMap map_identity() { return GaeMap{1.f, 0.f, 0.f, 0.f, kPassV | kPassRoll, 0, 0}; }
// the zero state beyond the last chunk
__device__ __forceinline__ GaeMap map_zero() { return GaeMap{0.f, 0.f, 0.f, 0.f, kClosed, 0, 0}; }

// F o G: G (the tokens to the right) acts first.
__device__ __forceinline__ GaeMap compose(const GaeMap &F, const GaeMap &G) {
    GaeMap r;
    r.p = F.p * G.p;
    r.q = fmaf(F.p, G.q, (G.bits & kPassV) ? F.q : 0.f);
    r.c = fmaf(F.q, G.vf, fmaf(F.p, G.c, F.c));
    r.vf = (F.bits & kPassV) ? G.vf : F.vf;
    r.bits = (F.bits & G.bits & (kPassV | kPassRoll)) | ((F.bits | G.bits) & kClosed);
    r.n_resp = F.n_resp + ((F.bits & kClosed) ? 0 : G.n_resp);
    r.n_roll = F.n_roll + ((F.bits & kPassRoll) ? G.n_roll : 0);
    return r;
}

__device__ __forceinline__ GaeMap shfl_down_map(const GaeMap &a, int off) {
    GaeMap r;
    r.p = __shfl_down_sync(kFull, a.p, off);
    r.q = __shfl_down_sync(kFull, a.q, off);
    r.c = __shfl_down_sync(kFull, a.c, off);
    r.vf = __shfl_down_sync(kFull, a.vf, off);
    r.bits = __shfl_down_sync(kFull, a.bits, off);
    r.n_resp = __shfl_down_sync(kFull, a.n_resp, off);
    r.n_roll = __shfl_down_sync(kFull, a.n_roll, off);
    return r;
}

__device__ __forceinline__ GaeMap shfl_map(const GaeMap &a, int src) {
    GaeMap r;
    r.p = __shfl_sync(kFull, a.p, src);
    r.q = __shfl_sync(kFull, a.q, src);
    r.c = __shfl_sync(kFull, a.c, src);
    r.vf = __shfl_sync(kFull, a.vf, src);
    r.bits = __shfl_sync(kFull, a.bits, src);
    r.n_resp = __shfl_sync(kFull, a.n_resp, src);
    r.n_roll = __shfl_sync(kFull, a.n_roll, src);
    return r;
}

// Inclusive suffix scan within a warp: lane l gets M_l o M_{l+1} o ... o M_31.
__device__ __forceinline__ GaeMap warp_suffix(GaeMap x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const GaeMap o = shfl_down_map(x, off);
        if (lane + off < 32) x = compose(x, o);
    }
    return x;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits (bounded) until *flag >= want; returns the flag, 0 on timeout.
__device__ __forceinline__ uint32_t wait_flag(const uint32_t *flag, uint32_t want, uint32_t *status) {
    uint32_t f = ld_acquire(flag);
    if (f >= want) return f;
    const unsigned long long t0 = global_ns();
    while (true) {
        __nanosleep(64);
        f = ld_acquire(flag);
        if (f >= want) return f;
        if (global_ns() - t0 > kWaitNs) {
            gae_raise(status, RL_ERR_TIMEOUT);
            return 0;
        }
    }
}

__device__ __forceinline__ GaeMap load_record(const ChunkRecord *rec) {
    const float4 a = __ldcg(reinterpret_cast<const float4 *>(rec));
    const int4 b = __ldcg(reinterpret_cast<const int4 *>(rec) + 1);
    return GaeMap{a.x, a.y, a.z, a.w, (uint32_t)b.x, b.y, b.z};
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

__device__ Scale cross_scale(int n, const GaeParams &p) {
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

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Shared-memory rows of one thread's 16 tokens: 64 bytes of data at a stride of
// 80 bytes, so that the 16-byte reads of a quarter warp hit distinct banks.
constexpr int kRowFloats = kTok + 4;

template <bool kCross>
__global__ void __launch_bounds__(kThreads, 4) gae_chunk_kernel(GaeParams p) {
    __shared__ __align__(16) float s_r[kThreads * kRowFloats];
    __shared__ __align__(16) float s_v[kThreads * kRowFloats];
    __shared__ __align__(16) uint32_t s_m[kThreads * kTok / 4];
    __shared__ uint32_t s_last[kWords];  // bit: the token is the last of its response
    __shared__ uint32_t s_cont[kWords];  // bit: ... and its rollout continues into the next response
    __shared__ GaeMap s_wtot[kThreads / 32];
    __shared__ GaeMap s_after[kThreads / 32];
    __shared__ int s_k, s_sa, s_sb, s_lo, s_hi;
    __shared__ float s_EA, s_EV;
    __shared__ int s_EP, s_ER;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = p.num_tokens, S = p.num_seqs;
    const int nchunks = (T + kChunk - 1) / kChunk;
    WsHeader *hdr = reinterpret_cast<WsHeader *>(p.workspace);
    ChunkRecord *recs = reinterpret_cast<ChunkRecord *>(static_cast<char *>(p.workspace) + kWsHeader);

    if (tid == 0) {
        const uint32_t ticket = atomicAdd(&hdr->ticket, 1u);
        s_k = nchunks - 1 - (int)ticket;
    }
    if (tid < kWords) {
        s_last[tid] = 0u;
        s_cont[tid] = 0u;
    }
    __syncthreads();
    const int k = s_k;
    if (k < 0) {  // a ticket counter left dirty (the workspace was not zeroed): flag and stop
        if (tid == 0) gae_raise(p.status, RL_ERR_INVALID_ARG);
        return;
    }
    const int cs = k * kChunk, ce = min(T, cs + kChunk);
    const int t0 = cs + tid * kTok;

    // stage the chunk: coalesced 16-byte copies straight into shared memory
    if (p.vec && ce - cs == kChunk) {
#pragma unroll
        for (int j = 0; j < kTok / 4; ++j) {
            const int f = j * kThreads + tid;  // float4 index within the chunk
            const int off = (f >> 2) * kRowFloats + (f & 3) * 4;
            cp_async16(s_r + off, p.rewards + cs + 4 * f);
            cp_async16(s_v + off, p.values + cs + 4 * f);
        }
        cp_async16(s_m + 4 * tid, p.mask + cs + kTok * tid);
    } else {
#pragma unroll 4
        for (int j = 0; j < kTok; ++j) {
            const int e = j * kThreads + tid, t = cs + e;
            const bool in = t < ce;
            const int off = (e / kTok) * kRowFloats + e % kTok;
            s_r[off] = in ? __ldg(p.rewards + t) : 0.f;
            s_v[off] = in ? __ldg(p.values + t) : 0.f;
            reinterpret_cast<uint8_t *>(s_m)[e] = in ? __ldg(p.mask + t) : (uint8_t)0;
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
    cp_async_wait_all();
    __syncthreads();

    const uint32_t last = (s_last[tid >> 1] >> (16 * (tid & 1))) & 0xffffu;
    const uint32_t cont = kCross ? (s_cont[tid >> 1] >> (16 * (tid & 1))) & 0xffffu : 0u;
    uint32_t inr = 0u, act = 0u, msk = 0u;
    {
        const uint4 m4 = *reinterpret_cast<const uint4 *>(s_m + 4 * tid);
        const uint32_t mw[4] = {m4.x, m4.y, m4.z, m4.w};
        const int lo = s_lo, hi = s_hi;
#pragma unroll
        for (int i = 0; i < kTok; ++i) {
            const int t = t0 + i;
            const bool in = t >= lo && t < hi;
            const bool m = ((mw[i >> 2] >> (8 * (i & 3))) & 0xffu) != 0u;
            inr |= (uint32_t)in << i;
            msk |= (uint32_t)(in && m) << i;
            act |= (uint32_t)(in && (m || !p.skip_observations)) << i;
        }
    }
    const float gamma = p.gamma, gl = p.gl;
    const float *row_r = s_r + tid * kRowFloats;
    const float *row_v = s_v + tid * kRowFloats;

    // fold the thread's tokens, right to left
    GaeMap F = map_identity();
#pragma unroll
    for (int j = kTok / 4 - 1; j >= 0; --j) {
        const float4 r4 = *reinterpret_cast<const float4 *>(row_r + 4 * j);
        const float4 v4 = *reinterpret_cast<const float4 *>(row_v + 4 * j);
        const float rr[4] = {r4.x, r4.y, r4.z, r4.w}, vv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
        for (int u = 3; u >= 0; --u) {
            const int i = 4 * j + u;
            if ((last >> i) & 1u) {  // a response ends here: the state from the right is dropped
                const bool c = (cont >> i) & 1u;
                F.bits = kClosed | ((c && (F.bits & kPassRoll)) ? kPassRoll : 0u);
                F.p = F.q = F.c = F.vf = 0.f;
                F.n_resp = 0;
                F.n_roll = c ? F.n_roll : 0;
            }
            if ((act >> i) & 1u) {
                F.c = fmaf(gl, F.c, fmaf(gamma, F.vf, rr[u] - vv[u]));
                F.q = fmaf(gl, F.q, (F.bits & kPassV) ? gamma : 0.f);
                F.p = gl * F.p;
                F.vf = vv[u];
                F.bits &= ~kPassV;
            }
            if (kCross && ((msk >> i) & 1u)) {
                F.n_resp += 1;
                F.n_roll += 1;
            }
        }
    }

    // exclusive suffix over the block's threads, and the chunk's map
    const GaeMap incl = warp_suffix(F);
    if (lane == 0) s_wtot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const GaeMap wi = warp_suffix(lane < kThreads / 32 ? s_wtot[lane] : map_identity());
        GaeMap after = shfl_down_map(wi, 1);
        if (lane == 31) after = map_identity();
        if (lane < kThreads / 32) s_after[lane] = after;
        const GaeMap agg = shfl_map(wi, 0);
        if (lane == 0) {
            ChunkRecord *rec = recs + k;
            *reinterpret_cast<float4 *>(rec) = make_float4(agg.p, agg.q, agg.c, agg.vf);
            *(reinterpret_cast<int4 *>(rec) + 1) = make_int4((int)agg.bits, agg.n_resp, agg.n_roll, 0);
            st_release(&rec->flag, 1u);
        }
        // Look back over the chunks to the right. The maps: composed in a fixed
        // tree up to the first chunk that holds a response end. The rollout
        // count (kCross): summed up to the first chunk with a rollout end or an
        // inclusive count.
        GaeMap acc = map_identity();
        int R = 0;
        bool need_map = true, need_roll = kCross;
        for (int base = k + 1; need_map || need_roll; base += 32) {
            const int j = base + lane;
            GaeMap m = map_zero();
            uint32_t f = 0u;
            int incl_roll = 0;
            if (j < nchunks) {
                f = wait_flag(&recs[j].flag, 1u, p.status);
                if (f) m = load_record(recs + j);
                if (kCross && f >= 2u) incl_roll = __ldcg(&recs[j].roll_incl);
            }
            if (need_map) {
                const unsigned cb = __ballot_sync(kFull, (m.bits & kClosed) != 0u);
                const int fc = __ffs(cb) - 1;
                GaeMap mm = (fc >= 0 && lane > fc) ? map_identity() : m;
                acc = compose(acc, shfl_map(warp_suffix(mm), 0));
                need_map = fc < 0;
            }
            if (kCross && need_roll) {
                const bool stop = f >= 2u || (m.bits & kPassRoll) == 0u;
                const unsigned sb = __ballot_sync(kFull, stop);
                const int fs = __ffs(sb) - 1;
                int val = f >= 2u ? incl_roll : m.n_roll;
                if (fs >= 0 && lane > fs) val = 0;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) val += __shfl_xor_sync(kFull, val, off);
                R += val;
                need_roll = fs < 0;
            }
        }
        if (lane == 0) {
            if (kCross) {
                recs[k].roll_incl = agg.n_roll + ((agg.bits & kPassRoll) ? R : 0);
                st_release(&recs[k].flag, 2u);
            }
            // the state arriving at the chunk's right edge
            s_EA = acc.c;
            s_EV = acc.vf;
            s_EP = acc.n_resp;
            s_ER = R;
        }
    }
    __syncthreads();
    if (warp == 0) {
        // past the look-back: the last block to get here leaves the workspace zeroed for the next launch
        uint32_t d = 0u;
        if (lane == 0) asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(d) : "l"(&hdr->done) : "memory");
        d = __shfl_sync(kFull, d, 0);
        if (d == (uint32_t)nchunks - 1u) {
            for (int j = lane; j < nchunks; j += 32) recs[j].flag = 0u;
            if (lane == 0) {
                hdr->ticket = 0u;
                hdr->done = 0u;
            }
        }
    }

    // the state arriving at this thread's tokens
    GaeMap right = shfl_down_map(incl, 1);
    if (lane == 31) right = map_identity();
    const GaeMap X = compose(right, s_after[warp]);
    float A = fmaf(X.p, s_EA, fmaf(X.q, s_EV, X.c));
    float V = (X.bits & kPassV) ? s_EV : X.vf;
    int P = X.n_resp + ((X.bits & kClosed) ? 0 : s_EP);
    int R = X.n_roll + ((X.bits & kPassRoll) ? s_ER : 0);

    // re-walk: advantages, scaled per response; written 4 tokens at a time
    const bool vec_out = p.vec && inr == 0xffffu;
    int cached = -1;
    Scale sc{1.f, 1.f, 1.f, 1.f};
#pragma unroll
    for (int j = kTok / 4 - 1; j >= 0; --j) {
        const float4 r4 = *reinterpret_cast<const float4 *>(row_r + 4 * j);
        const float4 v4 = *reinterpret_cast<const float4 *>(row_v + 4 * j);
        const float rr[4] = {r4.x, r4.y, r4.z, r4.w}, vv[4] = {v4.x, v4.y, v4.z, v4.w};
        float out[4], ret[4];
#pragma unroll
        for (int u = 3; u >= 0; --u) {
            const int i = 4 * j + u;
            if ((last >> i) & 1u) {
                A = V = 0.f;
                P = 0;
                R = ((cont >> i) & 1u) ? R : 0;
            }
            if (kCross && ((msk >> i) & 1u)) {
                P += 1;
                R += 1;
            }
            out[u] = 0.f;
            ret[u] = 0.f;
            if ((act >> i) & 1u) {
                A = fmaf(gl, A, fmaf(gamma, V, rr[u] - vv[u]));
                V = vv[u];
                float o = A;
                if (kCross) {
                    const int later = R - P;
                    if (later != cached) {
                        sc = cross_scale(later, p);
                        cached = later;
                    }
                    o = apply_scale(o, sc);
                }
                out[u] = o;
                ret[u] = o + vv[u];
            }
        }
        if (vec_out) {
            __stcs(reinterpret_cast<float4 *>(p.adv + t0) + j, make_float4(out[0], out[1], out[2], out[3]));
            if (p.returns)
                __stcs(reinterpret_cast<float4 *>(p.returns + t0) + j, make_float4(ret[0], ret[1], ret[2], ret[3]));
        } else {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = 4 * j + u;
                if (!((inr >> i) & 1u)) continue;
                p.adv[t0 + i] = out[u];
                if (p.returns) p.returns[t0 + i] = ret[u];
            }
        }
    }
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
    if (p.rollout_ids)
        gae_chunk_kernel<true><<<(unsigned)nchunks, kThreads, 0, stream>>>(p);
    else
        gae_chunk_kernel<false><<<(unsigned)nchunks, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace rlk
