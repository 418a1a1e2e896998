// The library handle behind rl_loss_t (internal; shared by the C-ABI files).
#pragma once

#include <cuda_runtime.h>

#include <vector>

#include "common.cuh"

// Kernel classes timed by rl_loss_profile_start / rl_loss_profile_read.
enum RlKernelClass {
    kSegPrep = 0,
    kTokenPrep,
    kRowLoss,
    kSegReduce,
    kFinalReduce,
    kProjGemm,
    kProjRows,
    kProjBwd,     // both products of the projection backward (one tcgen05 launch per chunk)
    kEntropyFix,  // the entropy of rows holding -inf logits
    kNumKernels
};
static const char *const kKernelNames[kNumKernels] = {"seg_prep",  "token_prep", "row_loss", "seg_reduce",
                                                      "final_reduce", "proj_gemm", "proj_rows", "proj_bwd",
                                                      "entropy_fix"};
constexpr size_t kProfSlotsPerCall = 160;  // enough for a projection call of 32 chunks (or a host call of 64 blocks)
constexpr int kMaxCopyChunks = 64;         // logits blocks of rl_loss_forward_backward_from_host

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct rl_loss_handle_s {
    rl_loss_config cfg;
    int device;
    rlk::LossConsts consts;
    // workspace (one cudaMalloc, carved below)
    void *ws;
    size_t ws_bytes;
    uint32_t *status;
    float *seq_adv, *seq_w;
    double *seq_w64, *seq_obj, *seq_ent;
    int32_t *seq_n, *seq_cnt;
    float *tok_obj, *tok_ent;
    uint8_t *tok_flags;
    uint8_t *tok_fix;  // rows whose entropy the fix kernel redoes (zero between calls)
    float4 *tok_rec;
    uint32_t *tok_meta;
    float *loss_scratch;
    // bookkeeping
    int64_t launches;
    cudaError_t last_cuda_error;  // the CUDA error behind the last RL_ERR_CUDA of this handle

    // profiling: one event pair per timed launch
    std::vector<cudaEvent_t> prof_events;  // [capacity][2]
    std::vector<int> prof_cls;             // kernel class of each used slot
    int prof_capacity = 0, prof_used = 0;

    // fused projection path (rl_loss_projection_setup)
    int32_t proj_hidden = 0, proj_chunk = 0, proj_n_tiles = 0;
    int64_t proj_ldp = 0;
    void *proj_ws = nullptr;  // one cudaMalloc: the bf16 chunk, statistics, block references, target logits
    void *proj_p = nullptr;   // [chunk x ldp] bf16: scaled probabilities, then dZ in place
    float4 *proj_stats = nullptr;
    float4 *proj_refs = nullptr;
    float *proj_zy = nullptr;

    bool prof_reset(size_t slots) {
        for (cudaEvent_t e : prof_events) cudaEventDestroy(e);
        prof_events.assign(2 * slots, nullptr);
        prof_cls.assign(slots, 0);
        prof_capacity = 0;
        prof_used = 0;
        for (auto &e : prof_events)
            if (cudaEventCreate(&e) != cudaSuccess) return false;
        prof_capacity = (int)slots;
        return true;
    }
    // Returns the slot to close with prof_end, or -1 when not recording.
    int prof_begin(int cls, cudaStream_t stream) {
        if (prof_used >= prof_capacity) return -1;
        const int s = prof_used++;
        prof_cls[s] = cls;
        cudaEventRecord(prof_events[2 * (size_t)s], stream);
        return s;
    }
    void prof_end(int slot, cudaStream_t stream) {
        if (slot >= 0) cudaEventRecord(prof_events[2 * (size_t)slot + 1], stream);
    }
    void proj_release();  // defined with the projection path

    // host-input path (rl_loss_forward_backward_from_host): a copy stream and its events, made on first use
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t copy_entry = nullptr;
    cudaEvent_t copy_done[kMaxCopyChunks] = {};

    cudaError_t copy_setup() {
        if (copy_stream) return cudaSuccess;
        cudaStream_t st = nullptr;
        cudaError_t e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
        if (e != cudaSuccess) return e;
        cudaEvent_t ev[kMaxCopyChunks + 1] = {};
        int made = 0;
        for (; made < kMaxCopyChunks + 1 && e == cudaSuccess; ++made)
            e = cudaEventCreateWithFlags(&ev[made], cudaEventDisableTiming);
        if (e != cudaSuccess) {
            for (int i = 0; i < made; ++i)
                if (ev[i]) cudaEventDestroy(ev[i]);
            cudaStreamDestroy(st);
            return e;
        }
        copy_entry = ev[0];
        for (int i = 0; i < kMaxCopyChunks; ++i) copy_done[i] = ev[i + 1];
        copy_stream = st;
        return cudaSuccess;
    }
    void copy_release() {
        if (!copy_stream) return;
        cudaEventDestroy(copy_entry);
        for (cudaEvent_t e : copy_done) cudaEventDestroy(e);
        cudaStreamDestroy(copy_stream);
        copy_stream = nullptr;
    }
};
