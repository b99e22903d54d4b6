// The persistent single-launch batch-1 decode kernel (persistent.cu).
#pragma once

#include "common.cuh"
#include "ctx.h"

namespace qwen2 {

constexpr int kPersistStage = 28672;  // bytes per shared-memory ring stage (16 rows of 896 f16)
constexpr int kPersistStages = 6;     // ring depth (168 KB)

struct PersistentArgs {
    const PersistLayer* layers;
    const __half* E;    // token embedding [V][H]
    const __half* Wlm;  // LM head [V][H] (E itself when tied)
    const float* final_norm;
    float* kv;
    const float2* rope;
    int* tok;
    int* pos;
    int* slot;
    int* step;
    int* ids_hist;
    int hist_stride;
    unsigned* epoch;
    unsigned long long* pk;
    float* logits;
    float* hidden;
    int* err;
    int H, I, V, L, nh, nkv, n_ctx, nqkv;
    float eps;
    int stages, rows_h, rows_i, act_floats, max_chunks, max_seqs, merge_group;
    unsigned long long* cnt;  // per-phase arrival counters, one line each
    long long* prof;   // nullable: [grid][prof_marks] timestamps
    int prof_marks;
    unsigned long long wait_ns;  // every bounded wait gives up after this many ns
    int test_stall;              // test hook: wait on a counter nothing arrives at
};

constexpr unsigned long long kPersistWaitNs = kWaitNs;  // a wait gives up after 2 s unless shortened

// Profiling slots per CTA: 0 launch start; per layer l, 1 + 16 l + k with
// k = 0 x gathered, 1 normed, 2 Q/K/V done, 3 q ready (attention CTAs),
// 4 attention done, 5 partials counted, 6 merge done, 7 o_proj done,
// 8 x1 counted, 9 x1 gathered, 10 gate/up done, 11 m counted,
// 12 m gathered, 13 down done (14 and 15 unused); then 1 + 16 L final x
// gathered, 2 + 16 L LM head done, 3 + 16 L argmax done.
inline int persistent_marks(int n_layer) { return 4 + 16 * n_layer; }

// Size the kernel for this context and allocate its packet buffers; leaves
// c.pers.ok false (and returns cudaSuccess) when the shape or device does
// not fit it.
cudaError_t persistent_setup(Ctx& c);
cudaError_t enqueue_decode_persistent(Ctx& c, bool want_logits, cudaStream_t st);
// Zero the packets, counters and epoch (after a launch gave up part-way).
cudaError_t persistent_reset(Ctx& c);

}  // namespace qwen2
