// The persistent single-launch batch-1 decode kernel (persistent.cu).
#pragma once

#include "ctx.h"

namespace qwen2 {

constexpr int kPersistStage = 32768;  // bytes per shared-memory ring stage
constexpr int kPersistStages = 5;     // ring depth (160 KB)

struct PersistentArgs {
    const PersistLayer* layers;
    const __half* E;
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
    long long* prof;   // nullable: [grid][prof_marks] timestamps
    int prof_marks;
};

inline int persistent_marks(int n_layer) { return 1 + 6 * n_layer + 2; }

// Size the kernel for this context and allocate its packet buffers; leaves
// c.pers.ok false (and returns cudaSuccess) when the shape or device does
// not fit it.
cudaError_t persistent_setup(Ctx& c);
cudaError_t enqueue_decode_persistent(Ctx& c, bool want_logits, cudaStream_t st);

}  // namespace qwen2
