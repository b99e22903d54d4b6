// An LM head + greedy argmax that allocates no device memory and needs no
// context.
//
// Some callers own all of a GPU's memory through their own allocator (a
// serving engine that carves one pool at start-up, say): a library that
// calls cudaMalloc behind their back can fail or fragment that pool, and a
// context holds workspace they did not account for.  This entry point takes
// every buffer from the caller except its scratch -- each block's best
// (value, index) per row and the counter that elects the block doing the
// final merge -- which lives in one file-scope __device__ array that every
// GPU loading the library holds (about 32 KB) until the process exits.
//
// The computation is the tied LM head of the decode path applied to rows
// that are already normalised: logits[r][v] = E[v] . hidden[r], then the
// lowest index of each row's maximum.  It uses the same row dot product as
// the decode path's LM head, so its logits match those bit for bit.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <mutex>
#include <string>

#include "ctx.h"
#include "rowdot.cuh"

using namespace qwen2;

namespace {

constexpr int kNaMaxRows = 8;      // rows one call may carry
constexpr int kNaMaxHidden = 1024; // largest hidden size (activations sit in 32 KB of shared memory)
constexpr int kNaBlocks = 512;     // blocks of the head kernel
constexpr int kNaThreads = 256;
constexpr int kNaWarps = kNaThreads / 32;
constexpr int kNaMaxDevices = 64;

struct NaScratch {
    float val[kNaBlocks][kNaMaxRows];
    int idx[kNaBlocks][kNaMaxRows];
    int count;  // blocks finished; must be 0 when a launch starts
};

static __device__ __align__(256) NaScratch g_na_scratch;

// The scratch's device address per device, with the context it was looked
// up in: a context created later on the same device (a driver-API context
// made current by the caller, or the primary context re-created after a
// reset) holds its own instance of the module, so the address is looked up
// again whenever the current context is not the recorded one.
struct NaAddr {
    CUcontext ctx;
    NaScratch* addr;
};
std::mutex g_na_mutex;
NaAddr g_na_addr[kNaMaxDevices] = {};

// The driver's cuCtxGetCurrent, looked up once through the runtime (the
// library does not link libcuda).
PFN_cuCtxGetCurrent_v4000 ctx_get_current() {
    static PFN_cuCtxGetCurrent_v4000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        cudaGetLastError();
        return reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    }();
    return fn;
}

template <int NB>
__global__ void __launch_bounds__(kNaThreads) k_lm_head_noalloc(const __half* __restrict__ E,
                                                                const float* __restrict__ hidden, int B, int H,
                                                                int V, int span, float* logits, int* ids,
                                                                NaScratch* sc) {
    __shared__ __align__(16) float xs[NB * kNaMaxHidden];
    __shared__ float wv_s[kNaWarps][NB];
    __shared__ int wi_s[kNaWarps][NB];
    __shared__ int last_s;
    for (int b = 0; b < NB; ++b)
        for (int j = threadIdx.x; j < H; j += blockDim.x) xs[b * H + j] = b < B ? hidden[(size_t)b * H + j] : 0.f;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r_begin = blockIdx.x * span;
    const int r_end = min(V, r_begin + span);
    float best_v[NB];
    int best_i[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        best_v[b] = -INFINITY;
        best_i[b] = 0x7fffffff;
    }
    for (int r = r_begin + 2 * warp; r < r_end; r += 2 * kNaWarps) {
        const bool two = r + 1 < r_end;
        const __half* rows[2] = {E + (size_t)r * H, E + (size_t)(two ? r + 1 : r) * H};
        float acc[2][NB];
        warp_rows_dot<NB, 2>(rows, H, xs, H, acc);
        if (lane == 0) {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (b >= B) continue;
                if (logits) {
                    logits[(size_t)b * V + r] = acc[0][b];
                    if (two) logits[(size_t)b * V + r + 1] = acc[1][b];
                }
                argmax_merge(best_v[b], best_i[b], acc[0][b], r);
                if (two) argmax_merge(best_v[b], best_i[b], acc[1][b], r + 1);
            }
        }
    }
    if (lane == 0)
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            wv_s[warp][b] = best_v[b];
            wi_s[warp][b] = best_i[b];
        }
    __syncthreads();
    if (threadIdx.x < NB) {
        const int b = threadIdx.x;
        float v = wv_s[0][b];
        int i = wi_s[0][b];
        for (int w = 1; w < kNaWarps; ++w) argmax_merge(v, i, wv_s[w][b], wi_s[w][b]);
        sc->val[blockIdx.x][b] = v;
        sc->idx[blockIdx.x][b] = i;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last_s = (atomicAdd(&sc->count, 1) == (int)gridDim.x - 1);
    __syncthreads();
    if (!last_s) return;
    __threadfence();
    if (warp < B && warp < NB) {
        const int b = warp;
        float v = -INFINITY;
        int i = 0x7fffffff;
        for (int k = lane; k < (int)gridDim.x; k += 32) argmax_merge(v, i, __ldcg(&sc->val[k][b]), __ldcg(&sc->idx[k][b]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, v, o);
            const int oi = __shfl_xor_sync(0xffffffffu, i, o);
            argmax_merge(v, i, ov, oi);
        }
        if (lane == 0) ids[b] = i;
    }
    __syncthreads();
    if (threadIdx.x == 0) sc->count = 0;
}

template <int NB>
cudaError_t launch_na(const __half* E, const float* hidden, int B, int H, int V, float* logits, int* ids,
                      NaScratch* sc, cudaStream_t st) {
    int span = (V + kNaBlocks - 1) / kNaBlocks;
    span = (span + 1) & ~1;
    k_lm_head_noalloc<NB><<<kNaBlocks, kNaThreads, 0, st>>>(E, hidden, B, H, V, span, logits, ids, sc);
    return cudaGetLastError();
}

}  // namespace

extern "C" int qwen2_lm_head_argmax_noalloc(const uint16_t* embed, const float* hidden, int32_t n_rows,
                                            int32_t hidden_size, int32_t vocab, float* logits, int32_t* ids,
                                            void* stream) {
    if (!embed || !hidden || !ids) {
        set_thread_error("qwen2_lm_head_argmax_noalloc: embed, hidden and ids must not be NULL");
        return QWEN2_E_ARG;
    }
    if (n_rows < 1 || n_rows > kNaMaxRows) {
        set_thread_error("qwen2_lm_head_argmax_noalloc: n_rows " + std::to_string(n_rows) +
                         " outside [1, 8] (the static scratch holds 8 rows)");
        return QWEN2_E_ARG;
    }
    if (hidden_size < 8 || hidden_size > kNaMaxHidden || hidden_size % 8 || vocab < 1) {
        set_thread_error("qwen2_lm_head_argmax_noalloc: hidden_size must be a multiple of 8 in [8, 1024] "
                         "and vocab >= 1");
        return QWEN2_E_ARG;
    }
    if (reinterpret_cast<uintptr_t>(embed) & 15) {
        // Rows are streamed with 16-byte vector loads.
        set_thread_error("qwen2_lm_head_argmax_noalloc: embed must be 16-byte aligned");
        return QWEN2_E_ARG;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNaMaxDevices) {
        cudaGetLastError();
        set_thread_error("qwen2_lm_head_argmax_noalloc: no usable current CUDA device");
        return QWEN2_E_CUDA;
    }
    CUcontext ctx = nullptr;
    PFN_cuCtxGetCurrent_v4000 get_ctx = ctx_get_current();
    if (!get_ctx || get_ctx(&ctx) != CUDA_SUCCESS) {
        set_thread_error("qwen2_lm_head_argmax_noalloc: cannot query the current CUDA context");
        return QWEN2_E_CUDA;
    }
    NaScratch* sc;
    {
        // First call on this device (and context): look up the device
        // address of the static scratch with that device current.
        std::lock_guard<std::mutex> lock(g_na_mutex);
        if (!ctx || !g_na_addr[dev].addr || g_na_addr[dev].ctx != ctx) {
            void* p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_na_scratch);
            // With no context current before, the runtime has now made the
            // device's primary context current.
            if (e == cudaSuccess && !ctx && get_ctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;
            if (e != cudaSuccess || !p || !ctx) {
                cudaGetLastError();
                set_thread_error(std::string("qwen2_lm_head_argmax_noalloc: cudaGetSymbolAddress failed: ") +
                                 cudaGetErrorString(e));
                return QWEN2_E_CUDA;
            }
            g_na_addr[dev] = NaAddr{ctx, static_cast<NaScratch*>(p)};
        }
        sc = g_na_addr[dev].addr;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The arrival counter must start at zero (a launch that stopped part-way
    // could have left it set).
    cudaError_t e = cudaMemsetAsync(&sc->count, 0, sizeof(int), st);
    if (e == cudaSuccess) {
        const __half* E = reinterpret_cast<const __half*>(embed);
        if (n_rows <= 1) e = launch_na<1>(E, hidden, n_rows, hidden_size, vocab, logits, ids, sc, st);
        else if (n_rows <= 2) e = launch_na<2>(E, hidden, n_rows, hidden_size, vocab, logits, ids, sc, st);
        else if (n_rows <= 4) e = launch_na<4>(E, hidden, n_rows, hidden_size, vocab, logits, ids, sc, st);
        else e = launch_na<8>(E, hidden, n_rows, hidden_size, vocab, logits, ids, sc, st);
    }
    if (e != cudaSuccess) {
        set_thread_error(std::string("qwen2_lm_head_argmax_noalloc: launch failed: ") + cudaGetErrorString(e));
        return QWEN2_E_CUDA;
    }
    return QWEN2_OK;
}
