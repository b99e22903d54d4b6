// Device helpers shared by the kernels of libqwen2 (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qwen2 {

// Guard codes a kernel writes into the context's error word (first one wins).
enum GuardCode : int {
    kGuardNone = 0,
    kGuardPosition = 1,     // a position outside [0, n_ctx) reached a kernel
    kGuardToken = 2,        // a token outside [0, V) reached a kernel
    kGuardShape = 3,        // a launch got a shape it was not built for
    kGuardTimeout = 4,      // a bounded spin-wait gave up
};

__device__ __forceinline__ void raise_guard(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// 16-byte streaming load of data that no kernel writes during the launch
// (weights): read-only path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float2 h2_to_f2(uint32_t v) {
    __half2 h = *reinterpret_cast<__half2*>(&v);
    return __half22float2(h);
}

// acc += sum_{e<8} w[e] * x[e], with w eight f16 values packed in a uint4 and
// x eight f32 values in shared or global memory (16-byte aligned).  The
// products are added in element order; every kernel that dots a weight row
// uses this one routine so that fused and unfused paths round alike.
__device__ __forceinline__ float dot8_f16(uint4 w, const float* x, float acc) {
    const float4 xa = *reinterpret_cast<const float4*>(x);
    const float4 xb = *reinterpret_cast<const float4*>(x + 4);
    float2 f;
    f = h2_to_f2(w.x); acc = fmaf(f.x, xa.x, acc); acc = fmaf(f.y, xa.y, acc);
    f = h2_to_f2(w.y); acc = fmaf(f.x, xa.z, acc); acc = fmaf(f.y, xa.w, acc);
    f = h2_to_f2(w.z); acc = fmaf(f.x, xb.x, acc); acc = fmaf(f.y, xb.y, acc);
    f = h2_to_f2(w.w); acc = fmaf(f.x, xb.z, acc); acc = fmaf(f.y, xb.w, acc);
    return acc;
}

// The same sum as dot8_f16 with the eight activations already in registers
// (xa = x[0..3], xb = x[4..7]), for kernels that share one load of x
// between several weight rows.
__device__ __forceinline__ float dot8_f16_r(uint4 w, float4 xa, float4 xb, float acc) {
    float2 f;
    f = h2_to_f2(w.x); acc = fmaf(f.x, xa.x, acc); acc = fmaf(f.y, xa.y, acc);
    f = h2_to_f2(w.y); acc = fmaf(f.x, xa.z, acc); acc = fmaf(f.y, xa.w, acc);
    f = h2_to_f2(w.z); acc = fmaf(f.x, xb.x, acc); acc = fmaf(f.y, xb.y, acc);
    f = h2_to_f2(w.w); acc = fmaf(f.x, xb.z, acc); acc = fmaf(f.y, xb.w, acc);
    return acc;
}

// Sum over the 32 lanes by a fixed xor butterfly; lane 0's value is the one
// every kernel uses.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Thread-group barriers.  Kernels whose 256 threads are the whole block use
// SyncBlock; the persistent decode kernel's 256 compute threads (warps 0-7,
// beside a producer warp) use named barrier 1.
struct SyncBlock {
    __device__ __forceinline__ static void sync() { __syncthreads(); }
};
struct SyncCompute {
    __device__ __forceinline__ static void sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
};

// Sum over a 256-thread group with a fixed reduction order; `red` is shared
// scratch of at least 8 floats.  Every thread of the group gets the result.
template <class S = SyncBlock>
__device__ __forceinline__ float block_sum(float v, float* red) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    v = warp_sum(v);
    S::sync();
    if (lane == 0) red[wid] = v;
    S::sync();
    float t = 0.f;
    if (wid == 0) {
        t = lane < 8 ? red[lane] : 0.f;
        t = warp_sum(t);
        if (lane == 0) red[0] = t;
    }
    S::sync();
    t = red[0];
    S::sync();
    return t;
}

// RMSNorm statistic: 1 / sqrt(mean(x^2) + eps), from a sum of squares.
__device__ __forceinline__ float rms_scale(float sumsq, int n, float eps) {
    return 1.0f / sqrtf(sumsq / (float)n + eps);
}

// Greedy argmax merge: larger value wins, equal values keep the lower index.
__device__ __forceinline__ void argmax_merge(float& v, int& i, float ov, int oi) {
    if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
}

// SiLU(z) = z / (1 + e^-z) (hidden_act "silu").
__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

}  // namespace qwen2
