// Device helpers shared by the kernels of libqwen2 (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace qwen2 {

// Guard codes a kernel writes into the context's error word (first one wins).
enum GuardCode : int {
    kGuardNone = 0,
    kGuardPosition = 1,     // a position outside [0, n_ctx) reached a kernel
    kGuardToken = 2,        // a token outside [0, V) reached a kernel
    kGuardShape = 3,        // a launch got a shape it was not built for
    kGuardTimeout = 4,      // a bounded spin-wait gave up
};

// Every spin-wait of every kernel gives up after this many ns of the global
// timer (2 s), raises kGuardTimeout and lets its kernel finish.
constexpr unsigned long long kWaitNs = 2000000000ull;

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

// Four-way split of a lane's partial dot product: products of elements
// (0,1), (2,3), (4,5), (6,7) of every 8-element chunk go to a[0..3], each
// in chunk order; dot4_total adds them as (a0 + a1) + (a2 + a3).  Four
// independent chains keep the FMA pipes busy with few warps.  Every f16
// GEMV kernel uses these, so all paths round alike.
struct Acc4 {
    float a[4];
};
__device__ __forceinline__ void dot8_f16_4(uint4 w, float4 xa, float4 xb, Acc4& acc) {
    float2 f;
    f = h2_to_f2(w.x); acc.a[0] = fmaf(f.x, xa.x, acc.a[0]); acc.a[0] = fmaf(f.y, xa.y, acc.a[0]);
    f = h2_to_f2(w.y); acc.a[1] = fmaf(f.x, xa.z, acc.a[1]); acc.a[1] = fmaf(f.y, xa.w, acc.a[1]);
    f = h2_to_f2(w.z); acc.a[2] = fmaf(f.x, xb.x, acc.a[2]); acc.a[2] = fmaf(f.y, xb.y, acc.a[2]);
    f = h2_to_f2(w.w); acc.a[3] = fmaf(f.x, xb.z, acc.a[3]); acc.a[3] = fmaf(f.y, xb.w, acc.a[3]);
}
__device__ __forceinline__ float dot4_total(const Acc4& acc) { return (acc.a[0] + acc.a[1]) + (acc.a[2] + acc.a[3]); }

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

// Greedy argmax merge.  Keeps the lowest index of the maximum.  NaN orders above every number
// (the first NaN of a row wins, as numpy's argmax has it), so a row whose
// logits are all NaN still yields an index inside the vocabulary.
__device__ __forceinline__ void argmax_merge(float& v, int& i, float ov, int oi) {
    const bool vn = v != v, on = ov != ov;
    const bool take = on ? (!vn || oi < i) : (!vn && (ov > v || (ov == v && oi < i)));
    if (take) { v = ov; i = oi; }
}

// Programmatic dependent launch (a kernel launched with the programmatic
// stream-serialisation attribute may start before the previous kernel of
// the stream ends): pdl_wait() blocks until the previous kernel has
// completed and its writes are visible -- every read of data that kernel
// produces, and every write to data it reads, comes after it.
// pdl_launch_dependents() lets the next kernel of the stream be scheduled
// once every CTA of this one has issued it (or exited).  Without the
// attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch with programmatic stream serialisation: the kernel may start
// while the previous kernel of the stream drains; it calls pdl_wait()
// before touching anything that kernel (or one before it) writes or reads.
template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// SiLU(z) = z / (1 + e^-z) (hidden_act "silu").
__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

}  // namespace qwen2
