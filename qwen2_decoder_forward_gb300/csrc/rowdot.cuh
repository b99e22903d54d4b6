// The canonical weight-row dot product every f16 GEMV kernel of libqwen2 uses.
//
// A row of K f16 weights is read as K/8 chunks of 16 bytes; lane l of the
// warp takes chunks l, l+32, l+64, ... in that order and adds each chunk's
// eight products into four partial sums by element pair (dot8_f16_4); the
// lane's total (a0 + a1) + (a2 + a3) is then summed over the 32 lanes by
// the xor butterfly of warp_sum (lane 0's value).  Because the lane
// assignment depends on the row alone, a row's result does not depend on
// which rows share the warp, on the number of activation vectors, on where
// the weights are read from, or on which kernel computes it: fused and
// unfused paths, per-step and persistent kernels, batch 1 and batch B, all
// round alike.
#pragma once

#include "common.cuh"

namespace qwen2 {

// Where a weight row is read from: global memory (streamed, read-only path)
// or shared memory (a stage the persistent kernel's producer filled).
struct LdGlobal {
    __device__ __forceinline__ static uint4 ld(const __half* p) { return ld_stream_v4(p); }
};
struct LdShared {
    __device__ __forceinline__ static uint4 ld(const __half* p) { return *reinterpret_cast<const uint4*>(p); }
};

// Dot products of R weight rows with NB activation vectors held in shared
// memory (xs + nb*ldx, 16-byte aligned, K floats each; xs must point into
// shared memory).  Loads of all R rows
// are issued together, U chunks per lane per row at a time.  acc[r][nb] is
// valid in lane 0.
template <int NB, int R, class Ld = LdGlobal, int U = 8>
__device__ __forceinline__ void warp_rows_dot(const __half* const (&rows)[R], int K,
                                              const float* xs, int ldx, float (&acc)[R][NB]) {
    const int lane = threadIdx.x & 31;
    const int kc = K >> 3;
    Acc4 part[R][NB];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int e = 0; e < 4; ++e) part[r][nb].a[e] = 0.f;
    for (int i0 = 0; i0 * 32 < kc; i0 += U) {
        uint4 wv[R][U];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = lane + 32 * (i0 + u);
                wv[r][u] = c < kc ? Ld::ld(rows[r] + (size_t)c * 8) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = lane + 32 * (i0 + u);
            if (c < kc) {
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
                    const float4 xa = *reinterpret_cast<const float4*>(xs + nb * ldx + c * 8);
                    const float4 xb = *reinterpret_cast<const float4*>(xs + nb * ldx + c * 8 + 4);
#pragma unroll
                    for (int r = 0; r < R; ++r) dot8_f16_4(wv[r][u], xa, xb, part[r][nb]);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) acc[r][nb] = warp_sum(dot4_total(part[r][nb]));
}

// RMSNorm of NB rows into shared memory: xs[b][j] = (x[b][j] * s_b) * w[j]
// with s_b = rms_scale(sum_j x[b][j]^2).  Rows b >= B are zero-filled.  The
// sum of squares is accumulated per thread in index order (stride 256 over
// a 256-thread group) and reduced by block_sum, so the statistic rounds
// alike in every kernel.  `x` may point to global or shared memory.
template <int NB, class S = SyncBlock>
__device__ __forceinline__ void norm_rows_to_smem(const float* __restrict__ x, int B, int H,
                                                  const float* __restrict__ w, float eps,
                                                  float* xs, int ldx, float* red) {
    const int tid = threadIdx.x;
#pragma unroll 1
    for (int b = 0; b < NB; ++b) {
        if (b >= B) {
            for (int j = tid; j < H; j += 256) xs[b * ldx + j] = 0.f;
            continue;
        }
        const float* xr = x + (size_t)b * H;
        float ss = 0.f;
        for (int j = tid; j < H; j += 256) {
            const float v = xr[j];
            ss = fmaf(v, v, ss);
        }
        const float s = rms_scale(block_sum<S>(ss, red), H, eps);
        for (int j = tid; j < H; j += 256) xs[b * ldx + j] = __fmul_rn(__fmul_rn(xr[j], s), w[j]);
    }
    S::sync();
}

// NeoX rotation of the pair (a, b) = (x_i, x_{i+hd/2}) by (cos, sin):
// a' = a cos - b sin, b' = b cos + a sin.
__device__ __forceinline__ void rope_pair(float a, float b, float2 cs, float& ra, float& rb) {
    ra = fmaf(a, cs.x, -__fmul_rn(b, cs.y));
    rb = fmaf(b, cs.x, __fmul_rn(a, cs.y));
}

}  // namespace qwen2
