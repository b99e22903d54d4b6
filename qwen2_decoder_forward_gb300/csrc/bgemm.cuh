// Batched decode product on Q8_0 weights with the warp-level tensor-core
// MMA (m16n8k16, f16 operands, f32 accumulation):
//   C[b][n] = sum_k x[b][k] * (d[n][k / 32] * q[n][k]),  b < B <= 32,
// with the dequantisation of minfer "Qwen2 / Qwen2.5 Architecture
// Support" section 6 (Q8_0: 32 int8 values and one f16 scale per block of
// 32 along k).  The int8 values are exact in f16; the activations enter as
// an f16 hi / lo pair (x = hi + lo, two MMAs), so each 32-block's partial
// product is the f32 dot of x with q to about 22 bits, and the block scale
// d is applied to it in f32: acc += d * partial.
//
// Inside each 32-block the MMA's k order is a fixed permutation of the
// stored order, chosen so that a thread's fragments of both operands are 8
// contiguous elements (8 bytes of q, 8 halves of x): thread (g, t) of a
// warp holds stored columns 8t .. 8t+7 of the block, which the MMA treats as
// k = {2t, 2t+1, 2t+8, 2t+9} of the first k-step and the same plus 16 of
// the second.  Both operands use the same map, so the sum is unchanged.
//
// A CTA of 8 warps owns kGroups x NTW x 8 consecutive weight rows (n);
// warp w takes n-tile group w % kGroups and every KS-th block of each
// staged k-chunk (KS warps share a group and add their partials in a fixed
// order at the end).  The activation rows are staged in shared memory, k
// chunk by k chunk, as f16 hi / lo.
#pragma once

#include "common.cuh"

namespace qwen2 {
namespace bg {

constexpr int kThreads = 256;
constexpr int kWarps = 8;
constexpr int kKc = 1024;   // activation columns staged per chunk
constexpr int kPad = 32;    // row padding in halves (64 bytes: conflict-free 16-byte fragment loads)

__host__ __device__ constexpr size_t smem_bytes(int mt) {
    return (size_t)2 * (mt * 16) * (kKc + kPad) * 2;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two int8 values (bytes picked by `sel` from w) as an exact f16 pair: the
// biased byte u = q + 128 becomes the f16 1024 + u (exponent 10, u in the
// mantissa), and 1152 is subtracted.
__device__ __forceinline__ uint32_t i8x2_to_h2(uint32_t w, uint32_t sel) {
    const uint32_t u = w ^ 0x80808080u;
    uint32_t h = __byte_perm(u, 0x64u, sel);
    const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&h), __float2half2_rn(1152.f));
    return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ void split_store(__half* hi, __half* lo, float4 v) {
    const __half2 h01 = __floats2half2_rn(v.x, v.y), h23 = __floats2half2_rn(v.z, v.w);
    const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
    *reinterpret_cast<__half2*>(hi) = h01;
    *reinterpret_cast<__half2*>(hi + 2) = h23;
    *reinterpret_cast<__half2*>(lo) = __floats2half2_rn(v.x - f01.x, v.y - f01.y);
    *reinterpret_cast<__half2*>(lo + 2) = __floats2half2_rn(v.z - f23.x, v.w - f23.y);
}

// Epi::pair(b, n, v0, v1): outputs (b, n) and (b, n + 1), n even.
template <int MT, int NTW, int KS, class Epi>
__global__ void __launch_bounds__(kThreads) k_bgemm_q8(const float* __restrict__ X, int B, int K,
                                                       const int8_t* __restrict__ Q, const __half* __restrict__ D,
                                                       int N, Epi epi) {
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int kRows = MT * 16;
    constexpr int kLd = kKc + kPad;
    constexpr int kGroups = kWarps / KS;
    static_assert(kWarps % KS == 0, "KS divides the warps");
    __half* ah = reinterpret_cast<__half*>(smem);
    __half* al = ah + kRows * kLd;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gi = lane >> 2, ti = lane & 3;
    const int grp = warp % kGroups, ks = warp / kGroups;
    const int n0 = blockIdx.x * (kGroups * NTW * 8) + grp * NTW * 8;
    const int kblocks = K / 32;

    float acc[MT][NTW][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int t = 0; t < NTW; ++t) acc[m][t][0] = acc[m][t][1] = acc[m][t][2] = acc[m][t][3] = 0.f;

    for (int kc0 = 0; kc0 < K; kc0 += kKc) {
        const int kc = min(kKc, K - kc0);
        __syncthreads();
        for (int e = tid; e < kRows * (kc / 4); e += kThreads) {
            const int r = e / (kc / 4), k4 = 4 * (e % (kc / 4));
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < B) v = *reinterpret_cast<const float4*>(X + (size_t)r * K + kc0 + k4);
            split_store(ah + r * kLd + k4, al + r * kLd + k4, v);
        }
        __syncthreads();
        const int nb = kc / 32;
        for (int kb = ks; kb < nb; kb += KS) {
            const int kg = kc0 + kb * 32;
            uint2 w[NTW];
            float d0[NTW], d1[NTW];
#pragma unroll
            for (int t = 0; t < NTW; ++t) {
                const int row = n0 + t * 8 + gi, rs = n0 + t * 8 + 2 * ti;
                w[t] = row < N ? __ldg(reinterpret_cast<const uint2*>(Q + (size_t)row * K + kg + 8 * ti))
                               : make_uint2(0u, 0u);
                d0[t] = rs < N ? __half2float(D[(size_t)rs * kblocks + kg / 32]) : 0.f;
                d1[t] = rs + 1 < N ? __half2float(D[(size_t)(rs + 1) * kblocks + kg / 32]) : 0.f;
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const __half* hr = ah + (m * 16 + gi) * kLd + kb * 32 + 8 * ti;
                const __half* lr = al + (m * 16 + gi) * kLd + kb * 32 + 8 * ti;
                const uint4 h0 = *reinterpret_cast<const uint4*>(hr);
                const uint4 h1 = *reinterpret_cast<const uint4*>(hr + 8 * kLd);
                const uint4 l0 = *reinterpret_cast<const uint4*>(lr);
                const uint4 l1 = *reinterpret_cast<const uint4*>(lr + 8 * kLd);
#pragma unroll
                for (int t = 0; t < NTW; ++t) {
                    const uint32_t b00 = i8x2_to_h2(w[t].x, 0x4140u), b01 = i8x2_to_h2(w[t].x, 0x4342u);
                    const uint32_t b10 = i8x2_to_h2(w[t].y, 0x4140u), b11 = i8x2_to_h2(w[t].y, 0x4342u);
                    float p[4] = {0.f, 0.f, 0.f, 0.f};
                    mma16816(p, h0.x, h1.x, h0.y, h1.y, b00, b01);
                    mma16816(p, l0.x, l1.x, l0.y, l1.y, b00, b01);
                    mma16816(p, h0.z, h1.z, h0.w, h1.w, b10, b11);
                    mma16816(p, l0.z, l1.z, l0.w, l1.w, b10, b11);
                    acc[m][t][0] = fmaf(d0[t], p[0], acc[m][t][0]);
                    acc[m][t][1] = fmaf(d1[t], p[1], acc[m][t][1]);
                    acc[m][t][2] = fmaf(d0[t], p[2], acc[m][t][2]);
                    acc[m][t][3] = fmaf(d1[t], p[3], acc[m][t][3]);
                }
            }
        }
    }
    if (KS > 1) {
        // Warps ks > 0 hand their partials to warp ks = 0 of the group,
        // which adds them in ks order.
        float* red = reinterpret_cast<float*>(smem);
        constexpr int kVals = MT * NTW * 4;
        __syncthreads();
        if (ks > 0) {
            float* dst = red + (((ks - 1) * kGroups + grp) * 32 + lane) * kVals;
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int t = 0; t < NTW; ++t)
#pragma unroll
                    for (int i = 0; i < 4; ++i) dst[(m * NTW + t) * 4 + i] = acc[m][t][i];
        }
        __syncthreads();
        if (ks == 0) {
            for (int s = 1; s < KS; ++s) {
                const float* src = red + (((s - 1) * kGroups + grp) * 32 + lane) * kVals;
#pragma unroll
                for (int m = 0; m < MT; ++m)
#pragma unroll
                    for (int t = 0; t < NTW; ++t)
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc[m][t][i] += src[(m * NTW + t) * 4 + i];
            }
        }
    }
    if (ks == 0) {
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int t = 0; t < NTW; ++t) {
                const int n = n0 + t * 8 + 2 * ti;
                const int b0 = m * 16 + gi, b1 = b0 + 8;
                if (n < N) {
                    if (b0 < B) epi.pair(b0, n, acc[m][t][0], acc[m][t][1]);
                    if (b1 < B) epi.pair(b1, n, acc[m][t][2], acc[m][t][3]);
                }
            }
    }
    epi.finish(ks == 0);
}

}  // namespace bg
}  // namespace qwen2
