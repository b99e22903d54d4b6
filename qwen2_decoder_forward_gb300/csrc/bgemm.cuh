// Batched decode product on Q8_0 weights with the warp-level tensor-core
// MMA (m16n8k16, f16 operands, f32 accumulation):
//   C[b][n] = sum_k x[b][k] * (d[n][k / 32] * q[n][k]),  b < B <= 32,
// with the dequantisation of minfer "Qwen2 / Qwen2.5 Architecture
// Support" section 6 (Q8_0: 32 int8 values and one f16 scale per block of
// 32 along k).  The int8 values are exact in f16; the activations come as
// an f16 hi / lo pair (x = hi + lo, two MMAs, written so by the kernel that
// produces them), so each 32-block's partial product is the f32 dot of x
// with q to about 22 bits, and the block scale d is applied to it in f32:
// acc += d * partial.
//
// Inside each 32-block the MMA's k order is a fixed permutation of the
// stored order, chosen so that a thread's fragments of both operands are 8
// contiguous elements (8 bytes of q, 8 halves of x): thread (g, t) of a
// warp holds stored columns 8t .. 8t+7 of the block, which the MMA treats as
// k = {2t, 2t+1, 2t+8, 2t+9} of the first k-step and the same plus 16 of
// the second.  Both operands use the same map, so the sum is unchanged.
//
// Grid: x over groups of weight rows, y over k chunks of kc columns (a
// split of k whose partial sums the epilogue receives with the chunk
// index).  A CTA of 8 warps owns kGroups x NTW x 8 consecutive weight rows;
// warp w takes n-tile group w % kGroups and every KS-th 32-block of the
// chunk (the KS warps of a group add their partials in a fixed order at the
// end).  The chunk's activation rows are brought into shared memory with
// one bulk copy per row (hi and lo) on an mbarrier; weights stream from
// global memory one block ahead of the MMAs.
#pragma once

#include "common.cuh"
#include "sm100.cuh"

namespace qwen2 {
namespace bg {

constexpr int kThreads = 256;
constexpr int kWarps = 8;
constexpr int kKc = 1024;   // largest k chunk
constexpr int kPad = 32;    // row padding in halves (64 bytes: conflict-free 16-byte fragment loads)
constexpr unsigned long long kWaitNs = 2000000000ull;

__host__ __device__ constexpr size_t smem_bytes(int mt) {
    return (size_t)2 * (mt * 16) * (kKc + kPad) * 2 + 16;
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

__device__ __forceinline__ uint2 ld_stream_u2(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// v as an f16 hi / lo pair (hi = f16(v), lo = f16(v - hi)).
__device__ __forceinline__ void split_h(float v, __half& hi, __half& lo) {
    hi = __float2half_rn(v);
    lo = __float2half_rn(v - __half2float(hi));
}

struct WeightBlock {
    uint2 q;
    float d0, d1;
};

template <int NTW>
__device__ __forceinline__ void load_block(const int8_t* __restrict__ Q, const __half* __restrict__ D, int N, int K,
                                           int n0, int gi, int ti, int kg, WeightBlock (&w)[NTW]) {
#pragma unroll
    for (int t = 0; t < NTW; ++t) {
        const int row = n0 + t * 8 + gi, rs = n0 + t * 8 + 2 * ti;
        w[t].q = row < N ? ld_stream_u2(Q + (size_t)row * K + kg + 8 * ti) : make_uint2(0u, 0u);
        w[t].d0 = rs < N ? __half2float(D[(size_t)rs * (K / 32) + kg / 32]) : 0.f;
        w[t].d1 = rs + 1 < N ? __half2float(D[(size_t)(rs + 1) * (K / 32) + kg / 32]) : 0.f;
    }
}

// Epi::pair(b, n, v0, v1, chunk): outputs (b, n) and (b, n + 1), n even,
// partial over k chunk `chunk`.  Epi::finish(err): once per CTA, all threads.
template <int MT, int NTW, int KS, class Epi>
__global__ void __launch_bounds__(kThreads) k_bgemm_q8(const __half* __restrict__ Ah, const __half* __restrict__ Al,
                                                       int B, int K, int kc_len, const int8_t* __restrict__ Q,
                                                       const __half* __restrict__ D, int N, Epi epi, int* err) {
    using namespace sm100;
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int kRows = MT * 16;
    constexpr int kLd = kKc + kPad;
    constexpr int kGroups = kWarps / KS;
    static_assert(kWarps % KS == 0, "KS divides the warps");
    __half* ah = reinterpret_cast<__half*>(smem);
    __half* al = ah + kRows * kLd;
    uint64_t* bar = reinterpret_cast<uint64_t*>(al + kRows * kLd);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gi = lane >> 2, ti = lane & 3;
    const int grp = warp % kGroups, ks = warp / kGroups;
    const int n0 = blockIdx.x * (kGroups * NTW * 8) + grp * NTW * 8;
    const int kc0 = blockIdx.y * kc_len;
    const int kc = min(kc_len, K - kc0);
    const int Bc = min(B, kRows);

    // Stage rows 0..Bc-1 of the chunk (hi and lo); rows past B are never
    // read for a kept output (each MMA row is its own output row).
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (tid == 0) {
        const unsigned row_bytes = (unsigned)kc * 2;
        mbar_expect_tx(bar, 2u * row_bytes * (unsigned)Bc);
        for (int r = 0; r < Bc; ++r) {
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_addr(ah + r * kLd)),
                "l"(Ah + (size_t)r * K + kc0), "r"(row_bytes), "r"(smem_addr(bar))
                : "memory");
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_addr(al + r * kLd)),
                "l"(Al + (size_t)r * K + kc0), "r"(row_bytes), "r"(smem_addr(bar))
                : "memory");
        }
    }
    float acc[MT][NTW][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int t = 0; t < NTW; ++t) acc[m][t][0] = acc[m][t][1] = acc[m][t][2] = acc[m][t][3] = 0.f;
    const int nb = kc / 32;
    WeightBlock wc[NTW];
    if (ks < nb) load_block<NTW>(Q, D, N, K, n0, gi, ti, kc0 + ks * 32, wc);
    const bool staged = mbar_wait(bar, 0, global_ns() + kWaitNs);
    if (!staged && lane == 0) raise_guard(err, kGuardTimeout);
    if (staged) {
        for (int kb = ks; kb < nb; kb += KS) {
            WeightBlock wn[NTW];
            if (kb + KS < nb) load_block<NTW>(Q, D, N, K, n0, gi, ti, kc0 + (kb + KS) * 32, wn);
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
                    const uint32_t b00 = i8x2_to_h2(wc[t].q.x, 0x4140u), b01 = i8x2_to_h2(wc[t].q.x, 0x4342u);
                    const uint32_t b10 = i8x2_to_h2(wc[t].q.y, 0x4140u), b11 = i8x2_to_h2(wc[t].q.y, 0x4342u);
                    float p[4] = {0.f, 0.f, 0.f, 0.f};
                    mma16816(p, h0.x, h1.x, h0.y, h1.y, b00, b01);
                    mma16816(p, l0.x, l1.x, l0.y, l1.y, b00, b01);
                    mma16816(p, h0.z, h1.z, h0.w, h1.w, b10, b11);
                    mma16816(p, l0.z, l1.z, l0.w, l1.w, b10, b11);
                    acc[m][t][0] = fmaf(wc[t].d0, p[0], acc[m][t][0]);
                    acc[m][t][1] = fmaf(wc[t].d1, p[1], acc[m][t][1]);
                    acc[m][t][2] = fmaf(wc[t].d0, p[2], acc[m][t][2]);
                    acc[m][t][3] = fmaf(wc[t].d1, p[3], acc[m][t][3]);
                }
            }
#pragma unroll
            for (int t = 0; t < NTW; ++t) wc[t] = wn[t];
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
                    if (b0 < B) epi.pair(b0, n, acc[m][t][0], acc[m][t][1], blockIdx.y);
                    if (b1 < B) epi.pair(b1, n, acc[m][t][2], acc[m][t][3], blockIdx.y);
                }
            }
    }
    epi.finish();
}

}  // namespace bg
}  // namespace qwen2
