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
// end).  The CTA's weight tile is staged in shared memory by bulk copies
// issued before anything else (k_bgemm_q8s); the LM head's persistent tile
// walker instead keeps about eight blocks per warp in flight in registers.  The
// chunk's activation rows reach shared memory through a prologue: either one
// bulk copy per row (hi and lo, issued by the 32 lanes of warp 0 on one
// mbarrier), or an RMSNorm of f32 rows computed in the CTA (one warp per
// row), which saves the separate normalisation kernel.
#pragma once

#include "common.cuh"
#include "sm100.cuh"

namespace qwen2 {
namespace bg {

constexpr int kThreads = 256;
constexpr int kWarps = 8;
constexpr int kKc = 1024;   // largest k chunk

// Shared-memory row stride (halves) of a k chunk of kc columns: kc rounded
// up to 64, plus 32, so consecutive rows sit 64 bytes apart modulo 128 and
// the 16-byte fragment loads of 8 rows x 4 lanes are conflict-free.
__host__ __device__ constexpr int row_ld(int kc) { return (kc + 63) / 64 * 64 + 32; }
__host__ __device__ constexpr size_t smem_bytes(int mt, int kc) {
    return (size_t)2 * (mt * 16) * row_ld(kc) * 2 + 16;
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

// Eight Q4_0 codes (a 32-bit word, element 2j in the low nibble of byte j)
// as four exact f16 pairs of (code - 8), in element order: the nibble u
// becomes the f16 1024 + u (exponent 10, u in the mantissa) and 1032 is
// subtracted.
__device__ __forceinline__ void q4x8_to_h2(uint32_t w, uint32_t (&h)[4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t b = (w >> (8 * j)) & 0xFFu;
        uint32_t v = (b & 0xFu) | ((b & 0xF0u) << 12) | 0x64006400u;
        const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&v), __float2half2_rn(1032.f));
        h[j] = *reinterpret_cast<const uint32_t*>(&r);
    }
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

__device__ __forceinline__ uint32_t ld_stream_u16(const void* p) {
    unsigned short v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float h_bits_to_f(uint32_t bits) {
    return __half2float(__ushort_as_half((unsigned short)bits));
}

// ---- prologues: the chunk's activation rows into shared memory -------------
// stage(ah, al, ld, rows, K, kc0, kc, bar, err): rows 0..rows-1 of columns
// [kc0, kc0 + kc) as f16 hi / lo, row stride ld halves.  Returns false if a
// bounded wait gave up.  Every thread of the CTA calls it.

// Rows already split into hi / lo in global memory: one bulk copy per row
// and half, issued by the lanes of warp 0.
struct ProCopy {
    const __half* hi;
    const __half* lo;
    __device__ __forceinline__ bool stage(__half* ah, __half* al, int ld, int rows, int K, int kc0, int kc,
                                          uint64_t* bar) const {
        using namespace sm100;
        const int tid = threadIdx.x;
        const unsigned row_bytes = (unsigned)kc * 2;
        if (tid == 0) mbar_expect_tx(bar, 2u * row_bytes * (unsigned)rows);
        __syncwarp();
        if (tid < rows) {
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_addr(ah + tid * ld)),
                "l"(hi + (size_t)tid * K + kc0), "r"(row_bytes), "r"(smem_addr(bar))
                : "memory");
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_addr(al + tid * ld)),
                "l"(lo + (size_t)tid * K + kc0), "r"(row_bytes), "r"(smem_addr(bar))
                : "memory");
        }
        return mbar_wait(bar, 0, kWaitNs);
    }
};

// RMSNorm of f32 rows x (nnterp encyclopedia "qwen2": x / sqrt(mean x^2 +
// eps) * w), computed here and split into hi / lo; the chunk must be the
// whole row (kc0 = 0, kc = K <= kKc, K a multiple of 4).  With W warps,
// warp w takes rows w and w + W (then w + 2W, w + 3W), a pair at a time
// with all of the pair's loads issued together: one round trip per pair
// (a single one for 32 rows and 16 warps); the norm weights are loaded
// once per warp.  If `out` is set, the normalised f32
// rows are also written there (by the CTA with blockIdx (0, 0)).
struct ProNorm {
    const float* x;
    const float* w;
    float eps;
    float* out;

    __device__ __forceinline__ static void emit(__half* ah, __half* al, float* out, int ld, int r, int K, int j,
                                                float4 v, float4 g, float sc, bool write_out) {
        const float n0 = __fmul_rn(__fmul_rn(v.x, sc), g.x), n1 = __fmul_rn(__fmul_rn(v.y, sc), g.y);
        const float n2 = __fmul_rn(__fmul_rn(v.z, sc), g.z), n3 = __fmul_rn(__fmul_rn(v.w, sc), g.w);
        if (write_out) *reinterpret_cast<float4*>(out + (size_t)r * K + j) = make_float4(n0, n1, n2, n3);
        __half h[4], l[4];
        split_h(n0, h[0], l[0]);
        split_h(n1, h[1], l[1]);
        split_h(n2, h[2], l[2]);
        split_h(n3, h[3], l[3]);
        *reinterpret_cast<uint2*>(ah + r * ld + j) = *reinterpret_cast<const uint2*>(h);
        *reinterpret_cast<uint2*>(al + r * ld + j) = *reinterpret_cast<const uint2*>(l);
    }

    __device__ __forceinline__ bool stage(__half* ah, __half* al, int ld, int rows, int K, int, int,
                                          uint64_t*) const {
        constexpr int kSteps = kKc / 128;
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
        const bool write_out = out && blockIdx.x == 0 && blockIdx.y == 0;
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        float4 g[kSteps];
#pragma unroll
        for (int i = 0; i < kSteps; ++i) {
            const int j = 4 * lane + 128 * i;
            g[i] = j < K ? *reinterpret_cast<const float4*>(w + j) : z;
        }
        for (int r0 = warp; r0 < rows; r0 += 2 * nw) {
            const int r1 = r0 + nw;
            const bool has1 = r1 < rows;
            float4 v0[kSteps], v1[kSteps];
#pragma unroll
            for (int i = 0; i < kSteps; ++i) {
                const int j = 4 * lane + 128 * i;
                v0[i] = j < K ? *reinterpret_cast<const float4*>(x + (size_t)r0 * K + j) : z;
                v1[i] = (j < K && has1) ? *reinterpret_cast<const float4*>(x + (size_t)r1 * K + j) : z;
            }
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int i = 0; i < kSteps; ++i) {
                s0 = fmaf(v0[i].x, v0[i].x, s0); s0 = fmaf(v0[i].y, v0[i].y, s0);
                s0 = fmaf(v0[i].z, v0[i].z, s0); s0 = fmaf(v0[i].w, v0[i].w, s0);
                s1 = fmaf(v1[i].x, v1[i].x, s1); s1 = fmaf(v1[i].y, v1[i].y, s1);
                s1 = fmaf(v1[i].z, v1[i].z, s1); s1 = fmaf(v1[i].w, v1[i].w, s1);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                s0 += __shfl_xor_sync(0xffffffffu, s0, o);
                s1 += __shfl_xor_sync(0xffffffffu, s1, o);
            }
            const float sc0 = 1.0f / sqrtf(s0 / (float)K + eps);
            const float sc1 = 1.0f / sqrtf(s1 / (float)K + eps);
#pragma unroll
            for (int i = 0; i < kSteps; ++i) {
                const int j = 4 * lane + 128 * i;
                if (j < K) {
                    emit(ah, al, out, ld, r0, K, j, v0[i], g[i], sc0, write_out);
                    if (has1) emit(ah, al, out, ld, r1, K, j, v1[i], g[i], sc1, write_out);
                }
            }
        }
        __syncthreads();
        return true;
    }
};

// Epi::start(n_cta0, rows_cta, B): all threads, before the main loop (the
// CTA's output rows are n_cta0 .. n_cta0 + rows_cta - 1).
// Epi::pair(b, n, v0, v1, chunk): outputs (b, n) and (b, n + 1), n even,
// partial over k chunk `chunk`.  Epi::finish(): once per CTA, all threads,
// after every pair of the CTA.
// W warps per CTA (32 W threads).  Grid (ceil(N / rows_cta), ceil(K /
// kc_len)), rows_cta = (W / KS) NTW 8; dynamic shared memory
// smem_bytes_s(MT, kc_len, rows_cta, q4); kc_len a multiple of 32, <= kKc.
// With KS > 1 the KS warps of a group exchange their partial tiles through
// shared memory and warp ks finishes the tiles j = m NTW + t with j % KS ==
// ks (sum over the KS partials in ks order, then the epilogue), so the
// epilogue work is spread over all warps.
//
// The product with the CTA's whole weight tile staged in shared memory.
// Before waiting for the previous kernel (pdl_wait), one warp issues a bulk
// copy of each of the CTA's weight rows (kc bytes of int8 at row stride
// kc + 32 bytes in shared memory: the 8-row x 32-byte fragment loads then
// fall on distinct banks) and every thread loads a share of the block
// scales: the weights never depend on an earlier kernel, so their whole
// stream is in flight while the previous kernel drains and while the
// activation rows are staged.
// Q4_0 tiles hold kc / 2 bytes a row at stride kc / 2 + 16 (the 8 rows x
// 4 lanes of a 32-bit fragment load then fall on 32 distinct banks).
__host__ __device__ constexpr int wrow_ld(int kc, bool q4 = false) { return q4 ? kc / 2 + 16 : kc + 32; }
__host__ __device__ constexpr size_t smem_bytes_s(int mt, int kc, int rows_cta, bool q4 = false) {
    return (size_t)2 * (mt * 16) * row_ld(kc) * 2 + (size_t)rows_cta * wrow_ld(kc, q4) +
           (size_t)rows_cta * (kc / 32) * 2 + 64;
}

template <int MT, int NTW, int KS, class Epi, class Pro, bool Q4 = false, int W = kWarps>
__global__ void __launch_bounds__(W * 32) k_bgemm_q8s(Pro pro, int B, int K, int kc_len,
                                                      const int8_t* __restrict__ Q, const __half* __restrict__ D,
                                                      int N, Epi epi, int* err) {
    using namespace sm100;
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int kRows = MT * 16;
    constexpr int kGroups = W / KS;
    constexpr int kRowsCta = kGroups * NTW * 8;
    static_assert(W % KS == 0, "KS divides the warps");
    const int ld = row_ld(kc_len), wld = wrow_ld(kc_len, Q4);
    constexpr int kEpb = Q4 ? 2 : 1;  // weights per byte
    __half* ah = reinterpret_cast<__half*>(smem);
    __half* al = ah + kRows * ld;
    int8_t* wq = reinterpret_cast<int8_t*>(al + kRows * ld);
    const int nbl = kc_len / 32;  // scale columns per weight row in shared memory
    uint16_t* wd = reinterpret_cast<uint16_t*>(wq + (size_t)kRowsCta * wld);
    uint64_t* bar = reinterpret_cast<uint64_t*>(
        (reinterpret_cast<uintptr_t>(wd + (size_t)kRowsCta * nbl) + 15) & ~uintptr_t(15));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gi = lane >> 2, ti = lane & 3;
    const int grp = warp % kGroups, ks = warp / kGroups;
    const int n_cta0 = blockIdx.x * kRowsCta;
    const int r0 = grp * NTW * 8;  // this warp's first row within the tile
    const int n0 = n_cta0 + r0;
    const int kc0 = blockIdx.y * kc_len;
    const int kc = min(kc_len, K - kc0);
    const int Bc = min(B, kRows);
    const int nb = kc / 32;
    const int rows = min(kRowsCta, N - n_cta0);

    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        mbar_init_fence();
    }
    __syncthreads();
    // The weight tile: one bulk copy per row (16-byte aligned: K, kc0 and kc
    // are multiples of 32), completion counted on bar[1].
    if (warp == 0) {
        if (lane == 0) mbar_expect_tx(&bar[1], (unsigned)(rows * (kc / kEpb)));
        __syncwarp();
        for (int r = lane; r < rows; r += 32)
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_addr(wq + (size_t)r * wld)),
                "l"(Q + (size_t)(n_cta0 + r) * (K / kEpb) + kc0 / kEpb), "r"((unsigned)(kc / kEpb)),
                "r"(smem_addr(&bar[1]))
                : "memory");
    }
    for (int e = tid; e < rows * nb; e += W * 32) {
        const int r = e / nb, b = e % nb;
        wd[r * nbl + b] = (uint16_t)ld_stream_u16(D + (size_t)(n_cta0 + r) * (K / 32) + kc0 / 32 + b);
    }
    pdl_launch_dependents();
    // An epilogue whose set-up reads only what stays fixed for the step
    // (positions, slots, biases, tables) does it while the previous kernel
    // drains.
    if (Epi::kStartBeforeWait) epi.start(n_cta0, kRowsCta, B);
    pdl_wait();
    if (!Epi::kStartBeforeWait) epi.start(n_cta0, kRowsCta, B);
    __syncthreads();
    const bool staged = pro.stage(ah, al, ld, Bc, K, kc0, kc, &bar[0]);
    const bool loaded = mbar_wait(&bar[1], 0, kWaitNs);
    if ((!staged || !loaded) && lane == 0) raise_guard(err, kGuardTimeout);
    __syncthreads();  // the scales

    float acc[MT][NTW][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int t = 0; t < NTW; ++t) acc[m][t][0] = acc[m][t][1] = acc[m][t][2] = acc[m][t][3] = 0.f;
    if (staged && loaded) {
        for (int kb = ks; kb < nb; kb += KS) {
            uint32_t bw[NTW][4];
            float dsc[NTW][2];
#pragma unroll
            for (int t = 0; t < NTW; ++t) {
                if (Q4) {
                    const uint32_t q = *reinterpret_cast<const uint32_t*>(wq + (size_t)(r0 + t * 8 + gi) * wld +
                                                                          kb * 16 + 4 * ti);
                    q4x8_to_h2(q, bw[t]);
                } else {
                    const uint2 q =
                        *reinterpret_cast<const uint2*>(wq + (size_t)(r0 + t * 8 + gi) * wld + kb * 32 + 8 * ti);
                    bw[t][0] = i8x2_to_h2(q.x, 0x4140u);
                    bw[t][1] = i8x2_to_h2(q.x, 0x4342u);
                    bw[t][2] = i8x2_to_h2(q.y, 0x4140u);
                    bw[t][3] = i8x2_to_h2(q.y, 0x4342u);
                }
                dsc[t][0] = h_bits_to_f(wd[(r0 + t * 8 + 2 * ti) * nbl + kb]);
                dsc[t][1] = h_bits_to_f(wd[(r0 + t * 8 + 2 * ti + 1) * nbl + kb]);
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const __half* hr = ah + (m * 16 + gi) * ld + kb * 32 + 8 * ti;
                const __half* lr = al + (m * 16 + gi) * ld + kb * 32 + 8 * ti;
                const uint4 h0 = *reinterpret_cast<const uint4*>(hr);
                const uint4 h1 = *reinterpret_cast<const uint4*>(hr + 8 * ld);
                const uint4 l0 = *reinterpret_cast<const uint4*>(lr);
                const uint4 l1 = *reinterpret_cast<const uint4*>(lr + 8 * ld);
#pragma unroll
                for (int t = 0; t < NTW; ++t) {
                    float p[4] = {0.f, 0.f, 0.f, 0.f};
                    mma16816(p, h0.x, h1.x, h0.y, h1.y, bw[t][0], bw[t][1]);
                    mma16816(p, l0.x, l1.x, l0.y, l1.y, bw[t][0], bw[t][1]);
                    mma16816(p, h0.z, h1.z, h0.w, h1.w, bw[t][2], bw[t][3]);
                    mma16816(p, l0.z, l1.z, l0.w, l1.w, bw[t][2], bw[t][3]);
                    acc[m][t][0] = fmaf(dsc[t][0], p[0], acc[m][t][0]);
                    acc[m][t][1] = fmaf(dsc[t][1], p[1], acc[m][t][1]);
                    acc[m][t][2] = fmaf(dsc[t][0], p[2], acc[m][t][2]);
                    acc[m][t][3] = fmaf(dsc[t][1], p[3], acc[m][t][3]);
                }
            }
        }
    }
    auto emit_tile = [&](int m, int t, const float (&v)[4]) {
        const int n = n0 + t * 8 + 2 * ti;
        const int b0 = m * 16 + gi, b1 = b0 + 8;
        if (n < N) {
            if (b0 < B) epi.pair(b0, n, v[0], v[1], blockIdx.y);
            if (b1 < B) epi.pair(b1, n, v[2], v[3], blockIdx.y);
        }
    };
    if (KS == 1) {
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int t = 0; t < NTW; ++t) emit_tile(m, t, acc[m][t]);
    } else {
        float4* red = reinterpret_cast<float4*>(smem);
        constexpr int kTiles = MT * NTW;
        __syncthreads();
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int t = 0; t < NTW; ++t)
                red[((ks * kGroups + grp) * kTiles + m * NTW + t) * 32 + lane] =
                    make_float4(acc[m][t][0], acc[m][t][1], acc[m][t][2], acc[m][t][3]);
        __syncthreads();
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int t = 0; t < NTW; ++t) {
                const int j = m * NTW + t;
                if (j % KS != ks) continue;
                float4 a = red[(grp * kTiles + j) * 32 + lane];
                for (int s = 1; s < KS; ++s) {
                    const float4 b = red[((s * kGroups + grp) * kTiles + j) * 32 + lane];
                    a.x += b.x;
                    a.y += b.y;
                    a.z += b.z;
                    a.w += b.w;
                }
                const float v[4] = {a.x, a.y, a.z, a.w};
                emit_tile(m, t, v);
            }
    }
    epi.finish();
}

// The same product for tall N (the LM head) with KS = 1: a persistent grid
// whose CTA stages the activation rows once and then walks row tiles
// blockIdx.x, blockIdx.x + gridDim.x, ...  Grid: up to the SM count (one
// CTA per SM); the k chunk is the whole row (kc_len = K, a multiple of
// 128).  With LO = false only the f16 hi part of the activations enters
// the MMAs (half the tensor work; the activation then carries 11 bits, as
// in an f16 GEMM).
//
// Each warp's weight stream is a sequence of groups of kWalkG consecutive
// 32-blocks of its NTW n-tiles, running straight on from one tile into the
// next, held in a ring of kWalkRing groups in registers: the ring slot a
// group was read from is refilled, block by block as its blocks are
// converted, with the group kWalkRing places ahead, so kWalkRing x kWalkG
// blocks per warp stay in flight.  The load and compute positions advance
// as (tile, group) counters, so the loop does no division, and a group's
// scales (kWalkG f16 values per output row) come in one 8-byte load per
// row.
constexpr int kWalkG = 4;     // 32-blocks per group
constexpr int kWalkRing = 1;  // groups in flight per warp

// One group of one lane: the q words of its row of each n-tile (Q8: 8
// bytes a block, Q4: 4 bytes) and the raw f16 scales of its two output
// rows, two per 32-bit word (converted at use, so the loads stay in flight).
template <int NTW, bool Q4>
struct WalkGroup {
    uint32_t q[NTW][kWalkG][Q4 ? 1 : 2];
    uint32_t d0[NTW][kWalkG / 2], d1[NTW][kWalkG / 2];
};

// Where the lane's loads of one group start: the first q byte of its row
// in n-tile 0 (tile t adds 8 t rows) and the first scale of its first
// output row; the rows past N load zeros.
struct WalkCursor {
    const int8_t* q;
    const __half* d;
    int row, rs;  // the lane's q row and first output row in n-tile 0
};

template <bool Q4>
__device__ __forceinline__ WalkCursor walk_cursor(const int8_t* __restrict__ Q, const __half* __restrict__ D, int K,
                                                  int n_w, int g, int gi, int ti) {
    const int nb = K / 32;
    const int kb0 = g * kWalkG;
    WalkCursor c;
    c.row = n_w + gi;
    c.rs = n_w + 2 * ti;
    c.q = Q4 ? Q + (size_t)c.row * (K / 2) + kb0 * 16 + 4 * ti : Q + (size_t)c.row * K + kb0 * 32 + 8 * ti;
    c.d = D + (size_t)c.rs * nb + kb0;
    return c;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// Block i of the group at cursor c into w.q[.][i].
template <int NTW, bool Q4>
__device__ __forceinline__ void walk_load_q(const WalkCursor& c, int K, int N, int i, WalkGroup<NTW, Q4>& w) {
    const size_t tstride = Q4 ? (size_t)8 * (K / 2) : (size_t)8 * K;
#pragma unroll
    for (int t = 0; t < NTW; ++t) {
        const int8_t* p = c.q + t * tstride + i * (Q4 ? 16 : 32);
        const bool ok = c.row + 8 * t < N;
        if (Q4) {
            w.q[t][i][0] = ok ? ld_stream_u32(p) : 0u;
        } else {
            const uint2 v = ok ? ld_stream_u2(p) : make_uint2(0u, 0u);
            w.q[t][i][0] = v.x;
            w.q[t][i][Q4 ? 0 : 1] = v.y;
        }
    }
}

// The group's scales at cursor c into w.d0 / w.d1 (8-byte loads: K / 32
// and the group's first block are multiples of 4).
template <int NTW, bool Q4>
__device__ __forceinline__ void walk_load_d(const WalkCursor& c, int K, int N, WalkGroup<NTW, Q4>& w) {
    const int nb = K / 32;
#pragma unroll
    for (int t = 0; t < NTW; ++t) {
        const __half* p = c.d + (size_t)8 * t * nb;
        const int rs = c.rs + 8 * t;
        const uint2 a = rs < N ? ld_stream_u2(p) : make_uint2(0u, 0u);
        const uint2 b = rs + 1 < N ? ld_stream_u2(p + nb) : make_uint2(0u, 0u);
        w.d0[t][0] = a.x;
        w.d0[t][1] = a.y;
        w.d1[t][0] = b.x;
        w.d1[t][1] = b.y;
    }
}

template <int MT, int NTW, class Epi, class Pro, bool LO = true, bool Q4 = false>
__global__ void __launch_bounds__(kThreads) k_bgemm_q8_tiles(Pro pro, int B, int K, const int8_t* __restrict__ Q,
                                                             const __half* __restrict__ D, int N, Epi epi, int* err) {
    using namespace sm100;
    static_assert(kWalkG == 4, "a group's scales are one 8-byte load per row");
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int kRows = MT * 16;
    constexpr int kRowsCta = kWarps * NTW * 8;
    const int ld = row_ld(K);
    __half* ah = reinterpret_cast<__half*>(smem);
    __half* al = ah + kRows * ld;
    uint64_t* bar = reinterpret_cast<uint64_t*>(al + kRows * ld);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gi = lane >> 2, ti = lane & 3;
    const int Bc = min(B, kRows);
    const int ng = K / (32 * kWalkG);  // groups per tile
    const int n_tiles = (N + kRowsCta - 1) / kRowsCta;
    const int wrow = warp * NTW * 8;   // the warp's first row within a tile

    // The first kRing groups go out before the wait: weights do not depend
    // on the previous kernel.
    WalkGroup<NTW, Q4> wg[kWalkRing];
    int l_tile = blockIdx.x, l_g = 0;  // the next group to load
#pragma unroll
    for (int r = 0; r < kWalkRing; ++r) {
        if (l_tile < n_tiles) {
            const WalkCursor c = walk_cursor<Q4>(Q, D, K, l_tile * kRowsCta + wrow, l_g, gi, ti);
#pragma unroll
            for (int i = 0; i < kWalkG; ++i) walk_load_q<NTW, Q4>(c, K, N, i, wg[r]);
            walk_load_d<NTW, Q4>(c, K, N, wg[r]);
        }
        if (++l_g == ng) {
            l_g = 0;
            l_tile += gridDim.x;
        }
    }
    pdl_launch_dependents();
    pdl_wait();  // the activation rows come from the previous kernel
    epi.start(0, 0, B);
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    const bool staged = pro.stage(ah, al, ld, Bc, K, 0, K, bar);
    if (!staged && lane == 0) raise_guard(err, kGuardTimeout);

    float acc[MT][NTW][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int t = 0; t < NTW; ++t) acc[m][t][0] = acc[m][t][1] = acc[m][t][2] = acc[m][t][3] = 0.f;
    if (staged) {
        int c_tile = blockIdx.x, c_g = 0;  // the group being multiplied
        while (c_tile < n_tiles) {
#pragma unroll
            for (int r = 0; r < kWalkRing; ++r) {
                if (c_tile < n_tiles) {
                    const bool refill = l_tile < n_tiles;
                    const WalkCursor lc = walk_cursor<Q4>(Q, D, K, l_tile * kRowsCta + wrow, l_g, gi, ti);
#pragma unroll
                    for (int i = 0; i < kWalkG; ++i) {
                        const int kb = c_g * kWalkG + i;
                        uint32_t bw[NTW][4];
                        float dsc[NTW][2];
#pragma unroll
                        for (int t = 0; t < NTW; ++t) {
                            if (Q4) {
                                q4x8_to_h2(wg[r].q[t][i][0], bw[t]);
                            } else {
                                bw[t][0] = i8x2_to_h2(wg[r].q[t][i][0], 0x4140u);
                                bw[t][1] = i8x2_to_h2(wg[r].q[t][i][0], 0x4342u);
                                bw[t][2] = i8x2_to_h2(wg[r].q[t][i][Q4 ? 0 : 1], 0x4140u);
                                bw[t][3] = i8x2_to_h2(wg[r].q[t][i][Q4 ? 0 : 1], 0x4342u);
                            }
                            const uint32_t w0 = wg[r].d0[t][i >> 1], w1 = wg[r].d1[t][i >> 1];
                            dsc[t][0] = h_bits_to_f((i & 1) ? (w0 >> 16) : (w0 & 0xffffu));
                            dsc[t][1] = h_bits_to_f((i & 1) ? (w1 >> 16) : (w1 & 0xffffu));
                        }
                        if (refill) {
                            walk_load_q<NTW, Q4>(lc, K, N, i, wg[r]);
                            if (i == kWalkG - 1) walk_load_d<NTW, Q4>(lc, K, N, wg[r]);
                        }
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            const __half* hr = ah + (m * 16 + gi) * ld + kb * 32 + 8 * ti;
                            const __half* lr = al + (m * 16 + gi) * ld + kb * 32 + 8 * ti;
                            const uint4 h0 = *reinterpret_cast<const uint4*>(hr);
                            const uint4 h1 = *reinterpret_cast<const uint4*>(hr + 8 * ld);
                            const uint4 l0 = LO ? *reinterpret_cast<const uint4*>(lr) : make_uint4(0u, 0u, 0u, 0u);
                            const uint4 l1 =
                                LO ? *reinterpret_cast<const uint4*>(lr + 8 * ld) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                            for (int t = 0; t < NTW; ++t) {
                                float p[4] = {0.f, 0.f, 0.f, 0.f};
                                mma16816(p, h0.x, h1.x, h0.y, h1.y, bw[t][0], bw[t][1]);
                                if (LO) mma16816(p, l0.x, l1.x, l0.y, l1.y, bw[t][0], bw[t][1]);
                                mma16816(p, h0.z, h1.z, h0.w, h1.w, bw[t][2], bw[t][3]);
                                if (LO) mma16816(p, l0.z, l1.z, l0.w, l1.w, bw[t][2], bw[t][3]);
                                acc[m][t][0] = fmaf(dsc[t][0], p[0], acc[m][t][0]);
                                acc[m][t][1] = fmaf(dsc[t][1], p[1], acc[m][t][1]);
                                acc[m][t][2] = fmaf(dsc[t][0], p[2], acc[m][t][2]);
                                acc[m][t][3] = fmaf(dsc[t][1], p[3], acc[m][t][3]);
                            }
                        }
                    }
                    if (++l_g == ng) {
                        l_g = 0;
                        l_tile += gridDim.x;
                    }
                    if (++c_g == ng) {
                        // The tile's last group: its outputs, then a fresh tile.
                        const int n0 = c_tile * kRowsCta + wrow;
#pragma unroll
                        for (int m = 0; m < MT; ++m)
#pragma unroll
                            for (int t = 0; t < NTW; ++t) {
                                const int n = n0 + t * 8 + 2 * ti;
                                const int b0 = m * 16 + gi, b1 = b0 + 8;
                                if (n < N) {
                                    if (b0 < B) epi.pair(b0, n, acc[m][t][0], acc[m][t][1], 0);
                                    if (b1 < B) epi.pair(b1, n, acc[m][t][2], acc[m][t][3], 0);
                                }
                                acc[m][t][0] = acc[m][t][1] = acc[m][t][2] = acc[m][t][3] = 0.f;
                            }
                        c_g = 0;
                        c_tile += gridDim.x;
                    }
                }
            }
        }
    }
    epi.finish();
}

}  // namespace bg
}  // namespace qwen2
