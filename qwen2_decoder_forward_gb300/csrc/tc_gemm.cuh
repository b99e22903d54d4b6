// Tensor-core GEMM for prefill: C[M][N] = A[M][K] . B[N][K]^T with f16 A and
// B and f32 accumulation in tensor memory (tcgen05), operand tiles brought
// in by TMA with the 128-byte swizzle, and a caller-supplied epilogue that
// receives each output row in chunks of 32 columns.
//
// One CTA per SM, persistent over output tiles of 128 x BN, 192 threads in
// three roles:
//   warp 0    one lane issues the TMA loads of A and B k-blocks (64 wide)
//             into a ring of shared-memory stages;
//   warp 1    allocates tensor memory (two accumulators of BN columns, so
//             the epilogue of one tile overlaps the main loop of the next)
//             and one lane issues the MMAs (128 x BN x 16 each);
//   warps 2-5 the epilogue: warp w reads accumulator lanes 32 (w % 4) ..
//             32 (w % 4) + 31, i.e. one output row per thread.
// Every wait is bounded by the global timer; a wait that runs out sets the
// guard word, and the kernel still drains its copies and frees its tensor
// memory before it returns.
#pragma once

#include "common.cuh"
#include "sm100.cuh"

namespace qwen2 {
namespace tcg {

constexpr int kBM = 128;          // rows of an output tile (TMEM lanes)
constexpr int kBK = 64;           // k-block: 64 f16 = one 128-byte swizzle row
constexpr int kThreads = 192;

// SPLIT: A is given as two f16 matrices, A = A_hi + A_lo (A_hi = f16(a),
// A_lo = f16(a - A_hi)), and every k-step issues one MMA for each part into
// the same accumulator: the product then carries the f32 activation to
// about 22 bits instead of f16's 11, at twice the tensor work.
template <int BN, bool SPLIT>
struct GemmCfg {
    static constexpr int kABytes = kBM * kBK * 2;
    static constexpr int kBOff = SPLIT ? 2 * kABytes : kABytes;
    static constexpr int kBBytes = BN * kBK * 2;
    static constexpr int kStageBytes = kBOff + kBBytes;
    // As many stages as 220 KB holds: a CTA's loads in flight are bounded by
    // the ring, and the long-k products (down: 76 k-blocks a tile) keep the
    // tensor pipe fed only with the deepest ring that fits.
    static constexpr int kStages = (220 * 1024) / kStageBytes;
    // Two accumulators of BN columns, each at a power-of-two column offset
    // (kAccCols apart); the allocation is a power of two as well.
    static constexpr uint32_t kAccCols = BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
    static constexpr uint32_t kTmemCols = 2 * kAccCols;
    static constexpr size_t kSmem = (size_t)kStages * kStageBytes + 1024 + 256;
    static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "UMMA N for M = 128, whole 32-column epilogue chunks");
    static_assert(kStages >= 2, "at least two stages");
};

template <int BN, bool SPLIT, class Epi>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
              const __grid_constant__ CUtensorMap tmB, int M, int N, int K, Epi epi, int* err) {
    using C = GemmCfg<BN, SPLIT>;
    using namespace sm100;
    extern __shared__ unsigned char smem_raw[];
    // Stage buffers start on a 1024-byte boundary (the swizzle atom).
    const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
    unsigned char* base = smem_raw + pad;
    uint64_t* full = reinterpret_cast<uint64_t*>(base + (size_t)C::kStages * C::kStageBytes);
    uint64_t* empty = full + C::kStages;
    uint64_t* tfull = empty + C::kStages;
    uint64_t* tempty = tfull + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_m = (M + kBM - 1) / kBM, n_n = (N + BN - 1) / BN;
    const int n_tiles = n_m * n_n, nk = K / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 4);
        }
        mbar_init_fence();
        tma_prefetch_desc(&tmA);
        if (SPLIT) tma_prefetch_desc(&tmA2);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;
    // Launched with programmatic stream serialisation: everything above
    // overlaps the previous kernel; operands and outputs only after it.
    pdl_launch_dependents();
    pdl_wait();

    if (warp == 0) {
        if (lane == 0) {
            int s = 0;
            unsigned ph = 0;
            long long issued = 0;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                const int m0 = (t % n_m) * kBM, n0 = (t / n_m) * BN;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, kWaitNs)) {
                        ok = false;
                        break;
                    }
                    unsigned char* sa = base + (size_t)s * C::kStageBytes;
                    mbar_expect_tx(&full[s], C::kStageBytes);
                    tma_load_2d(sa, &tmA, kb * kBK, m0, &full[s]);
                    if (SPLIT) tma_load_2d(sa + C::kABytes, &tmA2, kb * kBK, m0, &full[s]);
                    tma_load_2d(sa + C::kBOff, &tmB, kb * kBK, n0, &full[s]);
                    ++issued;
                    if (++s == C::kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // Wait for this thread's last loads to land (immediate when the
            // MMAs consumed them) so no copy is in flight at exit.
            for (long long j = issued - 1; j >= 0 && j >= issued - C::kStages; --j)
                if (!mbar_wait(&full[j % C::kStages], (unsigned)((j / C::kStages) & 1), kWaitNs))
                    ok = false;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(kBM, BN);
            int s = 0, acc = 0;
            unsigned ph = 0, aph = 0;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                if (!mbar_wait(&tempty[acc], aph ^ 1u, kWaitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)acc * C::kAccCols;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(&full[s], ph, kWaitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_addr(base + (size_t)s * C::kStageBytes);
                    const uint64_t ad = desc_sw128(sa), bd = desc_sw128(sa + C::kBOff);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {
                        mma_f16(d, ad + 2 * k, bd + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
                        if (SPLIT) mma_f16(d, desc_sw128(sa + C::kABytes) + 2 * k, bd + 2 * k, idesc, 1u);
                    }
                    mma_commit(&empty[s]);
                    if (++s == C::kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(&tfull[acc]);
                if (++acc == 2) {
                    acc = 0;
                    aph ^= 1u;
                }
            }
        }
    } else {
        const int q = warp & 3;
        int acc = 0;
        unsigned aph = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
            const int m0 = (t % n_m) * kBM, n0 = (t / n_m) * BN;
            // One lane waits; the warp follows its verdict, so the
            // warp-collective TMEM loads below never diverge.
            int got = 1;
            if (lane == 0) got = mbar_wait(&tfull[acc], aph, kWaitNs) ? 1 : 0;
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int row = m0 + 32 * q + lane;
            const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)acc * C::kAccCols;
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                float v[32];
                tmem_ld32(tbase + (uint32_t)c, v);
                if (row < M && n0 + c < N) epi.store(row, n0 + c, v);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            if (++acc == 2) {
                acc = 0;
                aph ^= 1u;
            }
        }
    }
    if (!ok) raise_guard(err, kGuardTimeout);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

}  // namespace tcg
}  // namespace qwen2
