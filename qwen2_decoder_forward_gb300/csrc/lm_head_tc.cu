// Final RMSNorm + LM head + greedy argmax for the kept rows of the tensor-core
// prefill (minfer "Qwen2 / Qwen2.5 Architecture Support", section 1: the last
// norm, the readout by the tied embedding (or the untied head) and the
// greedy id of each row).
//
// logits[b][v] = E[v] . h_b for up to 8 rows h_b = RMSNorm(x_b), as a
// tcgen05 product: the vocabulary rows of E stream through a ring of
// shared-memory stages by TMA (128 rows x 64 k per stage, 128-byte
// swizzle) and form the MMA's M dimension; the normed rows, held in shared
// memory for the whole kernel as an f16 hi / lo pair (h = hi + lo), are its
// 16 N columns (0-7 hi, 8-15 lo), so one 128 x 16 x 16 MMA per k step
// covers both halves and logit = D[v][b] + D[v][8 + b] carries h to about
// 22 bits.  The kernel is bound by the stream of E (V x H f16).
//
// One CTA per SM, persistent over 128-row vocabulary tiles, 256 threads:
//   all       the RMSNorm prologue (block 0 also writes final_norm_output);
//   warp 0    one lane issues the TMA loads of E;
//   warp 1    allocates tensor memory (two accumulators) and one lane
//             issues the MMAs;
//   warps 4-7 read the accumulators (warp w: TMEM lanes 32 (w mod 4) ..
//             + 31, one vocabulary row per thread), write the logits and
//             keep each row b's best (value, lowest index).
// Per-CTA bests go to am_val / am_idx; the last CTA to finish merges them.
// Every wait is bounded by the global timer; a wait that runs out sets the
// guard word, and the kernel drains its copies and frees its tensor memory.
#include "common.cuh"
#include "prefill.h"
#include "rowdot.cuh"
#include "sm100.cuh"
#include "tmap.h"

namespace qwen2 {

namespace {

constexpr int kThreads = 256;
constexpr int kRowsMax = 8;            // hidden rows per launch
constexpr int kBM = 128;               // vocabulary rows per tile
constexpr int kBK = 64;                // k per stage (one 128-byte swizzle row)
constexpr int kN = 2 * kRowsMax;       // MMA N: hi and lo of each row
constexpr unsigned kStageBytes = kBM * kBK * 2;
constexpr uint32_t kAccCols = 64;      // accumulator column offsets 0 and 64
constexpr uint32_t kTmemCols = 2 * kAccCols;

struct LmTcArgs {
    const float* x;       // [B][H] rows before the final norm
    const float* norm_w;  // [H]
    float eps;
    int B, H, V, stages;
    float* logits;        // nullable [B][V]
    float* hidden;        // [B][H] final_norm_output
    int* ids;             // nullable [B]
    float* am_val;        // [gridDim][8]
    int* am_idx;
    int* count;
    int* err;
};

// Dynamic shared memory: stage ring, then the B operand (H / 64 k-blocks of
// 16 rows x 128 bytes); the prologue's f32 rows alias the ring.
__host__ __device__ constexpr size_t lm_tc_smem(int stages, int H) {
    return 1024 + (size_t)stages * kStageBytes + (size_t)(H / kBK) * kN * 128 + 256;
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint4 u;
    __half2 h;
    h = __floats2half2_rn(f[0], f[1]); u.x = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2half2_rn(f[2], f[3]); u.y = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2half2_rn(f[4], f[5]); u.z = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2half2_rn(f[6], f[7]); u.w = *reinterpret_cast<uint32_t*>(&h);
    return u;
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__global__ void __launch_bounds__(kThreads, 1) k_lm_head_tc(const __grid_constant__ CUtensorMap tmE, LmTcArgs a) {
    using namespace sm100;
    extern __shared__ unsigned char lm_smem_raw[];
    const uint32_t pad = (1024u - (smem_addr(lm_smem_raw) & 1023u)) & 1023u;
    unsigned char* base = lm_smem_raw + pad;
    unsigned char* ring = base;
    unsigned char* bop = base + (size_t)a.stages * kStageBytes;
    const int nkb = a.H / kBK;
    uint64_t* full = reinterpret_cast<uint64_t*>(bop + (size_t)nkb * kN * 128);
    uint64_t* empty = full + 8;
    uint64_t* tfull = empty + 8;
    uint64_t* tempty = tfull + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
    float* red = reinterpret_cast<float*>(tmem_slot + 4);   // 8 floats
    __shared__ float wv_s[4][kRowsMax];
    __shared__ int wi_s[4][kRowsMax];
    __shared__ int last_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_tiles = (a.V + kBM - 1) / kBM;

    if (tid == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(&tfull[k], 1);
            mbar_init(&tempty[k], 4);
        }
        mbar_init_fence();
        tma_prefetch_desc(&tmE);
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    // Launched with programmatic stream serialisation: the set-up above
    // overlaps the previous kernel; its rows are read only after it.
    pdl_launch_dependents();
    pdl_wait();

    // ---- prologue: normed rows -> f32 scratch (in the ring) -> B operand ----
    float* xs = reinterpret_cast<float*>(ring);
    norm_rows_to_smem<kRowsMax>(a.x, a.B, a.H, a.norm_w, a.eps, xs, a.H, red);
    if (blockIdx.x == 0)
        for (int b = 0; b < a.B; ++b)
            for (int j = tid; j < a.H; j += kThreads) a.hidden[(size_t)b * a.H + j] = xs[b * a.H + j];
    // Row b's hi goes to B row b, its lo to B row 8 + b; k-block kb of the
    // operand is 16 rows x 128 bytes at kb * 2048, chunk c of row r at
    // chunk c ^ (r mod 8) (the 128-byte swizzle).
    for (int e = tid; e < kRowsMax * (a.H / 8); e += kThreads) {
        const int b = e / (a.H / 8), c8 = e % (a.H / 8);
        const float4 x0 = *reinterpret_cast<const float4*>(xs + b * a.H + 8 * c8);
        const float4 x1 = *reinterpret_cast<const float4*>(xs + b * a.H + 8 * c8 + 4);
        const float f[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        const uint4 hi = pack8(f);
        const uint32_t hw[4] = {hi.x, hi.y, hi.z, hi.w};
        float lo[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 h2 = __half22float2(*reinterpret_cast<const __half2*>(&hw[q]));
            lo[2 * q] = f[2 * q] - h2.x;
            lo[2 * q + 1] = f[2 * q + 1] - h2.y;
        }
        const int kb = c8 >> 3, c = c8 & 7;
        unsigned char* blk = bop + (size_t)kb * kN * 128;
        *reinterpret_cast<uint4*>(blk + b * 128 + ((c ^ (b & 7)) << 4)) = hi;
        const int r = kRowsMax + b;
        *reinterpret_cast<uint4*>(blk + r * 128 + ((c ^ (r & 7)) << 4)) = pack8(lo);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();  // the f32 scratch is dead from here: the ring may fill
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;
    float best_v[kRowsMax];
    int best_i[kRowsMax];
#pragma unroll
    for (int b = 0; b < kRowsMax; ++b) {
        best_v[b] = -INFINITY;
        best_i[b] = 0x7fffffff;
    }

    if (warp == 0) {
        if (lane == 0) {
            int s = 0;
            unsigned ph = 0;
            long long issued = 0;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x)
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, kWaitNs)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&full[s], kStageBytes);
                    tma_load_2d(ring + (size_t)s * kStageBytes, &tmE, kb * kBK, t * kBM, &full[s]);
                    ++issued;
                    if (++s == a.stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            // Let the last copies land before the shared memory is released.
            for (long long j = issued - 1; j >= 0 && j >= issued - a.stages; --j)
                if (!mbar_wait(&full[j % a.stages], (unsigned)((j / a.stages) & 1), kWaitNs)) ok = false;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(kBM, kN);
            int s = 0, acc = 0;
            unsigned ph = 0, aph = 0;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                if (!mbar_wait(&tempty[acc], aph ^ 1u, kWaitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)acc * kAccCols;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&full[s], ph, kWaitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = desc_sw128(smem_addr(ring + (size_t)s * kStageBytes));
                    const uint64_t bd = desc_sw128(smem_addr(bop + (size_t)kb * kN * 128));
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) mma_f16(d, ad + 2 * k, bd + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
                    mma_commit(&empty[s]);
                    if (++s == a.stages) {
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
    } else if (warp >= 4) {
        const int q = warp & 3;
        int acc = 0;
        unsigned aph = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
            int got = 1;
            if (lane == 0) got = mbar_wait(&tfull[acc], aph, kWaitNs) ? 1 : 0;
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) {
                ok = false;
                break;
            }
            tc_fence_after();
            float v[16];
            tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)acc * kAccCols, v);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            const int row = t * kBM + 32 * q + lane;
            if (row < a.V) {
#pragma unroll
                for (int b = 0; b < kRowsMax; ++b) {
                    if (b >= a.B) break;
                    const float lg = v[b] + v[kRowsMax + b];
                    if (a.logits) a.logits[(size_t)b * a.V + row] = lg;
                    argmax_merge(best_v[b], best_i[b], lg, row);
                }
            }
            if (++acc == 2) {
                acc = 0;
                aph ^= 1u;
            }
        }
        // This warp's best per row, lowest index among equal values.
#pragma unroll
        for (int b = 0; b < kRowsMax; ++b) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, best_v[b], o);
                const int oi = __shfl_xor_sync(0xffffffffu, best_i[b], o);
                argmax_merge(best_v[b], best_i[b], ov, oi);
            }
            if (lane == 0) {
                wv_s[q][b] = best_v[b];
                wi_s[q][b] = best_i[b];
            }
        }
    }
    if (!ok) raise_guard(a.err, kGuardTimeout);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);

    // ---- this CTA's best per row; the last CTA merges every CTA's ----------
    if (tid < kRowsMax) {
        const int b = tid;
        float v = wv_s[0][b];
        int i = wi_s[0][b];
        for (int w = 1; w < 4; ++w) argmax_merge(v, i, wv_s[w][b], wi_s[w][b]);
        a.am_val[blockIdx.x * 8 + b] = v;
        a.am_idx[blockIdx.x * 8 + b] = i;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) last_s = (atomicAdd(a.count, 1) == (int)gridDim.x - 1);
    __syncthreads();
    if (!last_s) return;
    __threadfence();
    if (warp < a.B && warp < kRowsMax) {
        const int b = warp;
        float v = -INFINITY;
        int i = 0x7fffffff;
        for (int k = lane; k < (int)gridDim.x; k += 32)
            argmax_merge(v, i, __ldcg(a.am_val + k * 8 + b), __ldcg(a.am_idx + k * 8 + b));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, v, o);
            const int oi = __shfl_xor_sync(0xffffffffu, i, o);
            argmax_merge(v, i, ov, oi);
        }
        if (lane == 0) {
            if (i < 0 || i >= a.V) {
                raise_guard(a.err, kGuardShape);
                i = 0;
            }
            if (a.ids) a.ids[b] = i;
        }
    }
    __syncthreads();
    if (tid == 0) *a.count = 0;
}

int lm_stages(int H) {
    const size_t budget = 200 * 1024;
    int s = 8;
    while (s > 2 && lm_tc_smem(s, H) > budget) --s;
    return s;
}

}  // namespace

bool lm_head_tc_supported(const Ctx& c) {
    const int H = c.cfg.hidden;
    return c.tc.lm_ok && H % kBK == 0 && (size_t)kRowsMax * H * 4 <= (size_t)lm_stages(H) * kStageBytes &&
           lm_tc_smem(lm_stages(H), H) <= 227 * 1024;
}

cudaError_t lm_head_tc_setup(Ctx& c) {
    const int H = c.cfg.hidden;
    if (H % kBK != 0) return cudaSuccess;  // not supported: the CUDA-core head serves
    c.tc.lm_ok = encode_kmajor_f16(&c.tc.lm_e, c.lm_head.w, (uint64_t)c.cfg.vocab, (uint64_t)H, kBM);
    if (!c.tc.lm_ok) return cudaSuccess;
    return cudaFuncSetAttribute(k_lm_head_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)lm_tc_smem(lm_stages(H), H));
}

cudaError_t enqueue_lm_head_tc(Ctx& c, const float* xin, int B, float* logits, int* ids, cudaStream_t st) {
    const int H = c.cfg.hidden, V = c.cfg.vocab;
    const int n_tiles = (V + kBM - 1) / kBM;
    const int grid = n_tiles < c.n_sm ? n_tiles : c.n_sm;
    if (grid > c.ws.am_blocks) return cudaErrorInvalidValue;
    const int stages = lm_stages(H);
    for (int b0 = 0; b0 < B; b0 += kRowsMax) {
        LmTcArgs a{};
        a.x = xin + (size_t)b0 * H;
        a.norm_w = c.final_norm;
        a.eps = c.cfg.rms_eps;
        a.B = B - b0 < kRowsMax ? B - b0 : kRowsMax;
        a.H = H;
        a.V = V;
        a.stages = stages;
        a.logits = logits ? logits + (size_t)b0 * V : nullptr;
        a.hidden = c.ws.hidden + (size_t)b0 * H;
        a.ids = ids ? ids + b0 : nullptr;
        a.am_val = c.ws.am_val;
        a.am_idx = c.ws.am_idx;
        a.count = c.ws.am_count;
        a.err = c.err;
        cudaError_t e = launch_pdl(k_lm_head_tc, dim3(grid), dim3(kThreads), lm_tc_smem(stages, H), st, c.tc.lm_e, a);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace qwen2
