// Causal GQA attention for the tensor-core prefill (QWEN2_PREFILL_TENSOR) on
// the warp-level tensor-core MMA (m16n8k16, f16 operands, f32 accumulation),
// flash-style: scores, online softmax and the value product stay in
// registers (nnterp encyclopedia qwen2, "Grouped-query attention": kv head g
// serves query heads g*group .. g*group + group - 1; scores q . k / sqrt(64)
// over keys 0..p).
//
// Block (g, blk) takes up to 16 rows of one sequence; warp h < group owns
// query head g*group + h for those rows.  Keys come from the f32 KV cache in
// tiles of 64 positions, converted once into shared memory and shared by
// the whole group.  Precision: q, k and the probabilities enter the MMAs as
// f16; v enters as an f16 hi / lo pair (two MMAs), because its rounding is
// what the output is most sensitive to; the softmax statistics are f32 and
// the output is written as an f16 hi / lo pair (the o_proj operand).
#include "prefill.h"

namespace qwen2 {

namespace {

constexpr int kT = 256;
constexpr int kD = 64;          // head_dim
constexpr int kKT = 64;         // keys per tile
constexpr int kLd = kD + 8;     // padded shared row (halves): conflict-free ldmatrix
constexpr float kScaleLog2 = 0.125f * 1.4426950408889634f;  // 1/sqrt(64) * log2(e)

struct AttnTcSmem {
    float stage[2][2][kKT][kD];   // f32 K and V tiles in flight (double-buffered, cp.async)
    __half k[kKT][kLd];
    __half vh[kKT][kLd];
    __half vl[kKT][kLd];
    __half q[8][16][kLd];
};

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"((uint32_t)__cvta_generic_to_shared(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"((uint32_t)__cvta_generic_to_shared(p)));
}
// d += a . b for one 16 x 8 x 16 tile.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
    // 16 bytes from global to shared memory; zeros when !valid.
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}

__global__ void __launch_bounds__(kT, 2) k_attn_prefill_mma(PrefillAttnArgs a, int layer) {
    extern __shared__ __align__(16) unsigned char pa_smem[];
    AttnTcSmem& sm = *reinterpret_cast<AttnTcSmem*>(pa_smem);
    const int g = blockIdx.x, blk = blockIdx.y;
    const int r0 = a.blk_row0[blk], nr = a.blk_nrows[blk];
    const int group = a.nh / a.nkv;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gi = lane >> 2, ti = lane & 3;  // MMA fragment row group, thread in group
    const int slot = a.slot[r0];
    // Largest position of the block's rows (one load per lane, then a warp
    // max: no chain of dependent loads).
    int pmax = lane < nr ? a.pos[r0 + lane] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pmax = max(pmax, __shfl_xor_sync(0xffffffffu, pmax, o));
    const bool compute = warp < group;
    const int hq = g * group + warp;

    // This warp's 16 query rows as f16 (rows past nr are zero); lane l
    // takes dims 2l, 2l + 1 of every row, all 16 loads issued together.
    static_assert(kD == 64, "one float2 per lane per row");
    if (compute) {
        float2 qv[16];
#pragma unroll
        for (int r = 0; r < 16; ++r)
            qv[r] = r < nr ? *reinterpret_cast<const float2*>(a.q + (size_t)(r0 + r) * a.nh * kD + (size_t)hq * kD +
                                                               2 * lane)
                           : make_float2(0.f, 0.f);
#pragma unroll
        for (int r = 0; r < 16; ++r)
            *reinterpret_cast<__half2*>(&sm.q[warp][r][2 * lane]) = __floats2half2_rn(qv[r].x, qv[r].y);
    }
    const int pa = gi < nr ? a.pos[r0 + gi] : -1;          // positions of this thread's rows
    const int pb = gi + 8 < nr ? a.pos[r0 + gi + 8] : -1;
    float o[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
    uint32_t qf[4][4];

    const size_t head_stride = (size_t)a.n_ctx * kD;
    const size_t cache0 = ((size_t)slot * a.L + layer) * 2 * a.nkv;
    const float* kbase = a.kv + (cache0 + g) * head_stride;
    const float* vbase = a.kv + (cache0 + a.nkv + g) * head_stride;

    // Each tile's f32 K and V rows travel with cp.async into one of two
    // staging buffers, one tile ahead of the products; each thread then
    // converts its four (key, 4-dim) pieces of the current tile.
    constexpr int kPieces = kKT * (kD / 4) / kT;
    auto issue_tile = [&](int j0, int buf) {
        const int nj = min(kKT, pmax + 1 - j0);
#pragma unroll
        for (int i = 0; i < kPieces; ++i) {
            const int e = tid + kT * i, j = e / (kD / 4), d = 4 * (e % (kD / 4));
            const bool in = j < nj;
            const size_t off = (size_t)(in ? j0 + j : 0) * kD + d;
            cp_async16(&sm.stage[buf][0][j][d], kbase + off, in);
            cp_async16(&sm.stage[buf][1][j][d], vbase + off, in);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    issue_tile(0, 0);
    for (int j0 = 0, buf = 0; j0 <= pmax; j0 += kKT, buf ^= 1) {
        if (j0 + kKT <= pmax) {
            issue_tile(j0 + kKT, buf ^ 1);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();
        // Stage keys j0 .. j0 + 63 (zeros past the last): k and v rounded to
        // f16, v's remainder as a second f16.
#pragma unroll
        for (int i = 0; i < kPieces; ++i) {
            const int e = tid + kT * i, j = e / (kD / 4), d = 4 * (e % (kD / 4));
            const float4 kk = *reinterpret_cast<const float4*>(&sm.stage[buf][0][j][d]);
            const float4 vv = *reinterpret_cast<const float4*>(&sm.stage[buf][1][j][d]);
            const __half2 k01 = __floats2half2_rn(kk.x, kk.y), k23 = __floats2half2_rn(kk.z, kk.w);
            const __half2 v01 = __floats2half2_rn(vv.x, vv.y), v23 = __floats2half2_rn(vv.z, vv.w);
            const float2 f01 = __half22float2(v01), f23 = __half22float2(v23);
            *reinterpret_cast<__half2*>(&sm.k[j][d]) = k01;
            *reinterpret_cast<__half2*>(&sm.k[j][d + 2]) = k23;
            *reinterpret_cast<__half2*>(&sm.vh[j][d]) = v01;
            *reinterpret_cast<__half2*>(&sm.vh[j][d + 2]) = v23;
            *reinterpret_cast<__half2*>(&sm.vl[j][d]) = __floats2half2_rn(vv.x - f01.x, vv.y - f01.y);
            *reinterpret_cast<__half2*>(&sm.vl[j][d + 2]) = __floats2half2_rn(vv.z - f23.x, vv.w - f23.y);
        }
        __syncthreads();
        if (!compute) continue;
        if (j0 == 0) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                ldsm_x4(qf[kk], &sm.q[warp][(lane & 8) + (lane & 7)][16 * kk + ((lane >> 4) << 3)]);
        }
        // Scores for the 64 keys: eight 16 x 8 tiles.
        float s[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
#pragma unroll
            for (int kk = 0; kk < 4; kk += 2) {
                uint32_t b[4];
                ldsm_x4(b, &sm.k[8 * n + (lane & 7)][16 * kk + 8 * (lane >> 3)]);
                mma16816(s[n], qf[kk], b[0], b[1]);
                mma16816(s[n], qf[kk + 1], b[2], b[3]);
            }
        }
        // Causal mask, online softmax (base 2; the scale folds in log2 e).
        float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const int j = j0 + 8 * n + 2 * ti;
            s[n][0] = j <= pa ? s[n][0] * kScaleLog2 : -INFINITY;
            s[n][1] = j + 1 <= pa ? s[n][1] * kScaleLog2 : -INFINITY;
            s[n][2] = j <= pb ? s[n][2] * kScaleLog2 : -INFINITY;
            s[n][3] = j + 1 <= pb ? s[n][3] * kScaleLog2 : -INFINITY;
            mx_a = fmaxf(mx_a, fmaxf(s[n][0], s[n][1]));
            mx_b = fmaxf(mx_b, fmaxf(s[n][2], s[n][3]));
        }
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
        const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
        const float ua = mn_a == -INFINITY ? 0.f : mn_a, ub = mn_b == -INFINITY ? 0.f : mn_b;
        const float ca = exp2f(m_a - ua), cb = exp2f(m_b - ub);
        m_a = mn_a;
        m_b = mn_b;
        float sa = 0.f, sb = 0.f;
        uint32_t pf[4][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const float p0 = exp2f(s[n][0] - ua), p1 = exp2f(s[n][1] - ua);
            const float p2 = exp2f(s[n][2] - ub), p3 = exp2f(s[n][3] - ub);
            sa += p0 + p1;
            sb += p2 + p3;
            // Score tile n is half of the A fragment of key step n / 2.
            pf[n >> 1][(n & 1) * 2] = pack_h2(p0, p1);
            pf[n >> 1][(n & 1) * 2 + 1] = pack_h2(p2, p3);
        }
        l_a = fmaf(l_a, ca, sa);
        l_b = fmaf(l_b, cb, sb);
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            o[n][0] *= ca;
            o[n][1] *= ca;
            o[n][2] *= cb;
            o[n][3] *= cb;
        }
        // o += p . (v_hi + v_lo).
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
            for (int n = 0; n < 8; n += 2) {
                const int jr = 16 * kk + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int dc = 8 * n + (lane >> 4) * 8;
                uint32_t bh[4], bl[4];
                ldsm_x4_t(bh, &sm.vh[jr][dc]);
                ldsm_x4_t(bl, &sm.vl[jr][dc]);
                mma16816(o[n], pf[kk], bh[0], bh[1]);
                mma16816(o[n], pf[kk], bl[0], bl[1]);
                mma16816(o[n + 1], pf[kk], bh[2], bh[3]);
                mma16816(o[n + 1], pf[kk], bl[2], bl[3]);
            }
        }
    }
    if (!compute) return;
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
    const float ia = 1.f / l_a, ib = 1.f / l_b;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
        const int d = 8 * n + 2 * ti;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int r = gi + 8 * half;
            if (r >= nr) continue;
            const float inv = half ? ib : ia;
            const float v0 = o[n][2 * half] * inv, v1 = o[n][2 * half + 1] * inv;
            const size_t off = (size_t)(r0 + r) * a.nh * kD + (size_t)hq * kD + d;
            const __half2 h = __floats2half2_rn(v0, v1);
            const float2 hf = __half22float2(h);
            *reinterpret_cast<__half2*>(a.o_h + off) = h;
            *reinterpret_cast<__half2*>(a.o_l + off) = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
        }
    }
}

}  // namespace

cudaError_t enqueue_attn_prefill_mma(const PrefillAttnArgs& a, int layer, int n_blk, cudaStream_t st) {
    k_attn_prefill_mma<<<dim3(a.nkv, n_blk), kT, sizeof(AttnTcSmem), st>>>(a, layer);
    return cudaGetLastError();
}

cudaError_t prefill_attn_mma_set_smem() {
    return cudaFuncSetAttribute(k_attn_prefill_mma, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sizeof(AttnTcSmem));
}

}  // namespace qwen2
