// Decode kernels (one row per sequence, B <= 8 rows per launch):
// embedding gather, fused RMSNorm + QKV + bias + NeoX RoPE + KV store,
// split-K GQA attention with an in-kernel combine, o_proj / down GEMV with
// the residual add, fused RMSNorm + gate/up + SiLU*up, and the LM head fused
// with a two-stage block argmax.  Also the unfused variants the
// QWEN2_FLAG_NO_FUSE_* flags select.
#include <utility>

#include "attn.cuh"
#include "bgemm.cuh"
#include "ctx.h"
#include "flash_decode.cuh"
#include "rowdot.cuh"

namespace qwen2 {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kLmNtw = 4;   // Q8_0 LM head: n-tiles per warp (256 vocab rows per CTA)

struct StepArgs {
    const int* tok;
    const int* pos;
    const int* slot;
    int B;
    float* x;
    float* q;
    float* o;
    __half* o_hi;  // nullable: the attention output also as f16 hi / lo (Q8_0 product operand)
    __half* o_lo;
    float* mlp;
    float* kv;
    const float2* rope;
    int* err;
    int H, nh, nkv, I, V, n_ctx, L;
    int hd;  // head_dim: 64 or 128
    float eps;
};

__device__ __forceinline__ float* kv_ptr(const StepArgs& a, int slot, int layer, int which, int g, int p) {
    return a.kv + ((((size_t)slot * a.L + layer) * 2 + which) * a.nkv + g) * (size_t)a.n_ctx * a.hd +
           (size_t)p * a.hd;
}

// ---------------------------------------------------------------------------
// Embedding gather: x[b] = E[tok[b]] (nnterp "token_embeddings").
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) k_embed_f16(StepArgs a, const __half* __restrict__ E) {
    const int b = blockIdx.x;
    int t = a.tok[b];
    if (t < 0 || t >= a.V) {
        if (threadIdx.x == 0) raise_guard(a.err, kGuardToken);
        t = 0;
    }
    const __half* row = E + (size_t)t * a.H;
    for (int j = threadIdx.x; j < a.H; j += blockDim.x) a.x[(size_t)b * a.H + j] = __half2float(row[j]);
}

// Q8_0 embedding row: x[b][j] = f32(d[t][j / 32]) * q[t][j]; Q4_0 (q4):
// x[b][j] = f32(d[t][j / 32]) * (code - 8), code the nibble j % 2 of byte
// j / 2 of row t.
__global__ void __launch_bounds__(kThreads) k_embed_q8(StepArgs a, const int8_t* __restrict__ Eq,
                                                       const __half* __restrict__ Ed, int q4) {
    const int b = blockIdx.x;
    int t = a.tok[b];
    if (t < 0 || t >= a.V) {
        if (threadIdx.x == 0) raise_guard(a.err, kGuardToken);
        t = 0;
    }
    for (int j = threadIdx.x; j < a.H; j += blockDim.x) {
        float v;
        if (q4) {
            const unsigned byte = (unsigned char)Eq[(size_t)t * (a.H / 2) + j / 2];
            v = (float)((int)((j & 1) ? byte >> 4 : byte & 0xFu) - 8);
        } else {
            v = (float)Eq[(size_t)t * a.H + j];
        }
        a.x[(size_t)b * a.H + j] = __half2float(Ed[(size_t)t * (a.H / 32) + j / 32]) * v;
    }
}

// ---------------------------------------------------------------------------
// Epilogue of a Q/K/V row pair (packed rows 2t, 2t+1 = elements i and
// i + hd/2 of head slot s): bias, NeoX rotation for q and k, then q to the
// query buffer, k and v to the cache slot of the row's position.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void qkv_pair_epilogue(const StepArgs& a, int layer, int pair, int b, float d0,
                                                  float d1, const float* __restrict__ bias) {
    const int r0 = 2 * pair;
    const int hd = a.hd;
    const int s = r0 / hd;
    const int i = (r0 % hd) >> 1;
    const int p = a.pos[b];
    if (p < 0 || p >= a.n_ctx) {
        raise_guard(a.err, kGuardPosition);
        return;
    }
    const float v0 = d0 + bias[r0];
    const float v1 = d1 + bias[r0 + 1];
    if (s < a.nh + a.nkv) {
        float ra, rb;
        rope_pair(v0, v1, a.rope[(size_t)p * (hd / 2) + i], ra, rb);
        if (s < a.nh) {
            float* qr = a.q + (size_t)b * a.nh * hd + s * hd;
            qr[i] = ra;
            qr[i + hd / 2] = rb;
        } else {
            float* kr = kv_ptr(a, a.slot[b], layer, 0, s - a.nh, p);
            kr[i] = ra;
            kr[i + hd / 2] = rb;
        }
    } else {
        float* vr = kv_ptr(a, a.slot[b], layer, 1, s - a.nh - a.nkv, p);
        vr[i] = v0;
        vr[i + hd / 2] = v1;
    }
}

// Fused RMSNorm + stacked QKV GEMV + bias + RoPE + KV store.  One warp per
// row pair; grid-stride over the (nh + 2 nkv) hd / 2 pairs.
template <int NB>
__global__ void __launch_bounds__(kThreads) k_qkv_fused(StepArgs a, int layer, const __half* __restrict__ W,
                                                        const float* __restrict__ bias,
                                                        const float* __restrict__ norm_w, int npairs) {
    extern __shared__ __align__(16) float smem[];
    float* xs = smem;              // [NB][H]
    float* red = smem + NB * a.H;  // [kWarps]
    norm_rows_to_smem<NB>(a.x, a.B, a.H, norm_w, a.eps, xs, a.H, red);
    const int warp = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    for (int t = warp; t < npairs; t += gridDim.x * kWarps) {
        const __half* rows[2] = {W + (size_t)(2 * t) * a.H, W + (size_t)(2 * t + 1) * a.H};
        float acc[2][NB];
        warp_rows_dot<NB, 2>(rows, a.H, xs, a.H, acc);
        if (lane == 0) {
#pragma unroll
            for (int b = 0; b < NB; ++b)
                if (b < a.B) qkv_pair_epilogue(a, layer, t, b, acc[0][b], acc[1][b], bias);
        }
    }
}

// ---------------------------------------------------------------------------
// Unfused pieces (QWEN2_FLAG_NO_FUSE_QKV / _FFN): RMSNorm to a buffer, a
// plain GEMV over a row range, the QKV epilogue and SiLU*up as kernels of
// their own.  They share the norm, row-dot and epilogue routines with the
// fused kernels, so both paths produce the same bits.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) k_rmsnorm_rows(const float* __restrict__ x, int H,
                                                           const float* __restrict__ w, float eps,
                                                           float* __restrict__ out) {
    __shared__ float red[kWarps];
    const int b = blockIdx.x;
    const float* xr = x + (size_t)b * H;
    float ss = 0.f;
    for (int j = threadIdx.x; j < H; j += blockDim.x) {
        const float v = xr[j];
        ss = fmaf(v, v, ss);
    }
    const float s = rms_scale(block_sum(ss, red), H, eps);
    for (int j = threadIdx.x; j < H; j += blockDim.x)
        out[(size_t)b * H + j] = __fmul_rn(__fmul_rn(xr[j], s), w[j]);
}

// out[b][k] = W[r0 + stride*k] . xin[b] for k < n (n even); row pairs per
// warp.
template <int NB>
__global__ void __launch_bounds__(kThreads) k_gemv_rows(const __half* __restrict__ W, int K, int r0, int stride,
                                                        int n, const float* __restrict__ xin, int B,
                                                        float* __restrict__ out, int ldo) {
    extern __shared__ __align__(16) float smem[];
    float* xs = smem;
    for (int b = 0; b < NB; ++b)
        for (int j = threadIdx.x; j < K; j += blockDim.x) xs[b * K + j] = b < B ? xin[(size_t)b * K + j] : 0.f;
    __syncthreads();
    const int warp = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    for (int t = warp; 2 * t < n; t += gridDim.x * kWarps) {
        const __half* rows[2] = {W + (size_t)(r0 + stride * 2 * t) * K,
                                 W + (size_t)(r0 + stride * (2 * t + 1)) * K};
        float acc[2][NB];
        warp_rows_dot<NB, 2>(rows, K, xs, K, acc);
        if (lane == 0)
            for (int b = 0; b < NB && b < B; ++b) {
                out[(size_t)b * ldo + 2 * t] = acc[0][b];
                out[(size_t)b * ldo + 2 * t + 1] = acc[1][b];
            }
    }
}

__global__ void __launch_bounds__(kThreads) k_qkv_epilogue(StepArgs a, int layer, const float* __restrict__ raw,
                                                           int nqkv, const float* __restrict__ bias) {
    const int b = blockIdx.y;
    const int pair = blockIdx.x * blockDim.x + threadIdx.x;
    if (pair * 2 >= nqkv || b >= a.B) return;
    qkv_pair_epilogue(a, layer, pair, b, raw[(size_t)b * nqkv + 2 * pair], raw[(size_t)b * nqkv + 2 * pair + 1],
                      bias);
}

// raw[b] holds gate products in [0, I) and up products in [I, 2I).
__global__ void __launch_bounds__(kThreads) k_swiglu(const float* __restrict__ raw, int I, int B,
                                                     float* __restrict__ mlp) {
    const int b = blockIdx.y;
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= I || b >= B) return;
    const float g = raw[(size_t)b * 2 * I + j];
    const float u = raw[(size_t)b * 2 * I + I + j];
    mlp[(size_t)b * I + j] = silu_f(g) * u;
}

// ---------------------------------------------------------------------------
// Split-K GQA decode attention (head_dim HD).  Block (g, c, b) takes
// positions [c*64, min(c*64+64, p+1)) of kv head g for row b and all
// `group` query heads that read g (each K/V element is read once per
// group).  It writes the partial (max, sum, acc[HD]) per head; the last block of (b, g) to
// finish merges the partials in chunk order and writes the head outputs.
// ---------------------------------------------------------------------------
template <int HD>
__global__ void __launch_bounds__(kThreads) k_attn_decode(StepArgs a, int layer, float* __restrict__ part,
                                                          int* __restrict__ count, int max_chunks) {
    extern __shared__ __align__(16) unsigned char attn_dyn[];
    AttnSmemT<HD>& sm = *reinterpret_cast<AttnSmemT<HD>*>(attn_dyn);
    constexpr int kStride = HD + 2;  // one partial: m, l, acc[HD]
    __shared__ int last_s;
    const int g = blockIdx.x, c = blockIdx.y, b = blockIdx.z;
    const int group = a.nh / a.nkv;
    const int p = a.pos[b];
    if (p < 0 || p >= a.n_ctx) {
        if (threadIdx.x == 0 && g == 0 && c == 0) raise_guard(a.err, kGuardPosition);
        return;
    }
    const int n_pos = p + 1;
    const int n_chunks = (n_pos + kAttCh - 1) / kAttCh;
    const int j0 = c * kAttCh;
    if (j0 >= n_pos) return;
    const int nj = min(kAttCh, n_pos - j0);
    const int slot = a.slot[b];
    const int tid = threadIdx.x;

    for (int e = tid; e < group * HD; e += kThreads)
        sm.q[e / HD][e % HD] = a.q[(size_t)b * a.nh * HD + (size_t)g * group * HD + e];
    const float* kb = kv_ptr(a, slot, layer, 0, g, j0);
    const float* vb = kv_ptr(a, slot, layer, 1, g, j0);
    for (int e = tid; e < nj * (HD / 4); e += kThreads) {
        const int j = e / (HD / 4), d4 = (e % (HD / 4)) * 4;
        const float4 kk = __ldcg(reinterpret_cast<const float4*>(kb + (size_t)j * HD + d4));
        const float4 vv = __ldcg(reinterpret_cast<const float4*>(vb + (size_t)j * HD + d4));
        sm.k[j][d4] = kk.x;
        sm.k[j][d4 + 1] = kk.y;
        sm.k[j][d4 + 2] = kk.z;
        sm.k[j][d4 + 3] = kk.w;
        *reinterpret_cast<float4*>(&sm.v[j][d4]) = vv;
    }
    __syncthreads();
    attn_chunk<SyncBlock>(sm, group, nj, [&](int h, int d, float acc, float m, float l) {
        float* pr = part + (((size_t)b * a.nh + g * group + h) * max_chunks + c) * kStride;
        pr[2 + d] = acc;
        if (d == 0) {
            pr[0] = m;
            pr[1] = l;
        }
    });
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int prev = atomicAdd(&count[b * a.nkv + g], 1);
        last_s = (prev == n_chunks - 1);
    }
    __syncthreads();
    if (!last_s) return;
    __threadfence();
    // The last block of (b, g) merges the chunks in order.
    for (int e = tid; e < group * HD; e += kThreads) {
        const int h = e / HD, d = e % HD;
        const float* ph = part + (((size_t)b * a.nh + g * group + h) * max_chunks) * kStride;
        const size_t oi = (size_t)b * a.nh * HD + (size_t)(g * group + h) * HD + d;
        const float ov =
            attn_merge(n_chunks, d, [&](int cc, int i) { return __ldcg(ph + (size_t)cc * kStride + i); });
        a.o[oi] = ov;
        if (a.o_hi) bg::split_h(ov, a.o_hi[oi], a.o_lo[oi]);
    }
    if (tid == 0) count[b * a.nkv + g] = 0;
}

// ---------------------------------------------------------------------------
// y[b] += W . xin[b] over all rows of W (o_proj, down): the residual add.
// ---------------------------------------------------------------------------
template <int NB>
__global__ void __launch_bounds__(kThreads) k_gemv_residual(const __half* __restrict__ W, int N, int K,
                                                            const float* __restrict__ xin, int B,
                                                            float* __restrict__ y) {
    extern __shared__ __align__(16) float smem[];
    float* xs = smem;
    for (int b = 0; b < NB; ++b)
        for (int j = threadIdx.x; j < K; j += blockDim.x) xs[b * K + j] = b < B ? xin[(size_t)b * K + j] : 0.f;
    __syncthreads();
    const int warp = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    for (int t = warp; 2 * t < N; t += gridDim.x * kWarps) {
        const int r = 2 * t;
        const __half* rows[2] = {W + (size_t)r * K, W + (size_t)(r + 1) * K};
        float acc[2][NB];
        warp_rows_dot<NB, 2>(rows, K, xs, K, acc);
        if (lane == 0)
            for (int b = 0; b < NB && b < B; ++b) {
                y[(size_t)b * N + r] += acc[0][b];
                y[(size_t)b * N + r + 1] += acc[1][b];
            }
    }
}

// Fused RMSNorm + gate/up GEMV + SiLU(gate) * up.  Packed rows (2j, 2j+1)
// are (gate j, up j).
template <int NB>
__global__ void __launch_bounds__(kThreads) k_gateup_fused(StepArgs a, const __half* __restrict__ W,
                                                           const float* __restrict__ norm_w) {
    extern __shared__ __align__(16) float smem[];
    float* xs = smem;
    float* red = smem + NB * a.H;
    norm_rows_to_smem<NB>(a.x, a.B, a.H, norm_w, a.eps, xs, a.H, red);
    const int warp = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    for (int j = warp; j < a.I; j += gridDim.x * kWarps) {
        const __half* rows[2] = {W + (size_t)(2 * j) * a.H, W + (size_t)(2 * j + 1) * a.H};
        float acc[2][NB];
        warp_rows_dot<NB, 2>(rows, a.H, xs, a.H, acc);
        if (lane == 0)
            for (int b = 0; b < NB && b < a.B; ++b) a.mlp[(size_t)b * a.I + j] = silu_f(acc[0][b]) * acc[1][b];
    }
}

// ---------------------------------------------------------------------------
// Final RMSNorm + tied LM head + argmax.  Block k takes the vocabulary rows
// [k*span, (k+1)*span); each warp keeps its best (value, lowest index) per
// row b; the block writes its pair, and the last block to finish merges all
// pairs (stage 2) and writes the id.  In decode mode the id also becomes the
// next step's token, the position advances, and the id is recorded in the
// step history.
// ---------------------------------------------------------------------------
struct LmArgs {
    const float* xin;  // [B][H]
    const float* norm_w;
    const __half* E;
    int B, H, V, span;
    float eps;
    float* logits;  // nullable [B][V]
    float* hidden;  // [B][H]
    float* am_val;  // [gridDim][8]
    int* am_idx;
    int* count;
    int* ids;  // nullable [B]
    int decode;
    int* tok;
    int* pos;
    int* step;
    int* ids_hist;
    int hist_stride;
    int* err;
};

template <int NB>
__global__ void __launch_bounds__(kThreads) k_lm_head(LmArgs a) {
    extern __shared__ __align__(16) float smem[];
    float* xs = smem;
    float* red = smem + NB * a.H;
    __shared__ float wv_s[kWarps][NB];
    __shared__ int wi_s[kWarps][NB];
    __shared__ int last_s;
    norm_rows_to_smem<NB>(a.xin, a.B, a.H, a.norm_w, a.eps, xs, a.H, red);
    if (blockIdx.x == 0)
        for (int b = 0; b < a.B; ++b)
            for (int j = threadIdx.x; j < a.H; j += blockDim.x) a.hidden[(size_t)b * a.H + j] = xs[b * a.H + j];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r_begin = blockIdx.x * a.span;
    const int r_end = min(a.V, r_begin + a.span);
    float best_v[NB];
    int best_i[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        best_v[b] = -INFINITY;
        best_i[b] = 0x7fffffff;
    }
    for (int r = r_begin + 2 * warp; r < r_end; r += 2 * kWarps) {
        const bool two = r + 1 < r_end;
        const __half* rows[2] = {a.E + (size_t)r * a.H, a.E + (size_t)(two ? r + 1 : r) * a.H};
        float acc[2][NB];
        warp_rows_dot<NB, 2>(rows, a.H, xs, a.H, acc);
        if (lane == 0) {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (b >= a.B) continue;
                if (a.logits) {
                    a.logits[(size_t)b * a.V + r] = acc[0][b];
                    if (two) a.logits[(size_t)b * a.V + r + 1] = acc[1][b];
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
        for (int w = 1; w < kWarps; ++w) argmax_merge(v, i, wv_s[w][b], wi_s[w][b]);
        a.am_val[blockIdx.x * 8 + b] = v;
        a.am_idx[blockIdx.x * 8 + b] = i;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last_s = (atomicAdd(a.count, 1) == (int)gridDim.x - 1);
    __syncthreads();
    if (!last_s) return;
    __threadfence();
    // Stage 2: warp b merges the per-block pairs of row b.
    if (warp < a.B && warp < NB) {
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
            if (a.decode) {
                a.ids_hist[(size_t)(*a.step % kIdsHist) * a.hist_stride + b] = i;
                a.tok[b] = i;
                a.pos[b] = a.pos[b] + 1;
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        *a.count = 0;
        if (a.decode) *a.step = *a.step + 1;
    }
}

// ---------------------------------------------------------------------------
// The Q8_0 decode path: RMSNorm (with the split-k partials of the previous
// down product added first) writing the product operand as f16 hi / lo, and
// the epilogues of the batched product (bgemm.cuh).
// ---------------------------------------------------------------------------
// x[b] += sum_s part[s][b] (fixed order, when nparts > 0; x written back),
// then n = RMSNorm(x[b]) * w: to out (f32, nullable) and as hi / lo.
__global__ void __launch_bounds__(kThreads) k_norm_split(float* __restrict__ x, const float* __restrict__ part,
                                                         int nparts, size_t part_stride, int H,
                                                         const float* __restrict__ w, float eps,
                                                         float* __restrict__ out, __half* __restrict__ hi,
                                                         __half* __restrict__ lo) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ float red[kWarps];
    const int b = blockIdx.x;
    float* xr = x + (size_t)b * H;
    float ss = 0.f;
    for (int j = threadIdx.x; j < H; j += blockDim.x) {
        float v = xr[j];
        if (nparts > 0) {
            for (int s = 0; s < nparts; ++s) v += part[(size_t)s * part_stride + (size_t)b * H + j];
            xr[j] = v;
        }
        ss = fmaf(v, v, ss);
    }
    const float sc = rms_scale(block_sum(ss, red), H, eps);
    for (int j = threadIdx.x; j < H; j += blockDim.x) {
        const float v = __fmul_rn(__fmul_rn(xr[j], sc), w[j]);
        if (out) out[(size_t)b * H + j] = v;
        bg::split_h(v, hi[(size_t)b * H + j], lo[(size_t)b * H + j]);
    }
}

// Rows of f32 as hi / lo (the attention output of prefill's kept rows).
__global__ void __launch_bounds__(kThreads) k_split_rows(const float* __restrict__ src, int n, __half* __restrict__ hi,
                                                         __half* __restrict__ lo) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) bg::split_h(src[i], hi[i], lo[i]);
}

// Q/K/V pairs of the batched product.  start() brings the rows' positions
// and cache slots, the CTA's biases and the RoPE factors of its pairs into
// shared memory while the product runs, so the epilogue itself issues no
// dependent global loads.
constexpr int kQkvRowsMax = 16;   // output rows per CTA this epilogue supports
__shared__ int qkv_pos_s[32], qkv_slot_s[32];
__shared__ float qkv_bias_s[kQkvRowsMax];
__shared__ float2 qkv_rope_s[32][kQkvRowsMax / 2];
struct EpiQkvQ8 {
    // start() reads positions, slots, biases and the RoPE table only: they
    // stay fixed for the step, so it runs before griddepcontrol.wait.
    static constexpr bool kStartBeforeWait = true;
    StepArgs a;
    int layer;
    const float* bias;
    int n_cta0;
    __device__ __forceinline__ void start(int n0, int rows, int B) {
        n_cta0 = n0;
        const int tid = threadIdx.x;
        if (rows > kQkvRowsMax || B > 32) {
            if (tid == 0) raise_guard(a.err, kGuardShape);
            return;
        }
        const int N = (a.nh + 2 * a.nkv) * a.hd;
        if (tid < 32) {
            qkv_pos_s[tid] = tid < B ? a.pos[tid] : 0;
            qkv_slot_s[tid] = tid < B ? a.slot[tid] : 0;
        }
        if (tid < rows && n0 + tid < N) qkv_bias_s[tid] = bias[n0 + tid];
        const int np = rows / 2;
        for (int e = tid; e < 32 * np; e += blockDim.x) {
            const int b = e / np, k = e % np;
            const int p = b < B ? a.pos[b] : 0;
            const int i = ((n0 + 2 * k) % a.hd) >> 1;
            qkv_rope_s[b][k] = (p >= 0 && p < a.n_ctx) ? a.rope[(size_t)p * (a.hd / 2) + i] : make_float2(1.f, 0.f);
        }
    }
    // Packed rows (n, n + 1) = elements i and i + hd/2 of head slot s: bias,
    // NeoX rotation for q and k, then q to the query buffer, k and v to the
    // cache slot of the row's position (the arithmetic of qkv_pair_epilogue).
    __device__ __forceinline__ void pair(int b, int n, float d0, float d1, int) {
        const int s = n / a.hd, i = (n % a.hd) >> 1, k = (n - n_cta0) >> 1;
        const int p = qkv_pos_s[b];
        if (p < 0 || p >= a.n_ctx) {
            raise_guard(a.err, kGuardPosition);
            return;
        }
        const float v0 = d0 + qkv_bias_s[n - n_cta0];
        const float v1 = d1 + qkv_bias_s[n - n_cta0 + 1];
        if (s < a.nh + a.nkv) {
            float ra, rb;
            rope_pair(v0, v1, qkv_rope_s[b][k], ra, rb);
            if (s < a.nh) {
                float* qr = a.q + (size_t)b * a.nh * a.hd + s * a.hd;
                qr[i] = ra;
                qr[i + a.hd / 2] = rb;
            } else {
                float* kr = kv_ptr(a, qkv_slot_s[b], layer, 0, s - a.nh, p);
                kr[i] = ra;
                kr[i + a.hd / 2] = rb;
            }
        } else {
            float* vr = kv_ptr(a, qkv_slot_s[b], layer, 1, s - a.nh - a.nkv, p);
            vr[i] = v0;
            vr[i + a.hd / 2] = v1;
        }
    }
    __device__ __forceinline__ void finish() {}
};

// Residual add of the batched product: start() loads the CTA's slice of x
// (rows b < B, columns n_cta0 .. n_cta0 + rows - 1) into shared memory.
constexpr int kResRowsMax = 16;
__shared__ float res_x_s[32][kResRowsMax];
struct EpiResidualQ8 {
    // start() may read what the previous kernels write: after the wait.
    static constexpr bool kStartBeforeWait = false;
    float* x;
    int H;
    int n_cta0 = 0;
    int* err = nullptr;
    __device__ __forceinline__ void start(int n0, int rows, int B) {
        n_cta0 = n0;
        if (rows > kResRowsMax || B > 32) {
            if (threadIdx.x == 0) raise_guard(err, kGuardShape);
            return;
        }
        for (int e = threadIdx.x; e < B * rows; e += blockDim.x) {
            const int b = e / rows, c = e % rows;
            if (n0 + c < H) res_x_s[b][c] = x[(size_t)b * H + n0 + c];
        }
    }
    __device__ __forceinline__ void pair(int b, int n, float v0, float v1, int) {
        const int c = n - n_cta0;
        *reinterpret_cast<float2*>(x + (size_t)b * H + n) = make_float2(res_x_s[b][c] + v0, res_x_s[b][c + 1] + v1);
    }
    __device__ __forceinline__ void finish() {}
};

// Down product split over k: the partial sums of k chunk `chunk` go to
// part[chunk][b][n]; the last CTA of a row group to finish (all gridDim.y
// chunks written) adds them to the residual x in chunk order.
struct EpiDownQ8 {
    // start() may read what the previous kernels write: after the wait.
    static constexpr bool kStartBeforeWait = false;
    static constexpr int kMaxParts = 16;
    __device__ __forceinline__ void start(int, int, int) {}
    float* part;
    size_t stride;  // floats between chunks
    int N;          // output rows (hidden)
    int B;
    int rows_cta;
    float* x;
    int* count;     // [gridDim.x] arrival counters, zero between launches
    __device__ __forceinline__ void pair(int b, int n, float v0, float v1, int chunk) {
        *reinterpret_cast<float2*>(part + chunk * stride + (size_t)b * N + n) = make_float2(v0, v1);
    }
    __device__ void finish() {
        __shared__ int last_s;
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) last_s = atomicAdd(&count[blockIdx.x], 1) == (int)gridDim.y - 1;
        __syncthreads();
        if (!last_s) return;
        __threadfence();
        const int n0 = blockIdx.x * rows_cta;
        const int nr = min(rows_cta, N - n0);
        const int np = (int)gridDim.y;
        if (np <= kMaxParts && nr % 4 == 0 && N % 4 == 0 && stride % 4 == 0) {
            // Four outputs per thread step, every partial's load in flight
            // at once; the sum is still x + part 0 + part 1 + ... in order.
            const int nq = nr / 4;
            for (int e = threadIdx.x; e < B * nq; e += blockDim.x) {
                const int b = e / nq;
                const size_t i = (size_t)b * N + n0 + 4 * (e - b * nq);
                float4 pv[kMaxParts];
#pragma unroll
                for (int s = 0; s < kMaxParts; ++s)
                    if (s < np) pv[s] = __ldcg(reinterpret_cast<const float4*>(part + s * stride + i));
                float4 v = *reinterpret_cast<const float4*>(x + i);
#pragma unroll
                for (int s = 0; s < kMaxParts; ++s)
                    if (s < np) {
                        v.x += pv[s].x;
                        v.y += pv[s].y;
                        v.z += pv[s].z;
                        v.w += pv[s].w;
                    }
                *reinterpret_cast<float4*>(x + i) = v;
            }
        } else {
            for (int e = threadIdx.x; e < B * nr; e += blockDim.x) {
                const int b = e / nr;
                const size_t i = (size_t)b * N + n0 + (e - b * nr);
                float v = x[i];
                for (int s = 0; s < np; ++s) v += __ldcg(part + s * stride + i);
                x[i] = v;
            }
        }
        if (threadIdx.x == 0) count[blockIdx.x] = 0;
    }
};

// Packed rows (2j, 2j+1) = (gate j, up j): m[b][j] = SiLU(gate) * up, as
// hi / lo (the operand of the down product).
struct EpiSwigluQ8 {
    // start() may read what the previous kernels write: after the wait.
    static constexpr bool kStartBeforeWait = false;
    __half* hi;
    __half* lo;
    int I;
    __device__ __forceinline__ void start(int, int, int) {}
    __device__ __forceinline__ void pair(int b, int n, float g, float u, int) {
        const size_t i = (size_t)b * I + (n >> 1);
        bg::split_h(silu_f(g) * u, hi[i], lo[i]);
    }
    __device__ __forceinline__ void finish() {}
};

// Tied LM head + greedy argmax for up to 32 rows: logits (optional), then
// per CTA the best (value, lowest index) of each row, then the last CTA to
// finish merges them (and, for decode, feeds the ids back as next tokens).
struct EpiLmQ8 {
    // start() may read what the previous kernels write: after the wait.
    static constexpr bool kStartBeforeWait = false;
    float* logits;
    int V, B;
    float* am_val;  // [gridDim][32]
    int* am_idx;
    int* count;
    int* ids;
    int decode;
    int* tok;
    int* pos;
    int* step;
    int* ids_hist;
    int hist_stride;
    int* err;
    float bv[4];
    int bi[4];
    __device__ __forceinline__ void start(int, int, int) {}
    __device__ __forceinline__ void pair(int b, int n, float v0, float v1, int) {
        if (logits) {
            logits[(size_t)b * V + n] = v0;
            if (n + 1 < V) logits[(size_t)b * V + n + 1] = v1;
        }
        const int k = b >> 3;  // this thread's rows are m*16 + gi and m*16 + gi + 8
        argmax_merge(bv[k], bi[k], v0, n);
        if (n + 1 < V) argmax_merge(bv[k], bi[k], v1, n + 1);
    }
    __device__ void finish() {
        __shared__ float sv[bg::kWarps][32];
        __shared__ int si[bg::kWarps][32];
        __shared__ int last_s;
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, ti = lane & 3;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
#pragma unroll
            for (int o = 1; o <= 2; o <<= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv[k], o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi[k], o);
                argmax_merge(bv[k], bi[k], ov, oi);
            }
            if (ti == 0) {
                sv[warp][(k >> 1) * 16 + gi + (k & 1) * 8] = bv[k];
                si[warp][(k >> 1) * 16 + gi + (k & 1) * 8] = bi[k];
            }
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            const int b = threadIdx.x;
            float v = sv[0][b];
            int i = si[0][b];
            for (int w = 1; w < bg::kWarps; ++w) argmax_merge(v, i, sv[w][b], si[w][b]);
            am_val[blockIdx.x * 32 + b] = v;
            am_idx[blockIdx.x * 32 + b] = i;
        }
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) last_s = (atomicAdd(count, 1) == (int)gridDim.x - 1);
        __syncthreads();
        if (!last_s) return;
        __threadfence();
        for (int b = warp; b < B; b += bg::kWarps) {
            float v = -INFINITY;
            int i = 0x7fffffff;
            for (int k0 = lane; k0 < (int)gridDim.x; k0 += 32 * 8) {
                // Eight CTAs' pairs per lane in flight, merged in CTA order.
                float vv[8];
                int ii[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int k = k0 + 32 * j;
                    vv[j] = k < (int)gridDim.x ? __ldcg(am_val + k * 32 + b) : -INFINITY;
                    ii[j] = k < (int)gridDim.x ? __ldcg(am_idx + k * 32 + b) : 0x7fffffff;
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) argmax_merge(v, i, vv[j], ii[j]);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, v, o);
                const int oi = __shfl_xor_sync(0xffffffffu, i, o);
                argmax_merge(v, i, ov, oi);
            }
            if (lane == 0) {
                if (i < 0 || i >= V) {
                    raise_guard(err, kGuardShape);
                    i = 0;
                }
                if (ids) ids[b] = i;
                if (decode) {
                    ids_hist[(size_t)(*step % kIdsHist) * hist_stride + b] = i;
                    tok[b] = i;
                    pos[b] = pos[b] + 1;
                }
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            *count = 0;
            if (decode) *step = *step + 1;
        }
    }
};

// ---------------------------------------------------------------------------
// Launchers.
// ---------------------------------------------------------------------------
namespace {

StepArgs make_step_args(Ctx& c, int B, const int* tok, const int* pos, const int* slot, float* x) {
    StepArgs a;
    a.tok = tok;
    a.pos = pos;
    a.slot = slot;
    a.B = B;
    a.x = x;
    a.q = c.ws.q;
    a.o = c.ws.o;
    a.o_hi = nullptr;
    a.o_lo = nullptr;
    a.mlp = c.ws.mlp;
    a.kv = c.kv;
    a.rope = c.rope;
    a.err = c.err;
    a.H = c.cfg.hidden;
    a.nh = c.cfg.n_head;
    a.nkv = c.cfg.n_kv_head;
    a.I = c.cfg.intermediate;
    a.V = c.cfg.vocab;
    a.n_ctx = c.cfg.n_ctx;
    a.L = c.cfg.n_layer;
    a.hd = c.cfg.head_dim;
    a.eps = c.cfg.rms_eps;
    return a;
}

// The split-K decode attention for the context's head_dim.
void launch_attn_decode(const Ctx& c, const StepArgs& a, int l, cudaStream_t st) {
    const dim3 grid(c.cfg.n_kv_head, c.ws.att_max_chunks, a.B);
    if (c.cfg.head_dim == 128)
        k_attn_decode<128><<<grid, kThreads, sizeof(AttnSmemT<128>), st>>>(a, l, c.ws.att_part, c.ws.att_count,
                                                                           c.ws.att_max_chunks);
    else
        k_attn_decode<64><<<grid, kThreads, sizeof(AttnSmemT<64>), st>>>(a, l, c.ws.att_part, c.ws.att_count,
                                                                         c.ws.att_max_chunks);
}

int blocks_for(int warps_needed, int cap) {
    int b = (warps_needed + kWarps - 1) / kWarps;
    return b < 1 ? 1 : (b > cap ? cap : b);
}

template <int NB>
cudaError_t layer_step(Ctx& c, const StepArgs& a, int l, cudaStream_t st) {
    const DevLayer& L = c.layers[l];
    const int H = c.cfg.hidden, I = c.cfg.intermediate, nq = c.cfg.n_head * c.cfg.head_dim;
    const int cap = c.n_sm * 8;
    const bool fuse_qkv = !(c.cfg.flags & QWEN2_FLAG_NO_FUSE_QKV);
    const bool fuse_ffn = !(c.cfg.flags & QWEN2_FLAG_NO_FUSE_FFN);
    if (fuse_qkv) {
        const int np = c.nqkv / 2;
        k_qkv_fused<NB><<<blocks_for(np, cap), kThreads, (NB * H + kWarps) * 4, st>>>(a, l, L.wqkv.w, L.bqkv,
                                                                                      L.attn_norm, np);
    } else {
        k_rmsnorm_rows<<<a.B, kThreads, 0, st>>>(a.x, H, L.attn_norm, a.eps, c.ws.xn);
        const int nkvd = c.cfg.n_kv_head * c.cfg.head_dim;
        const int r0s[3] = {0, nq, nq + nkvd}, ns[3] = {nq, nkvd, nkvd};
        for (int part = 0; part < 3; ++part)
            k_gemv_rows<NB><<<blocks_for(ns[part] / 2, cap), kThreads, NB * H * 4, st>>>(
                L.wqkv.w, H, r0s[part], 1, ns[part], c.ws.xn, a.B, c.ws.raw + r0s[part], c.nqkv);
        k_qkv_epilogue<<<dim3((c.nqkv / 2 + kThreads - 1) / kThreads, a.B), kThreads, 0, st>>>(a, l, c.ws.raw,
                                                                                             c.nqkv, L.bqkv);
    }
    launch_attn_decode(c, a, l, st);
    k_gemv_residual<NB><<<blocks_for(H / 2, cap), kThreads, NB * nq * 4, st>>>(L.wo.w, H, nq, c.ws.o, a.B, a.x);
    if (fuse_ffn) {
        k_gateup_fused<NB><<<blocks_for(I, cap), kThreads, (NB * H + kWarps) * 4, st>>>(a, L.wgu.w, L.ffn_norm);
    } else {
        k_rmsnorm_rows<<<a.B, kThreads, 0, st>>>(a.x, H, L.ffn_norm, a.eps, c.ws.xn);
        // Gate rows (even packed rows) and up rows (odd) as two products.
        k_gemv_rows<NB><<<blocks_for(I / 2, cap), kThreads, NB * H * 4, st>>>(L.wgu.w, H, 0, 2, I, c.ws.xn, a.B,
                                                                              c.ws.raw, 2 * I);
        k_gemv_rows<NB><<<blocks_for(I / 2, cap), kThreads, NB * H * 4, st>>>(L.wgu.w, H, 1, 2, I, c.ws.xn, a.B,
                                                                              c.ws.raw + I, 2 * I);
        k_swiglu<<<dim3((I + kThreads - 1) / kThreads, a.B), kThreads, 0, st>>>(c.ws.raw, I, a.B, c.ws.mlp);
    }
    k_gemv_residual<NB><<<blocks_for(H / 2, cap), kThreads, NB * I * 4, st>>>(L.wd.w, H, I, c.ws.mlp, a.B, a.x);
    return cudaGetLastError();
}

template <int NB>
cudaError_t lm_head_nb(Ctx& c, const float* xin, int B, float* logits, int* ids, float* hidden, bool decode,
                       cudaStream_t st) {
    LmArgs la;
    la.xin = xin;
    la.norm_w = c.final_norm;
    la.E = c.lm_head.w;
    la.B = B;
    la.H = c.cfg.hidden;
    la.V = c.cfg.vocab;
    la.eps = c.cfg.rms_eps;
    const int grid = c.ws.am_blocks;
    int span = (la.V + grid - 1) / grid;
    span = (span + 1) & ~1;
    la.span = span;
    la.logits = logits;
    la.hidden = hidden;
    la.am_val = c.ws.am_val;
    la.am_idx = c.ws.am_idx;
    la.count = c.ws.am_count;
    la.ids = ids;
    la.decode = decode ? 1 : 0;
    la.tok = c.ds.tok;
    la.pos = c.ds.pos;
    la.step = c.ds.step;
    la.ids_hist = c.ds.ids_hist;
    la.hist_stride = c.cfg.max_seqs;
    la.err = c.err;
    k_lm_head<NB><<<grid, kThreads, (NB * la.H + kWarps) * 4, st>>>(la);
    return cudaGetLastError();
}

template <int NB>
cudaError_t decode_nb(Ctx& c, int B, bool want_logits, cudaStream_t st) {
    StepArgs a = make_step_args(c, B, c.ds.tok, c.ds.pos, c.ds.slot, c.ws.x);
    k_embed_f16<<<B, kThreads, 0, st>>>(a, c.embed.w);
    for (int l = 0; l < c.cfg.n_layer; ++l) {
        cudaError_t e = layer_step<NB>(c, a, l, st);
        if (e != cudaSuccess) return e;
    }
    return lm_head_nb<NB>(c, c.ws.x, B, want_logits ? c.ws.logits : nullptr, nullptr, c.ws.hidden, true, st);
}

// ---- Q8_0 weights: the batched tensor-core product for any B <= 32 ---------
// Shapes: QKV and o_proj 8 weight rows per CTA (8 warps split k); gate/up
// 64 rows per CTA; down 64 rows per CTA with k cut into chunks of
// kQ8DownKc columns (one wave of about 150 CTAs at the 0.5B shape), reduced
// into the residual by the last CTA of each row group; LM head 256 rows per
// CTA.  QKV and gate/up normalise their input rows themselves.
template <int MT, int NTW, int KS>
constexpr int bgemm_rows_cta() { return (bg::kWarps / KS) * NTW * 8; }

template <int MT, int NTW, int KS, class Epi, class Pro>
cudaError_t bgemm(const Ctx& c, const Pro& pro, int B, int K, int kc_len, const DevMat& W, int N, const Epi& e,
                  cudaStream_t st) {
    constexpr int rows_cta = bgemm_rows_cta<MT, NTW, KS>();
    const dim3 grid((N + rows_cta - 1) / rows_cta, (K + kc_len - 1) / kc_len);
    if (W.q4)
        return launch_pdl(bg::k_bgemm_q8s<MT, NTW, KS, Epi, Pro, true>, grid, dim3(bg::kThreads),
                          bg::smem_bytes_s(MT, kc_len, rows_cta, true), st, pro, B, K, kc_len, W.q, W.d, N, e,
                          c.err);
    return launch_pdl(bg::k_bgemm_q8s<MT, NTW, KS, Epi, Pro>, grid, dim3(bg::kThreads),
                      bg::smem_bytes_s(MT, kc_len, rows_cta), st, pro, B, K, kc_len, W.q, W.d, N, e, c.err);
}

constexpr int kDownNtw = 2, kDownKs = 2;
constexpr int kDownRows = (bg::kWarps / kDownKs) * kDownNtw * 8;

// The steps of one layer after the attention: o_proj + residual, RMSNorm +
// gate/up + SwiGLU, down + residual (split over k, reduced in-kernel).
template <int MT>
cudaError_t o_ffn_q8(Ctx& c, int l, float* x, int B, cudaStream_t st) {
    const DevLayer& L = c.layers[l];
    const int H = c.cfg.hidden, I = c.cfg.intermediate, nq = c.cfg.n_head * c.cfg.head_dim;
    Workspace& w = c.ws;
    cudaError_t e = bgemm<MT, 1, 8>(c, bg::ProCopy{w.q8_ah, w.q8_al}, B, nq, nq, L.wo, H, EpiResidualQ8{x, H, 0, c.err}, st);
    if (e != cudaSuccess) return e;
    e = bgemm<MT, 4, 4>(c, bg::ProNorm{x, L.ffn_norm, c.cfg.rms_eps, nullptr}, B, H, H, L.wgu, 2 * I,
                        EpiSwigluQ8{w.q8_mh, w.q8_ml, I}, st);
    if (e != cudaSuccess) return e;
    EpiDownQ8 ed{w.q8_part, (size_t)c.max_rows_q8 * H, H, B, kDownRows, x, w.q8_cnt};
    return bgemm<MT, kDownNtw, kDownKs>(c, bg::ProCopy{w.q8_mh, w.q8_ml}, B, I, kQ8DownKc, L.wd, H, ed, st);
}

// Batched decode attention of the Q8_0 path: the persistent flash-decoding
// kernel (any mix of positions, up to 32 rows, n_ctx <= 4096, group <= 8),
// else the split-K kernel.
cudaError_t attn_batched(const Ctx& c, const StepArgs& a, int l, cudaStream_t st) {
    const int group = a.nh / a.nkv;
    if (!c.kvmap_ok || a.B > fd::kMaxRows || c.ws.att_max_chunks > fd::kMaxChunks || group > fd::kGroupMax ||
        c.cfg.head_dim != fd::kDh) {
        launch_attn_decode(c, a, l, st);
        return cudaGetLastError();
    }
    fd::Args f;
    f.q = a.q;
    f.pos = a.pos;
    f.slot = a.slot;
    f.part = c.ws.att_part;
    f.count = c.ws.att_count;
    f.o = a.o;
    f.o_hi = a.o_hi;
    f.o_lo = a.o_lo;
    f.err = a.err;
    f.B = a.B;
    f.nh = a.nh;
    f.nkv = a.nkv;
    f.n_ctx = a.n_ctx;
    f.L = a.L;
    f.layer = l;
    f.max_chunks = c.ws.att_max_chunks;
    // The rest of this layer's weights (o_proj, gate/up, down, biases,
    // norms) and the next layer's Q/K/V, contiguous in the packed blob.
    f.pf = nullptr;
    f.pf_bytes = 0;
    if (block_quantised(c.cfg)) {
        const DevLayer& L = c.layers[l];
        const unsigned char* b0 = reinterpret_cast<const unsigned char*>(L.wo.q);
        const unsigned char* b1 = l + 1 < c.cfg.n_layer
                                      ? reinterpret_cast<const unsigned char*>(c.layers[l + 1].wqkv.d) +
                                            (size_t)c.layers[l + 1].wqkv.rows * (c.layers[l + 1].wqkv.k / 32) * 2
                                      : reinterpret_cast<const unsigned char*>(L.ffn_norm + c.cfg.hidden);
        if (b1 > b0 && (reinterpret_cast<uintptr_t>(b0) & 15) == 0) {
            f.pf = b0;
            f.pf_bytes = (size_t)(b1 - b0) & ~(size_t)15;
        }
    }
    const int grid = 2 * c.n_sm;
    cudaError_t e = launch_pdl(k_attn_flash, dim3(grid), dim3(fd::kThreads), fd::kSmemBytes, st, c.kvmap, f);
    if (e != cudaSuccess) return e;
    return launch_pdl(k_attn_merge, dim3(a.B * a.nkv), dim3(kMergeThreads), 0, st, f, grid);
}

template <int MT>
cudaError_t layer_q8(Ctx& c, const StepArgs& a, int l, cudaStream_t st) {
    const DevLayer& L = c.layers[l];
    const int H = c.cfg.hidden;
    Workspace& w = c.ws;
    cudaError_t e = bgemm<MT, 1, 8>(c, bg::ProNorm{a.x, L.attn_norm, a.eps, nullptr}, a.B, H, H, L.wqkv, c.nqkv,
                                    EpiQkvQ8{a, l, L.bqkv, 0}, st);
    if (e != cudaSuccess) return e;
    StepArgs ao = a;
    ao.o_hi = w.q8_ah;
    ao.o_lo = w.q8_al;
    e = attn_batched(c, ao, l, st);
    if (e != cudaSuccess) return e;
    return o_ffn_q8<MT>(c, l, a.x, a.B, st);
}

// Final RMSNorm and the tied LM head + argmax on B <= 32 rows.
template <int MT>
cudaError_t lm_head_q8(Ctx& c, float* x, int B, float* logits, int* ids, float* hidden, bool decode,
                       cudaStream_t st) {
    const int H = c.cfg.hidden;
    Workspace& w = c.ws;
    cudaError_t le = launch_pdl(k_norm_split, dim3(B), dim3(kThreads), 0, st, x, (const float*)nullptr, 0, 0, H,
                                c.final_norm, c.cfg.rms_eps, hidden, w.q8_ah, w.q8_al);
    if (le != cudaSuccess) return le;
    EpiLmQ8 e{};
    e.logits = logits;
    e.V = c.cfg.vocab;
    e.B = B;
    e.am_val = w.lm_val;
    e.am_idx = w.lm_idx;
    e.count = w.am_count;
    e.ids = ids;
    e.decode = decode ? 1 : 0;
    e.tok = c.ds.tok;
    e.pos = c.ds.pos;
    e.step = c.ds.step;
    e.ids_hist = c.ds.ids_hist;
    e.hist_stride = c.cfg.max_seqs;
    e.err = c.err;
    for (int k = 0; k < 4; ++k) {
        e.bv[k] = -INFINITY;
        e.bi[k] = 0x7fffffff;
    }
    // One CTA per SM walking the vocabulary's 256-row tiles: the activation
    // rows are staged once per SM, not once per tile.  The normalised rows
    // enter as f16 only (no lo part): the logits are the last product, and
    // an 11-bit activation rounding moves them by about 1e-3 at most at this
    // scale, far inside the 2e-2 bound, for half the tensor work.
    const int tiles = (c.cfg.vocab + bg::kWarps * kLmNtw * 8 - 1) / (bg::kWarps * kLmNtw * 8);
    const int grid = tiles < c.n_sm ? tiles : c.n_sm;
    if (c.lm_head.q4)
        return launch_pdl(bg::k_bgemm_q8_tiles<MT, kLmNtw, EpiLmQ8, bg::ProCopy, false, true>, dim3(grid),
                          dim3(bg::kThreads), bg::smem_bytes(MT, H), st, bg::ProCopy{w.q8_ah, w.q8_al}, B, H,
                          c.lm_head.q, c.lm_head.d, c.cfg.vocab, e, c.err);
    return launch_pdl(bg::k_bgemm_q8_tiles<MT, kLmNtw, EpiLmQ8, bg::ProCopy, false>, dim3(grid), dim3(bg::kThreads),
                      bg::smem_bytes(MT, H), st, bg::ProCopy{w.q8_ah, w.q8_al}, B, H, c.lm_head.q, c.lm_head.d,
                      c.cfg.vocab, e, c.err);
}

template <int MT>
cudaError_t decode_q8(Ctx& c, int B, bool want_logits, cudaStream_t st) {
    StepArgs a = make_step_args(c, B, c.ds.tok, c.ds.pos, c.ds.slot, c.ws.x);
    k_embed_q8<<<B, kThreads, 0, st>>>(a, c.embed.q, c.embed.d, c.embed.q4 ? 1 : 0);
    for (int l = 0; l < c.cfg.n_layer; ++l) {
        cudaError_t e = layer_q8<MT>(c, a, l, st);
        if (e != cudaSuccess) return e;
    }
    return lm_head_q8<MT>(c, c.ws.x, B, want_logits ? c.ws.logits : nullptr, nullptr, c.ws.hidden, true, st);
}

template <int MT>
cudaError_t rows_o_ffn_q8(Ctx& c, int l, float* x, const float* o, int B, cudaStream_t st) {
    const int nq = c.cfg.n_head * c.cfg.head_dim;
    k_split_rows<<<(B * nq + kThreads - 1) / kThreads, kThreads, 0, st>>>(o, B * nq, c.ws.q8_ah, c.ws.q8_al);
    return o_ffn_q8<MT>(c, l, x, B, st);
}

template <int NB>
cudaError_t rows_o_ffn_nb(Ctx& c, int l, float* x, const float* o, int B, cudaStream_t st) {
    const DevLayer& L = c.layers[l];
    const int H = c.cfg.hidden, I = c.cfg.intermediate, nq = c.cfg.n_head * c.cfg.head_dim;
    const int cap = c.n_sm * 8;
    StepArgs a = make_step_args(c, B, nullptr, nullptr, nullptr, x);
    k_gemv_residual<NB><<<blocks_for(H / 2, cap), kThreads, NB * nq * 4, st>>>(L.wo.w, H, nq, o, B, x);
    k_gateup_fused<NB><<<blocks_for(I, cap), kThreads, (NB * H + kWarps) * 4, st>>>(a, L.wgu.w, L.ffn_norm);
    k_gemv_residual<NB><<<blocks_for(H / 2, cap), kThreads, NB * I * 4, st>>>(L.wd.w, H, I, c.ws.mlp, B, x);
    return cudaGetLastError();
}

}  // namespace

cudaError_t enqueue_rows_o_ffn(Ctx& c, int layer, float* x, const float* o, int rows, cudaStream_t st) {
    const int H = c.cfg.hidden, nq = c.cfg.n_head * c.cfg.head_dim;
    if (block_quantised(c.cfg)) {
        for (int b0 = 0; b0 < rows; b0 += 32) {
            const int nb = rows - b0 < 32 ? rows - b0 : 32;
            cudaError_t e = nb <= 16 ? rows_o_ffn_q8<1>(c, layer, x + (size_t)b0 * H, o + (size_t)b0 * nq, nb, st)
                                     : rows_o_ffn_q8<2>(c, layer, x + (size_t)b0 * H, o + (size_t)b0 * nq, nb, st);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    for (int b0 = 0; b0 < rows; b0 += 8) {
        const int nb = rows - b0 < 8 ? rows - b0 : 8;
        float* xg = x + (size_t)b0 * H;
        const float* og = o + (size_t)b0 * nq;
        cudaError_t e;
        if (nb <= 1) e = rows_o_ffn_nb<1>(c, layer, xg, og, nb, st);
        else if (nb <= 2) e = rows_o_ffn_nb<2>(c, layer, xg, og, nb, st);
        else if (nb <= 4) e = rows_o_ffn_nb<4>(c, layer, xg, og, nb, st);
        else e = rows_o_ffn_nb<8>(c, layer, xg, og, nb, st);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t enqueue_lm_head(Ctx& c, const float* xin, int B, float* logits, int* ids, bool decode,
                            cudaStream_t st) {
    const int H = c.cfg.hidden;
    const size_t V = (size_t)c.cfg.vocab;
    if (block_quantised(c.cfg)) {
        if (decode && B > 32) return cudaErrorInvalidValue;
        for (int b0 = 0; b0 < B; b0 += 32) {
            const int nb = B - b0 < 32 ? B - b0 : 32;
            const float* xg = xin + (size_t)b0 * H;
            float* lg = logits ? logits + (size_t)b0 * V : nullptr;
            int* ig = ids ? ids + b0 : nullptr;
            float* hg = c.ws.hidden + (size_t)b0 * H;
            float* xw = const_cast<float*>(xg);
            cudaError_t e = nb <= 16 ? lm_head_q8<1>(c, xw, nb, lg, ig, hg, decode, st)
                                     : lm_head_q8<2>(c, xw, nb, lg, ig, hg, decode, st);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    if (decode && B > 8) return cudaErrorInvalidValue;
    for (int b0 = 0; b0 < B; b0 += 8) {
        const int nb = B - b0 < 8 ? B - b0 : 8;
        const float* xg = xin + (size_t)b0 * H;
        float* lg = logits ? logits + (size_t)b0 * V : nullptr;
        int* ig = ids ? ids + b0 : nullptr;
        float* hg = c.ws.hidden + (size_t)b0 * H;
        cudaError_t e;
        if (nb <= 1) e = lm_head_nb<1>(c, xg, nb, lg, ig, hg, decode, st);
        else if (nb <= 2) e = lm_head_nb<2>(c, xg, nb, lg, ig, hg, decode, st);
        else if (nb <= 4) e = lm_head_nb<4>(c, xg, nb, lg, ig, hg, decode, st);
        else e = lm_head_nb<8>(c, xg, nb, lg, ig, hg, decode, st);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t enqueue_decode_step(Ctx& c, int B, bool want_logits, cudaStream_t st) {
    if (block_quantised(c.cfg)) {
        if (B <= 16) return decode_q8<1>(c, B, want_logits, st);
        if (B <= 32) return decode_q8<2>(c, B, want_logits, st);
        return cudaErrorInvalidValue;
    }
    if (B <= 1) return decode_nb<1>(c, B, want_logits, st);
    if (B <= 2) return decode_nb<2>(c, B, want_logits, st);
    if (B <= 4) return decode_nb<4>(c, B, want_logits, st);
    if (B <= 8) return decode_nb<8>(c, B, want_logits, st);
    return cudaErrorInvalidValue;
}

// Dynamic shared-memory opt-in for the templated kernels (once at create):
// each may use the device's opt-in maximum less its static shared memory.
template <class K>
static cudaError_t allow_smem(K kern, int max_bytes) {
    cudaFuncAttributes at;
    cudaError_t e = cudaFuncGetAttributes(&at, kern);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                max_bytes - (int)at.sharedSizeBytes);
}

cudaError_t decode_set_smem_limits(int max_bytes) {
    cudaError_t e = cudaSuccess;
#define Q2_SMEM(kern) \
    if (e == cudaSuccess) e = allow_smem(kern, max_bytes);
#define Q2_SMEM_NB(NB)           \
    Q2_SMEM(k_qkv_fused<NB>)     \
    Q2_SMEM(k_gemv_rows<NB>)     \
    Q2_SMEM(k_gemv_residual<NB>) \
    Q2_SMEM(k_gateup_fused<NB>)  \
    Q2_SMEM(k_lm_head<NB>)
    Q2_SMEM_NB(1) Q2_SMEM_NB(2) Q2_SMEM_NB(4) Q2_SMEM_NB(8)
#undef Q2_SMEM_NB
#undef Q2_SMEM
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_attn_flash, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fd::kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_attn_decode<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)sizeof(AttnSmemT<128>));
#define Q2_BG(MT, NTW, KS, EPI, PRO)                                                                     \
    if (e == cudaSuccess)                                                                                \
        e = cudaFuncSetAttribute(bg::k_bgemm_q8s<MT, NTW, KS, EPI, PRO>,                                \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,                            \
                                 (int)bg::smem_bytes_s(MT, bg::kKc, bgemm_rows_cta<MT, NTW, KS>()));    \
    if (e == cudaSuccess)                                                                                \
        e = cudaFuncSetAttribute(bg::k_bgemm_q8s<MT, NTW, KS, EPI, PRO, true>,                          \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,                            \
                                 (int)bg::smem_bytes_s(MT, bg::kKc, bgemm_rows_cta<MT, NTW, KS>(), true));
#define Q2_BGT(MT)                                                                                          \
    if (e == cudaSuccess)                                                                                   \
        e = cudaFuncSetAttribute(bg::k_bgemm_q8_tiles<MT, kLmNtw, EpiLmQ8, bg::ProCopy, false>,                     \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bg::smem_bytes(MT, bg::kKc)); \
    if (e == cudaSuccess)                                                                                   \
        e = cudaFuncSetAttribute(bg::k_bgemm_q8_tiles<MT, kLmNtw, EpiLmQ8, bg::ProCopy, false, true>,               \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bg::smem_bytes(MT, bg::kKc));
    Q2_BGT(1) Q2_BGT(2)
#undef Q2_BGT
#define Q2_BG_MT(MT)                                          \
    Q2_BG(MT, 1, 8, EpiQkvQ8, bg::ProNorm)                    \
    Q2_BG(MT, 1, 8, EpiResidualQ8, bg::ProCopy)               \
    Q2_BG(MT, 4, 4, EpiSwigluQ8, bg::ProNorm)                 \
    Q2_BG(MT, kDownNtw, kDownKs, EpiDownQ8, bg::ProCopy)
    Q2_BG_MT(1) Q2_BG_MT(2)
#undef Q2_BG_MT
#undef Q2_BG
    return e;
}

namespace {

// Stop tokens (minfer page section 5, "Tokenizer and chat": generation ends
// at eos or im_end) over one chunk of the id history, one thread per
// sequence, steps in order: once a sequence has generated one of the stop
// ids, its later ids become -1; n_gen counts the ids kept, the stop id
// included.  done / n_gen carry over from the previous chunk of the same
// run unless `first`.
__global__ void k_stop_mask(int* ids_hist, int stride, int n_steps, int n_seq, const int* stop_ids, int n_stop,
                            int* done, int* n_gen, int first) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= n_seq) return;
    int stop[kMaxStopIds];
    for (int k = 0; k < kMaxStopIds; ++k) stop[k] = k < n_stop ? stop_ids[k] : -1;
    int d = first ? 0 : done[b];
    int g = first ? 0 : n_gen[b];
    for (int s = 0; s < n_steps; ++s) {
        int* p = ids_hist + (size_t)s * stride + b;
        if (d) {
            *p = -1;
            continue;
        }
        const int id = *p;
        ++g;
        for (int k = 0; k < kMaxStopIds; ++k)
            if (k < n_stop && id == stop[k]) d = 1;
    }
    done[b] = d;
    n_gen[b] = g;
}

// The guard write of a kernel whose bounded wait gave up, on its own.
__global__ void k_raise_guard(int* err, int code) { raise_guard(err, code); }

}  // namespace

cudaError_t enqueue_raise_guard(Ctx& c, int code, cudaStream_t st) {
    k_raise_guard<<<1, 1, 0, st>>>(c.err, code);
    return cudaGetLastError();
}

cudaError_t enqueue_stop_mask(Ctx& c, int n_seq, int n_steps, int n_stop, bool first, cudaStream_t st) {
    if (n_seq < 1 || n_seq > c.cfg.max_seqs || n_steps < 1 || n_steps > kIdsHist || n_stop < 0 ||
        n_stop > kMaxStopIds)
        return cudaErrorInvalidValue;
    const int threads = 128;
    k_stop_mask<<<(n_seq + threads - 1) / threads, threads, 0, st>>>(c.ds.ids_hist, c.cfg.max_seqs, n_steps, n_seq,
                                                                        c.ds.stop_ids, n_stop, c.ds.stop_done,
                                                                        c.ds.n_gen, first ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace qwen2
