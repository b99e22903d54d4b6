// Prefill on CUDA cores with f32 activations: per-row embedding gather and
// RMSNorm, a tiled f32 x f16 GEMM whose epilogues carry the QKV bias + NeoX
// RoPE + KV store, the residual add, or SiLU(gate) * up; a flash-style
// causal GQA attention over the KV cache; the tail-row cut (minfer "Qwen2 /
// Qwen2.5 Architecture Support", section 3, "G3 tail-row optimization"); and
// the LM head on the kept rows.
#include <algorithm>

#include "attn.cuh"
#include "prefill.h"
#include "rowdot.cuh"

namespace qwen2 {

namespace {

constexpr int kT = 256;
constexpr int kGemvRows = 32;   // at most this many rows: o_proj and FFN as GEMVs

// A weight matrix in f16 (w), Q8_0 (q, d) or Q4_0 (q4: q holds two codes
// a byte); see DevMat.
struct WMat {
    const __half* w;
    const int8_t* q;
    const __half* d;
    int q4;
};
WMat wmat(const DevMat& m) { return WMat{m.w, m.q, m.d, m.q4 ? 1 : 0}; }

// Element j of row r of a block-quantised matrix with K columns: the code
// as a signed integer (Q8_0: the int8; Q4_0: the nibble minus 8).
__device__ __forceinline__ int wq_code(const WMat& m, size_t r, int K, int j) {
    if (!m.q4) return m.q[r * K + j];
    const unsigned byte = (unsigned char)m.q[r * (K / 2) + j / 2];
    return (int)((j & 1) ? byte >> 4 : byte & 0xFu) - 8;
}

__global__ void __launch_bounds__(kT) k_embed_rows(const int* __restrict__ tok, int V, int H, WMat E,
                                                   float* __restrict__ x, int* err) {
    const int r = blockIdx.x;
    int t = tok[r];
    if (t < 0 || t >= V) {
        if (threadIdx.x == 0) raise_guard(err, kGuardToken);
        t = 0;
    }
    for (int j = threadIdx.x; j < H; j += blockDim.x)
        x[(size_t)r * H + j] = E.w ? __half2float(E.w[(size_t)t * H + j])
                                   : __half2float(E.d[(size_t)t * (H / 32) + j / 32]) * (float)wq_code(E, t, H, j);
}

// v as an f16 pair: hi = f16(v), lo = f16(v - hi) (v - hi is exact in f32).
__device__ __forceinline__ void put_split(__half* hi, __half* lo, size_t i, float v) {
    const __half h = __float2half_rn(v);
    hi[i] = h;
    lo[i] = __float2half_rn(v - __half2float(h));
}

// out[r] = RMSNorm(x[r]) * w in f32, or, for the tensor-core operands, as
// f16 hi / lo pairs.
__global__ void __launch_bounds__(kT) k_norm_rows_split(const float* __restrict__ x, int H,
                                                        const float* __restrict__ w, float eps,
                                                        __half* __restrict__ hi, __half* __restrict__ lo) {
    __shared__ float red[kT / 32];
    pdl_launch_dependents();
    pdl_wait();
    const int r = blockIdx.x;
    const float* xr = x + (size_t)r * H;
    float ss = 0.f;
    for (int j = threadIdx.x; j < H; j += blockDim.x) {
        const float v = xr[j];
        ss = fmaf(v, v, ss);
    }
    const float s = rms_scale(block_sum(ss, red), H, eps);
    for (int j = threadIdx.x; j < H; j += blockDim.x)
        put_split(hi, lo, (size_t)r * H + j, __fmul_rn(__fmul_rn(xr[j], s), w[j]));
}

// The same normalisation with one warp per row and every load of the row
// issued at once (H a multiple of 4, H <= 32 * 4 * kNormSteps): rows * 32
// threads in all, kT / 32 rows per CTA.
constexpr int kNormSteps = 8;
__global__ void __launch_bounds__(kT) k_norm_rows_split_w(const float* __restrict__ x, int rows, int H,
                                                          const float* __restrict__ w, float eps,
                                                          __half* __restrict__ hi, __half* __restrict__ lo) {
    const int r = blockIdx.x * (kT / 32) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    pdl_launch_dependents();
    if (r >= rows) return;
    pdl_wait();
    const float* xr = x + (size_t)r * H;
    float4 v[kNormSteps];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kNormSteps; ++i) {
        const int j = 4 * lane + 128 * i;
        v[i] = j < H ? *reinterpret_cast<const float4*>(xr + j) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < kNormSteps; ++i) {
        ss = fmaf(v[i].x, v[i].x, ss);
        ss = fmaf(v[i].y, v[i].y, ss);
        ss = fmaf(v[i].z, v[i].z, ss);
        ss = fmaf(v[i].w, v[i].w, ss);
    }
    const float s = rms_scale(warp_sum(ss), H, eps);
#pragma unroll
    for (int i = 0; i < kNormSteps; ++i) {
        const int j = 4 * lane + 128 * i;
        if (j >= H) break;
        const float4 g = *reinterpret_cast<const float4*>(w + j);
        const size_t o = (size_t)r * H + j;
        // The four elements' hi and lo halves, each written as one 8-byte
        // store (a warp writes 256 contiguous bytes of each array).
        const float n4[4] = {__fmul_rn(__fmul_rn(v[i].x, s), g.x), __fmul_rn(__fmul_rn(v[i].y, s), g.y),
                             __fmul_rn(__fmul_rn(v[i].z, s), g.z), __fmul_rn(__fmul_rn(v[i].w, s), g.w)};
        __align__(8) __half h4[4], l4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            h4[e] = __float2half_rn(n4[e]);
            l4[e] = __float2half_rn(n4[e] - __half2float(h4[e]));
        }
        *reinterpret_cast<uint2*>(hi + o) = *reinterpret_cast<const uint2*>(h4);
        *reinterpret_cast<uint2*>(lo + o) = *reinterpret_cast<const uint2*>(l4);
    }
}

// Normalise rows of x into the f16 hi / lo operand pair.
void launch_norm_split(const float* x, int rows, int H, const float* w, float eps, __half* hi, __half* lo,
                       cudaStream_t st) {
    if (H % 4 == 0 && H <= 32 * 4 * kNormSteps)
        launch_pdl(k_norm_rows_split_w, dim3((rows + kT / 32 - 1) / (kT / 32)), dim3(kT), 0, st, x, rows, H, w, eps,
                   hi, lo);
    else
        launch_pdl(k_norm_rows_split, dim3(rows), dim3(kT), 0, st, x, H, w, eps, hi, lo);
}

__global__ void __launch_bounds__(kT) k_norm_rows(const float* __restrict__ x, int H, const float* __restrict__ w,
                                                  float eps, float* __restrict__ out) {
    __shared__ float red[kT / 32];
    const int r = blockIdx.x;
    const float* xr = x + (size_t)r * H;
    float ss = 0.f;
    for (int j = threadIdx.x; j < H; j += blockDim.x) {
        const float v = xr[j];
        ss = fmaf(v, v, ss);
    }
    const float s = rms_scale(block_sum(ss, red), H, eps);
    for (int j = threadIdx.x; j < H; j += blockDim.x) out[(size_t)r * H + j] = __fmul_rn(__fmul_rn(xr[j], s), w[j]);
}

// ---------------------------------------------------------------------------
// C[M][N] = A[M][K] . W[N][K]^T, A f32 row-major, W f16 (packed rows).
// 128 x 128 tile, K step 16, 256 threads; thread (ty, tx) owns rows
// ty + 16 i and columns tx + 16 j (i, j < 8).
// ---------------------------------------------------------------------------
constexpr int GBM = 128, GBN = 128, GBK = 16;

__device__ __forceinline__ void epilogue_store(const PrefillEpi& e, int m, int n, float v, float v_next_col) {
    const int H = e.H;
    switch (e.kind) {
    case kEpiResidual:
        e.x[(size_t)m * H + n] += v;
        break;
    case kEpiSwiGLU:
        // Even column 2j holds gate j, column 2j+1 up j.
        if ((n & 1) == 0) e.mlp[(size_t)m * e.I + (n >> 1)] = silu_f(v) * v_next_col;
        break;
    case kEpiLogits:
        e.lg[(size_t)m * e.lg_ld + n] = v;
        break;
    case kEpiQKV: {
        if (n & 1) break;
        const int kHd = e.hd;
        const int s = n / kHd, i = (n % kHd) >> 1;
        const int p = e.pos[m];
        if (p < 0 || p >= e.n_ctx) {
            raise_guard(e.err, kGuardPosition);
            break;
        }
        const float v0 = v + e.bias[n], v1 = v_next_col + e.bias[n + 1];
        const size_t head_stride = (size_t)e.n_ctx * kHd;
        const size_t cache0 = ((size_t)e.slot[m] * e.L + e.layer) * 2 * e.nkv;
        if (s < e.nh + e.nkv) {
            float ra, rb;
            rope_pair(v0, v1, e.rope[(size_t)p * (kHd / 2) + i], ra, rb);
            if (s < e.nh) {
                float* qr = e.q + (size_t)m * e.nh * kHd + s * kHd;
                qr[i] = ra;
                qr[i + kHd / 2] = rb;
            } else {
                float* kr = e.kv + (cache0 + (s - e.nh)) * head_stride + (size_t)p * kHd;
                kr[i] = ra;
                kr[i + kHd / 2] = rb;
            }
        } else {
            float* vr = e.kv + (cache0 + e.nkv + (s - e.nh - e.nkv)) * head_stride + (size_t)p * kHd;
            vr[i] = v0;
            vr[i + kHd / 2] = v1;
        }
        break;
    }
    }
}

__global__ void __launch_bounds__(kT) k_gemm_f32(const float* __restrict__ A, WMat W, int M, int N, int K,
                                                 PrefillEpi e) {
    __shared__ float As[GBK][GBM + 1];
    __shared__ float Ws[GBK][GBN + 1];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int m0 = blockIdx.y * GBM, n0 = blockIdx.x * GBN;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    for (int k0 = 0; k0 < K; k0 += GBK) {
        // A tile: 128 rows x 16 k = 512 float4.
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int idx = tid + t * kT;
            const int r = idx >> 2, k4 = (idx & 3) * 4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (m0 + r < M) v = *reinterpret_cast<const float4*>(A + (size_t)(m0 + r) * K + k0 + k4);
            As[k4][r] = v.x;
            As[k4 + 1][r] = v.y;
            As[k4 + 2][r] = v.z;
            As[k4 + 3][r] = v.w;
        }
        {
            // W tile: 128 rows x 16 k = 256 x 8 values (Q8_0: the exact
            // product of the block scale and the int8 value, in f32).
            const int r = tid >> 1, k8 = (tid & 1) * 8;
            if (W.w) {
                uint4 w = make_uint4(0, 0, 0, 0);
                if (n0 + r < N) w = ld_stream_v4(W.w + (size_t)(n0 + r) * K + k0 + k8);
                float2 f;
                f = h2_to_f2(w.x); Ws[k8 + 0][r] = f.x; Ws[k8 + 1][r] = f.y;
                f = h2_to_f2(w.y); Ws[k8 + 2][r] = f.x; Ws[k8 + 3][r] = f.y;
                f = h2_to_f2(w.z); Ws[k8 + 4][r] = f.x; Ws[k8 + 5][r] = f.y;
                f = h2_to_f2(w.w); Ws[k8 + 6][r] = f.x; Ws[k8 + 7][r] = f.y;
            } else if (W.q4) {
                // Q4_0: 8 codes in one word, element 2j in the low nibble
                // of byte j; the exact product of the scale and code - 8.
                uint32_t q4 = 0x88888888u;
                float dsc = 0.f;
                if (n0 + r < N) {
                    q4 = *reinterpret_cast<const uint32_t*>(W.q + (size_t)(n0 + r) * (K / 2) + (k0 + k8) / 2);
                    dsc = __half2float(W.d[(size_t)(n0 + r) * (K / 32) + (k0 + k8) / 32]);
                }
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    Ws[k8 + i][r] = dsc * (float)((int)((q4 >> (4 * i)) & 0xFu) - 8);
            } else {
                uint2 q8 = make_uint2(0, 0);
                float dsc = 0.f;
                if (n0 + r < N) {
                    q8 = *reinterpret_cast<const uint2*>(W.q + (size_t)(n0 + r) * K + k0 + k8);
                    dsc = __half2float(W.d[(size_t)(n0 + r) * (K / 32) + (k0 + k8) / 32]);
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t word = i < 4 ? q8.x : q8.y;
                    Ws[k8 + i][r] = dsc * (float)(int8_t)((word >> (8 * (i & 3))) & 0xffu);
                }
            }
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < GBK; ++kk) {
            float av[8], bv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) av[i] = As[kk][ty + 16 * i];
#pragma unroll
            for (int j = 0; j < 8; ++j) bv[j] = Ws[kk][tx + 16 * j];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
    // Columns 2j and 2j+1 sit in lanes tx and tx+1 (tx even): pass the odd
    // column's value down one lane for the pair epilogues.
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float nxt = __shfl_down_sync(0xffffffffu, acc[i][j], 1);
            const int m = m0 + ty + 16 * i, n = n0 + tx + 16 * j;
            if (m < M && n < N) epilogue_store(e, m, n, acc[i][j], nxt);
        }
    }
}

// ---------------------------------------------------------------------------
// Quantised prefill products (QWEN2_PREFILL_Q8_ACT): activation rows in
// Q8_0 (reading of the minfer page, section 6: the CUDA prefill's int8
// "MMQ" product), weights in Q8_0.
// ---------------------------------------------------------------------------

// Each f32 row x[r][0..K) to Q8_0 blocks, as the weight packer quantises:
// d = max|x| / 127 (f32), q = clamp(round-half-away(x / d), -127, 127) with
// an f32 division by the unrounded d (q = 0 where d = 0), scale stored as
// f16(d).  One warp per 32-block, lane = element.
__global__ void __launch_bounds__(kT) k_quant_rows_q8(const float* __restrict__ x, int rows, int K,
                                                      int8_t* __restrict__ q, __half* __restrict__ d) {
    const int lane = threadIdx.x & 31;
    const int nb = K / 32;
    for (int blk = blockIdx.x * (kT / 32) + (threadIdx.x >> 5); blk < rows * nb; blk += gridDim.x * (kT / 32)) {
        const int r = blk / nb, b = blk % nb;
        const float v = x[(size_t)r * K + b * 32 + lane];
        const float amax = warp_max(fabsf(v));
        const float dd = amax / 127.0f;
        int c = 0;
        if (dd != 0.f) c = (int)fminf(127.f, fmaxf(-127.f, roundf(v / dd)));  // half away from zero
        q[(size_t)r * K + b * 32 + lane] = (int8_t)c;
        if (lane == 0) d[(size_t)r * nb + b] = __float2half_rn(dd);
    }
}

// C[M][N] = sum over 32-blocks kb of (sum_32 a[m][k] w[n][k]) * da[m][kb] * dw[n][kb]:
// each block's int8 products are summed exactly in int32 (dp4a), the
// integer scaled by the product of the two f16 scales in f32, and the
// blocks added in order.  128 x 128 tile, one 32-block per step; thread
// (ty, tx) owns rows ty + 16 i and columns tx + 16 j, as k_gemm_f32.
__global__ void __launch_bounds__(kT) k_gemm_q8a(const int8_t* __restrict__ A, const __half* __restrict__ Ad,
                                                 WMat W, int M, int N, int K, PrefillEpi e) {
    __shared__ int As[8][GBM + 1];   // [word of the block][row]
    __shared__ int Ws[8][GBN + 1];
    __shared__ float Asc[GBM], Wsc[GBN];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int m0 = blockIdx.y * GBM, n0 = blockIdx.x * GBN;
    const int nb = K / 32;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    for (int kb = 0; kb < nb; ++kb) {
        // 128 rows x 8 words of each operand: 1024 words, four per thread.
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int idx = tid + t * kT;
            const int r = idx >> 3, w = idx & 7;
            int av = 0, wv = 0;
            if (m0 + r < M) av = *reinterpret_cast<const int*>(A + (size_t)(m0 + r) * K + kb * 32 + 4 * w);
            if (n0 + r < N) wv = *reinterpret_cast<const int*>(W.q + (size_t)(n0 + r) * K + kb * 32 + 4 * w);
            As[w][r] = av;
            Ws[w][r] = wv;
        }
        if (tid < GBM) Asc[tid] = m0 + tid < M ? __half2float(Ad[(size_t)(m0 + tid) * nb + kb]) : 0.f;
        else Wsc[tid - GBM] = n0 + tid - GBM < N ? __half2float(W.d[(size_t)(n0 + tid - GBM) * nb + kb]) : 0.f;
        __syncthreads();
        int isum[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) isum[i][j] = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            int a[8], b[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] = As[w][ty + 16 * i];
#pragma unroll
            for (int j = 0; j < 8; ++j) b[j] = Ws[w][tx + 16 * j];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) isum[i][j] = __dp4a(a[i], b[j], isum[i][j]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j)
                acc[i][j] = fmaf((float)isum[i][j], Asc[ty + 16 * i] * Wsc[tx + 16 * j], acc[i][j]);
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float nxt = __shfl_down_sync(0xffffffffu, acc[i][j], 1);
            const int m = m0 + ty + 16 * i, n = n0 + tx + 16 * j;
            if (m < M && n < N) epilogue_store(e, m, n, acc[i][j], nxt);
        }
    }
}

// Greedy id of each logits row (lowest index of the maximum; NaN above
// every number), one block per row.
__global__ void __launch_bounds__(kT) k_argmax_rows(const float* __restrict__ lg, int V, int* __restrict__ ids) {
    __shared__ float sv[kT / 32];
    __shared__ int si[kT / 32];
    const int r = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float v = -INFINITY;
    int i = 0x7fffffff;
    for (int n = threadIdx.x; n < V; n += kT) argmax_merge(v, i, lg[(size_t)r * V + n], n);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, i, o);
        argmax_merge(v, i, ov, oi);
    }
    if (lane == 0) {
        sv[warp] = v;
        si[warp] = i;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kT / 32; ++w) argmax_merge(v, i, sv[w], si[w]);
        ids[r] = i;
    }
}

// ---------------------------------------------------------------------------
// Causal GQA attention for prefill rows.  Block (g, blk) takes up to 16
// rows of one sequence and, for each of their `group` query heads that read
// kv head g, runs an online softmax over key chunks of 64 positions from 0
// to the block's largest position; a row at position p sees keys 0..p.
// ---------------------------------------------------------------------------
constexpr int kQB = kPrefillQB;
constexpr int kMaxG = 8;
constexpr int kVecPerWarp = kQB * kMaxG / (kT / 32);
template <int HD>
constexpr int attn_prefill_smem() {
    return (kQB * kMaxG * HD + 64 * (HD + 1) + 64 * HD) * 4;
}

// head_dim HD (64 or 128): lane l accumulates output dims l + 32 u.
template <int HD>
__global__ void __launch_bounds__(kT) k_attn_prefill(PrefillAttnArgs a, int layer) {
    constexpr int kHd = HD, kU = HD / 32;
    extern __shared__ __align__(16) float sm[];
    float* q_s = sm;                       // [kQB*kMaxG][HD]
    float* v_s = q_s + kQB * kMaxG * kHd;  // [64][HD]
    float* k_s = v_s + 64 * kHd;           // [64][HD + 1]
    const int g = blockIdx.x, blk = blockIdx.y;
    const int r0 = a.blk_row0[blk], nr = a.blk_nrows[blk];
    const int group = a.nh / a.nkv;
    const int nv = nr * group;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int slot = a.slot[r0];
    // Largest position of the block's rows: one load per lane, a warp max.
    int pmax = lane < nr ? a.pos[r0 + lane] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pmax = max(pmax, __shfl_xor_sync(0xffffffffu, pmax, o));
    for (int e = tid; e < nv * kHd; e += kT) {
        const int v = e / kHd, d = e % kHd;
        const int ri = v / group, h = v % group;
        q_s[e] = a.q[(size_t)(r0 + ri) * a.nh * kHd + (size_t)(g * group + h) * kHd + d];
    }
    float m_[kVecPerWarp], l_[kVecPerWarp], o_[kVecPerWarp][kU];
    int p_[kVecPerWarp];
#pragma unroll
    for (int t = 0; t < kVecPerWarp; ++t) {
        m_[t] = -INFINITY;
        l_[t] = 0.f;
#pragma unroll
        for (int u = 0; u < kU; ++u) o_[t][u] = 0.f;
        const int v = warp + 8 * t;
        p_[t] = v < nv ? a.pos[r0 + v / group] : -1;
    }
    const size_t head_stride = (size_t)a.n_ctx * kHd;
    const size_t cache0 = ((size_t)slot * a.L + layer) * 2 * a.nkv;
    const float* kbase = a.kv + (cache0 + g) * head_stride;
    const float* vbase = a.kv + (cache0 + a.nkv + g) * head_stride;
    for (int j0 = 0; j0 <= pmax; j0 += 64) {
        const int nj = min(64, pmax + 1 - j0);
        __syncthreads();
        // Rows j >= nj are zeroed: their probabilities are 0, and 0 times
        // whatever an earlier kernel left in shared memory need not be 0.
        for (int e = tid; e < 64 * (kHd / 4); e += kT) {
            const int j = e / (kHd / 4), d4 = (e % (kHd / 4)) * 4;
            float4 kk = make_float4(0.f, 0.f, 0.f, 0.f), vv = kk;
            if (j < nj) {
                kk = __ldcg(reinterpret_cast<const float4*>(kbase + (size_t)(j0 + j) * kHd + d4));
                vv = __ldcg(reinterpret_cast<const float4*>(vbase + (size_t)(j0 + j) * kHd + d4));
            }
            float* kr = k_s + j * (kHd + 1) + d4;
            kr[0] = kk.x;
            kr[1] = kk.y;
            kr[2] = kk.z;
            kr[3] = kk.w;
            *reinterpret_cast<float4*>(v_s + j * kHd + d4) = vv;
        }
        __syncthreads();
#pragma unroll
        for (int t = 0; t < kVecPerWarp; ++t) {
            const int v = warp + 8 * t;
            if (v >= nv || j0 > p_[t]) continue;
            const float* qv = q_s + v * kHd;
            float s0 = 0.f, s1 = 0.f;
            const bool ok0 = lane < nj && j0 + lane <= p_[t];
            const bool ok1 = lane + 32 < nj && j0 + lane + 32 <= p_[t];
#pragma unroll 16
            for (int d = 0; d < kHd; ++d) {
                const float qd = qv[d];
                s0 = fmaf(qd, k_s[lane * (kHd + 1) + d], s0);
                s1 = fmaf(qd, k_s[(lane + 32) * (kHd + 1) + d], s1);
            }
            s0 = ok0 ? s0 * attn_scale<HD>() : -INFINITY;
            s1 = ok1 ? s1 * attn_scale<HD>() : -INFINITY;
            const float cm = warp_max(fmaxf(s0, s1));
            const float mn = fmaxf(m_[t], cm);
            const float corr = expf(m_[t] - mn);
            const float e0 = expf(s0 - mn), e1 = expf(s1 - mn);
            l_[t] = fmaf(l_[t], corr, warp_sum(e0 + e1));
            float acc[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) acc[u] = o_[t][u] * corr;
            for (int jj = 0; jj < 32; ++jj) {
                const float pj = __shfl_sync(0xffffffffu, e0, jj);
#pragma unroll
                for (int u = 0; u < kU; ++u) acc[u] = fmaf(pj, v_s[jj * kHd + lane + 32 * u], acc[u]);
            }
            for (int jj = 0; jj < 32; ++jj) {
                const float pj = __shfl_sync(0xffffffffu, e1, jj);
#pragma unroll
                for (int u = 0; u < kU; ++u) acc[u] = fmaf(pj, v_s[(jj + 32) * kHd + lane + 32 * u], acc[u]);
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) o_[t][u] = acc[u];
            m_[t] = mn;
        }
    }
#pragma unroll
    for (int t = 0; t < kVecPerWarp; ++t) {
        const int v = warp + 8 * t;
        if (v >= nv) continue;
        const int ri = v / group, h = v % group;
        const size_t off = (size_t)(r0 + ri) * a.nh * kHd + (size_t)(g * group + h) * kHd;
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (a.o_h) put_split(a.o_h, a.o_l, off + lane + 32 * u, o_[t][u] / l_[t]);
            else a.o[off + lane + 32 * u] = o_[t][u] / l_[t];
        }
    }
}

__global__ void k_gather_rows(const float* __restrict__ src, int width, const int* __restrict__ idx,
                              float* __restrict__ dst) {
    const int r = blockIdx.x;
    const float* s = src + (size_t)idx[r] * width;
    for (int j = threadIdx.x; j < width; j += blockDim.x) dst[(size_t)r * width + j] = s[j];
}

__global__ void k_gather_int(const int* __restrict__ src, const int* __restrict__ idx, int n,
                             int* __restrict__ dst) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r < n) dst[r] = src[idx[r]];
}

PrefillEpi base_epi(Ctx& c, int layer, const int* pos, const int* slot, float* x, float* q) {
    PrefillEpi e{};
    e.H = c.cfg.hidden;
    e.I = c.cfg.intermediate;
    e.nh = c.cfg.n_head;
    e.nkv = c.cfg.n_kv_head;
    e.n_ctx = c.cfg.n_ctx;
    e.L = c.cfg.n_layer;
    e.hd = c.cfg.head_dim;
    e.layer = layer;
    e.x = x;
    e.q = q;
    e.mlp = c.ws.mlp;
    e.kv = c.kv;
    e.rope = c.rope;
    e.pos = pos;
    e.slot = slot;
    e.err = c.err;
    return e;
}

dim3 gemm_grid(int M, int N) { return dim3((N + GBN - 1) / GBN, (M + GBM - 1) / GBM); }

}  // namespace

cudaError_t prefill_set_smem_limits() {
    cudaError_t e = cudaFuncSetAttribute(k_attn_prefill<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         attn_prefill_smem<64>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_attn_prefill<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 attn_prefill_smem<128>());
    return e == cudaSuccess ? prefill_attn_tc_set_smem() : e;
}

cudaError_t enqueue_prefill(Ctx& c, int rows, int n_keep, const PrefillPlan& plan, float* logits_dev,
                            int* ids_dev, cudaStream_t st) {
    const qwen2_config& g = c.cfg;
    const int H = g.hidden, I = g.intermediate, nq = g.n_head * g.head_dim;
    const bool tensor = g.prefill_mode == QWEN2_PREFILL_TENSOR;
    const bool q8a = g.prefill_mode == QWEN2_PREFILL_Q8_ACT;
    Workspace& w = c.ws;
    // A quantised-activation product: the rows of `act` to Q8_0, then the
    // exact int8 block sums against the Q8_0 weight matrix.
    auto q8a_gemm = [&](const float* act, int m, int K, const DevMat& Wm, int N, const PrefillEpi& ep) {
        const int blocks = std::min((m * (K / 32) + kT / 32 - 1) / (kT / 32), c.n_sm * 8);
        k_quant_rows_q8<<<blocks, kT, 0, st>>>(act, m, K, w.aq, w.ad);
        k_gemm_q8a<<<gemm_grid(m, N), kT, 0, st>>>(w.aq, w.ad, wmat(Wm), m, N, K, ep);
    };
    k_embed_rows<<<rows, kT, 0, st>>>(w.rows_tok, g.vocab, H, wmat(c.embed), w.x, c.err);
    float* x = w.x;
    float* q = w.q;
    const int* pos = w.rows_pos;
    const int* slot = w.rows_slot;
    int cur = rows;
    for (int l = 0; l < g.n_layer; ++l) {
        const DevLayer& L = c.layers[l];
        const bool last = l == g.n_layer - 1;
        PrefillEpi e = base_epi(c, l, pos, slot, x, q);
        // RMSNorm, stacked QKV product + bias + RoPE + KV store (all rows).
        e.kind = kEpiQKV;
        e.bias = L.bqkv;
        if (tensor) {
            launch_norm_split(x, cur, H, L.attn_norm, g.rms_eps, w.xn_h, w.xn_l, st);
            cudaError_t err = tc_gemm_qkv(c, l, cur, e, st);
            if (err != cudaSuccess) return err;
        } else if (q8a) {
            k_norm_rows<<<cur, kT, 0, st>>>(x, H, L.attn_norm, g.rms_eps, w.xn);
            q8a_gemm(w.xn, cur, H, L.wqkv, c.nqkv, e);
        } else {
            k_norm_rows<<<cur, kT, 0, st>>>(x, H, L.attn_norm, g.rms_eps, w.xn);
            k_gemm_f32<<<gemm_grid(cur, c.nqkv), kT, 0, st>>>(w.xn, wmat(L.wqkv), cur, c.nqkv, H, e);
        }
        const int* blk_row0 = plan.blk_row0;
        const int* blk_nrows = plan.blk_nrows;
        int n_blk = plan.n_blk;
        // The rest of the layer runs on tensor cores unless the tail cut
        // left only the kept rows (a handful: the CUDA-core kernels take them).
        bool tc = tensor;
        if (last && n_keep < cur) {
            // Tail cut: only the kept rows go on to attention, o_proj, FFN, head.
            k_gather_rows<<<n_keep, kT, 0, st>>>(x, H, w.keep_rows, w.x2);
            k_gather_rows<<<n_keep, kT, 0, st>>>(q, nq, w.keep_rows, w.q2);
            k_gather_int<<<(n_keep + 255) / 256, 256, 0, st>>>(w.rows_pos, w.keep_rows, n_keep, w.keep_pos);
            k_gather_int<<<(n_keep + 255) / 256, 256, 0, st>>>(w.rows_slot, w.keep_rows, n_keep, w.keep_slot);
            x = w.x2;
            q = w.q2;
            pos = w.keep_pos;
            slot = w.keep_slot;
            cur = n_keep;
            blk_row0 = plan.kblk_row0;
            blk_nrows = plan.kblk_nrows;
            n_blk = plan.n_kblk;
            e = base_epi(c, l, pos, slot, x, q);
            tc = false;
        }
        PrefillAttnArgs aa{q, w.o, tc ? w.o_h : nullptr, w.o_l, c.kv, pos, slot, blk_row0, blk_nrows,
                           g.n_head, g.n_kv_head, g.n_ctx, g.n_layer};
        if (tc) {
            cudaError_t err = enqueue_attn_prefill_tc(c, aa, plan, l, st);
            if (err != cudaSuccess) return err;
        } else {
            if (g.head_dim == 128)
                k_attn_prefill<128><<<dim3(g.n_kv_head, n_blk), kT, attn_prefill_smem<128>(), st>>>(aa, l);
            else
                k_attn_prefill<64><<<dim3(g.n_kv_head, n_blk), kT, attn_prefill_smem<64>(), st>>>(aa, l);
        }
        if (q8a) {
            e.kind = kEpiResidual;
            q8a_gemm(w.o, cur, nq, L.wo, H, e);
            k_norm_rows<<<cur, kT, 0, st>>>(x, H, L.ffn_norm, g.rms_eps, w.xn);
            e.kind = kEpiSwiGLU;
            q8a_gemm(w.xn, cur, H, L.wgu, 2 * I, e);
            e.kind = kEpiResidual;
            q8a_gemm(w.mlp, cur, I, L.wd, H, e);
        } else if (!tc && cur <= kGemvRows) {
            // A few rows (the tail cut's, or a short prompt): the decode GEMV
            // kernels stream each weight once for up to 8 rows.
            cudaError_t err = enqueue_rows_o_ffn(c, l, x, w.o, cur, st);
            if (err != cudaSuccess) return err;
        } else if (tc) {
            // o_proj + residual; RMSNorm, gate/up + SiLU * up, down + residual.
            cudaError_t err = tc_gemm_o(c, l, cur, x, st);
            if (err == cudaSuccess) {
                launch_norm_split(x, cur, H, L.ffn_norm, g.rms_eps, w.xn_h, w.xn_l, st);
                err = tc_gemm_gu(c, l, cur, st);
            }
            if (err == cudaSuccess) err = tc_gemm_down(c, l, cur, x, st);
            if (err != cudaSuccess) return err;
        } else {
            e.kind = kEpiResidual;
            k_gemm_f32<<<gemm_grid(cur, H), kT, 0, st>>>(w.o, wmat(L.wo), cur, H, nq, e);
            k_norm_rows<<<cur, kT, 0, st>>>(x, H, L.ffn_norm, g.rms_eps, w.xn);
            e.kind = kEpiSwiGLU;
            k_gemm_f32<<<gemm_grid(cur, 2 * I), kT, 0, st>>>(w.xn, wmat(L.wgu), cur, 2 * I, H, e);
            e.kind = kEpiResidual;
            k_gemm_f32<<<gemm_grid(cur, H), kT, 0, st>>>(w.mlp, wmat(L.wd), cur, H, I, e);
        }
        cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    if (q8a) {
        // Final RMSNorm (final_norm_output), then the LM head of the kept
        // rows as a quantised product into logits, and the greedy ids.
        k_norm_rows<<<n_keep, kT, 0, st>>>(x, H, c.final_norm, g.rms_eps, w.hidden);
        PrefillEpi el{};
        el.kind = kEpiLogits;
        el.lg = logits_dev ? logits_dev : w.q8a_lg;
        el.lg_ld = g.vocab;
        el.err = c.err;
        q8a_gemm(w.hidden, n_keep, H, c.lm_head, g.vocab, el);
        if (ids_dev) k_argmax_rows<<<n_keep, kT, 0, st>>>(el.lg, g.vocab, ids_dev);
        return cudaGetLastError();
    }
    if (tensor && lm_head_tc_supported(c)) return enqueue_lm_head_tc(c, x, n_keep, logits_dev, ids_dev, st);
    return enqueue_lm_head(c, x, n_keep, logits_dev, ids_dev, false, st);
}

}  // namespace qwen2
