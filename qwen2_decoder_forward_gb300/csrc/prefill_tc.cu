// Tensor-core prefill GEMMs (QWEN2_PREFILL_TENSOR): the four products of a
// layer on f16 operands with f32 accumulation, each with its epilogue fused
// (minfer "Qwen2 / Qwen2.5 Architecture Support", section 1 layer diagram;
// section 3 fused QKV and gate/up):
//   QKV   bias, NeoX RoPE on q and k, q to the workspace, k and v to the f32
//         KV cache at the row's position;
//   O     x += o . Wo^T;
//   GU    m = SiLU(gate) * up, written as the f16 operand of the down product;
//   DOWN  x += m . Wd^T.
// Operand rows arrive through TMA tensor maps encoded once per context.
#include "prefill.h"
#include "rowdot.cuh"
#include "tc_gemm.cuh"
#include "tmap.h"

namespace qwen2 {

namespace {

constexpr int kHdim = 64;

// Output chunk (m, n0..n0+31) of the packed Q/K/V product: 16 adjacent
// (2i, 2i+1) pairs of head slot n0 / 64, i = i0..i0+15.
struct EpiQKV {
    int nh, nkv, n_ctx, L, layer;
    float* q;
    float* kv;
    const float2* rope;
    const float* bias;
    const int* pos;
    const int* slot;
    int* err;
    // The attention's f16 operands of the row's key and value (see
    // prefill_attn_tc.cu): k as att_k [slot][kv head][n_ctx64][64], v
    // transposed as the hi / lo pair att_vt [slot][kv head][2][64][n_ctx64].
    __half* att_k;
    __half* att_vt;
    int n_ctx64;
    __device__ __forceinline__ void store(int m, int n0, const float (&v)[32]) const {
        const int s = n0 / kHdim, i0 = (n0 % kHdim) >> 1;
        const int p = pos[m];
        if (p < 0 || p >= n_ctx) {
            raise_guard(err, kGuardPosition);
            return;
        }
        float a[16], b[16];
        const float4* bias4 = reinterpret_cast<const float4*>(bias + n0);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 bb = bias4[j];
            a[2 * j] = v[4 * j] + bb.x;
            b[2 * j] = v[4 * j + 1] + bb.y;
            a[2 * j + 1] = v[4 * j + 2] + bb.z;
            b[2 * j + 1] = v[4 * j + 3] + bb.w;
        }
        float* dst;
        const size_t head_stride = (size_t)n_ctx * kHdim;
        const size_t cache0 = ((size_t)slot[m] * L + layer) * 2 * nkv;
        if (s < nh + nkv) {
            const float2* cs = rope + (size_t)p * (kHdim / 2) + i0;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                float ra, rb;
                rope_pair(a[j], b[j], cs[j], ra, rb);
                a[j] = ra;
                b[j] = rb;
            }
            dst = s < nh ? q + (size_t)m * nh * kHdim + (size_t)s * kHdim
                         : kv + (cache0 + (s - nh)) * head_stride + (size_t)p * kHdim;
        } else {
            dst = kv + (cache0 + nkv + (s - nh - nkv)) * head_stride + (size_t)p * kHdim;
        }
        float4* lo = reinterpret_cast<float4*>(dst + i0);
        float4* hi = reinterpret_cast<float4*>(dst + i0 + kHdim / 2);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            lo[j] = make_float4(a[4 * j], a[4 * j + 1], a[4 * j + 2], a[4 * j + 3]);
            hi[j] = make_float4(b[4 * j], b[4 * j + 1], b[4 * j + 2], b[4 * j + 3]);
        }
        if (s < nh) return;
        // Dims i0 .. i0 + 15 hold a[], dims i0 + 32 .. i0 + 47 hold b[].
        if (s < nh + nkv) {
            const size_t head = (size_t)slot[m] * nkv + (s - nh);
            __half* kr = att_k + (head * n_ctx64 + p) * kHdim;
            uint32_t ha[8], hb[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const __half2 x = __floats2half2_rn(a[2 * j], a[2 * j + 1]);
                const __half2 y = __floats2half2_rn(b[2 * j], b[2 * j + 1]);
                ha[j] = *reinterpret_cast<const uint32_t*>(&x);
                hb[j] = *reinterpret_cast<const uint32_t*>(&y);
            }
            uint4* da = reinterpret_cast<uint4*>(kr + i0);
            uint4* db = reinterpret_cast<uint4*>(kr + i0 + kHdim / 2);
            da[0] = make_uint4(ha[0], ha[1], ha[2], ha[3]);
            da[1] = make_uint4(ha[4], ha[5], ha[6], ha[7]);
            db[0] = make_uint4(hb[0], hb[1], hb[2], hb[3]);
            db[1] = make_uint4(hb[4], hb[5], hb[6], hb[7]);
        } else {
            const size_t head = (size_t)slot[m] * nkv + (s - nh - nkv);
            __half* vh = att_vt + (head * 2 * kHdim) * n_ctx64 + p;
            __half* vl = vh + (size_t)kHdim * n_ctx64;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const __half ah = __float2half_rn(a[j]), bh = __float2half_rn(b[j]);
                vh[(size_t)(i0 + j) * n_ctx64] = ah;
                vl[(size_t)(i0 + j) * n_ctx64] = __float2half_rn(a[j] - __half2float(ah));
                vh[(size_t)(i0 + 32 + j) * n_ctx64] = bh;
                vl[(size_t)(i0 + 32 + j) * n_ctx64] = __float2half_rn(b[j] - __half2float(bh));
            }
        }
    }
};

// x[m][n0..n0+31] += v.
struct EpiResidual {
    float* x;
    int H;
    __device__ __forceinline__ void store(int m, int n0, const float (&v)[32]) const {
        float4* d = reinterpret_cast<float4*>(x + (size_t)m * H + n0);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float4 t = d[j];
            t.x += v[4 * j];
            t.y += v[4 * j + 1];
            t.z += v[4 * j + 2];
            t.w += v[4 * j + 3];
            d[j] = t;
        }
    }
};

// Columns (2j, 2j+1) hold (gate j, up j): m[j] = SiLU(gate) * up, in f16.
struct EpiSwiGLU {
    __half* out;
    int I;
    __device__ __forceinline__ void store(int m, int n0, const float (&v)[32]) const {
        uint32_t h[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const __half2 t = __floats2half2_rn(silu_f(v[4 * j]) * v[4 * j + 1], silu_f(v[4 * j + 2]) * v[4 * j + 3]);
            h[j] = *reinterpret_cast<const uint32_t*>(&t);
        }
        uint4* d = reinterpret_cast<uint4*>(out + (size_t)m * I + (n0 >> 1));
        d[0] = make_uint4(h[0], h[1], h[2], h[3]);
        d[1] = make_uint4(h[4], h[5], h[6], h[7]);
    }
};

constexpr int kBnQKV = 128, kBnO = 224, kBnGU = 256, kBnDown = 224;
// Which products take their activation operand as an f16 hi + lo pair (see
// tc_gemm.cuh): the normed rows feeding QKV and gate/up and the attention
// output feeding o_proj.  With a single f16 rounding of those three operands
// the 24-layer residual stream drifts to a final-norm relative L2 of about
// 1.2e-3 on the 0.5B shape; the SwiGLU output alone (down's operand)
// contributes about 4e-4 and stays single.
constexpr bool kSplitQKV = true, kSplitO = true, kSplitGU = true, kSplitDown = false;

template <int BN, bool SPLIT, class Epi>
cudaError_t launch(const Ctx& c, const CUtensorMap& a, const CUtensorMap& a2, const CUtensorMap& b, int M, int N,
                   int K, const Epi& e, cudaStream_t st) {
    const int tiles = ((M + tcg::kBM - 1) / tcg::kBM) * ((N + BN - 1) / BN);
    const int grid = tiles < c.n_sm ? tiles : c.n_sm;
    return launch_pdl(tcg::k_gemm_tc<BN, SPLIT, Epi>, dim3(grid), dim3(tcg::kThreads), tcg::GemmCfg<BN, SPLIT>::kSmem,
                      st, a, a2, b, M, N, K, e, c.err);
}

template <int BN, bool SPLIT, class Epi>
cudaError_t allow_smem() {
    return cudaFuncSetAttribute(tcg::k_gemm_tc<BN, SPLIT, Epi>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)tcg::GemmCfg<BN, SPLIT>::kSmem);
}

}  // namespace

int tc_setup(Ctx& c, std::string& why) {
    const qwen2_config& g = c.cfg;
    const int H = g.hidden, I = g.intermediate, nq = g.n_head * kHdim, R = c.max_rows;
    TcState& t = c.tc;
    if (!tensor_map_encoder()) {
        why = "the driver has no cuTensorMapEncodeTiled";
        return QWEN2_E_CUDA;
    }
    bool ok = encode_kmajor_f16(&t.a_xn, c.ws.xn_h, R, H, tcg::kBM) &&
              encode_kmajor_f16(&t.a_xn_lo, c.ws.xn_l, R, H, tcg::kBM) &&
              encode_kmajor_f16(&t.a_o, c.ws.o_h, R, nq, tcg::kBM) &&
              encode_kmajor_f16(&t.a_o_lo, c.ws.o_l, R, nq, tcg::kBM) &&
              encode_kmajor_f16(&t.a_mlp, c.ws.mlp_h, R, I, tcg::kBM);
    // Attention operands: k rows [slot][kv head][position] of 64 dims, and
    // v^T rows [slot][kv head][hi / lo][dim] of n_ctx64 keys; 64 x 64 boxes.
    const uint64_t heads = (uint64_t)g.max_seqs * g.n_kv_head, n64 = (uint64_t)att_ctx64(g.n_ctx);
    ok = ok && encode_kmajor_f16(&t.att_k, c.ws.att_k, heads * n64, kHdim, 64) &&
         encode_kmajor_f16(&t.att_vt, c.ws.att_vt, heads * 2 * kHdim, n64, 64);
    t.layers.resize(g.n_layer);
    for (int l = 0; l < g.n_layer && ok; ++l) {
        const DevLayer& L = c.layers[l];
        TcLayerMaps& m = t.layers[l];
        ok = encode_kmajor_f16(&m.wqkv, L.wqkv.w, c.nqkv, H, kBnQKV) &&
             encode_kmajor_f16(&m.wo, L.wo.w, H, nq, kBnO) && encode_kmajor_f16(&m.wgu, L.wgu.w, 2 * I, H, kBnGU) &&
             encode_kmajor_f16(&m.wd, L.wd.w, H, I, kBnDown);
    }
    if (!ok) {
        why = "TMA tensor-map encoding failed";
        return QWEN2_E_CUDA;
    }
    if (allow_smem<kBnQKV, kSplitQKV, EpiQKV>() != cudaSuccess ||
        allow_smem<kBnO, kSplitO, EpiResidual>() != cudaSuccess ||
        allow_smem<kBnGU, kSplitGU, EpiSwiGLU>() != cudaSuccess ||
        allow_smem<kBnDown, kSplitDown, EpiResidual>() != cudaSuccess) {
        cudaGetLastError();
        why = "cannot raise the tensor-core GEMM shared-memory limit";
        return QWEN2_E_CUDA;
    }
    if (lm_head_tc_setup(c) != cudaSuccess) {
        cudaGetLastError();
        why = "cannot raise the tensor-core LM head's shared-memory limit";
        return QWEN2_E_CUDA;
    }
    t.ok = true;
    return QWEN2_OK;
}

cudaError_t tc_gemm_qkv(const Ctx& c, int layer, int M, const PrefillEpi& p, cudaStream_t st) {
    EpiQKV e{p.nh, p.nkv, p.n_ctx, p.L, p.layer, p.q, p.kv, p.rope, p.bias, p.pos, p.slot, p.err,
             c.ws.att_k, c.ws.att_vt, att_ctx64(p.n_ctx)};
    return launch<kBnQKV, kSplitQKV>(c, c.tc.a_xn, c.tc.a_xn_lo, c.tc.layers[layer].wqkv, M, c.nqkv, c.cfg.hidden,
                                     e, st);
}

cudaError_t tc_gemm_o(const Ctx& c, int layer, int M, float* x, cudaStream_t st) {
    EpiResidual e{x, c.cfg.hidden};
    return launch<kBnO, kSplitO>(c, c.tc.a_o, c.tc.a_o_lo, c.tc.layers[layer].wo, M, c.cfg.hidden,
                                 c.cfg.n_head * kHdim, e, st);
}

cudaError_t tc_gemm_gu(const Ctx& c, int layer, int M, cudaStream_t st) {
    EpiSwiGLU e{c.ws.mlp_h, c.cfg.intermediate};
    return launch<kBnGU, kSplitGU>(c, c.tc.a_xn, c.tc.a_xn_lo, c.tc.layers[layer].wgu, M, 2 * c.cfg.intermediate,
                                   c.cfg.hidden, e, st);
}

cudaError_t tc_gemm_down(const Ctx& c, int layer, int M, float* x, cudaStream_t st) {
    EpiResidual e{x, c.cfg.hidden};
    return launch<kBnDown, kSplitDown>(c, c.tc.a_mlp, c.tc.a_mlp, c.tc.layers[layer].wd, M, c.cfg.hidden,
                                       c.cfg.intermediate, e, st);
}

}  // namespace qwen2
