// Shared declarations of the prefill kernels (CUDA-core and tensor-core).
#pragma once

#include "ctx.h"

namespace qwen2 {

enum EpiKind : int { kEpiQKV = 0, kEpiResidual = 1, kEpiSwiGLU = 2, kEpiLogits = 3 };

// What a GEMM epilogue does with output element (m, n) of a layer's product.
//  kEpiQKV:      n indexes the packed Q/K/V rows; pairs (n, n+1) get the
//                bias, the NeoX rotation (q, k) and go to q / the KV cache
//  kEpiResidual: x[m][n] += value
//  kEpiSwiGLU:   pairs (gate j, up j) -> mlp[m][j] = SiLU(gate) * up
//  kEpiLogits:   lg[m][n] = value (the LM head of the kept rows)
// Optional f16 copies (q_h, mlp_h) feed the tensor-core path.
struct PrefillEpi {
    int kind;
    int H, I, nh, nkv, n_ctx, L, layer;
    int hd;  // head_dim (the QKV epilogue's head slots and RoPE pairs)
    float* lg;  // kEpiLogits: logits [rows][lg_ld]
    int lg_ld;
    float* x;
    float* q;
    __half* q_h;
    float* mlp;
    __half* mlp_h;
    float* kv;
    const float2* rope;
    const float* bias;
    const int* pos;
    const int* slot;
    int* err;
};

struct PrefillAttnArgs {
    const float* q;         // [rows][nh*hd] rotated queries
    float* o;               // [rows][nh*hd] head outputs (f32), or
    __half* o_h;            //   f16 hi / lo pairs when o_h is not null
    __half* o_l;            //   (tensor-core operands: o = o_h + o_l)
    const float* kv;
    const int* pos;
    const int* slot;
    const int* blk_row0;    // query blocks: first row and row count, one sequence each
    const int* blk_nrows;
    int nh, nkv, n_ctx, L;
};

// Device copies of the per-call row plan (built on the host).
struct PrefillPlan {
    const int* blk_row0;
    const int* blk_nrows;
    int n_blk;
    const int* kblk_row0;   // blocks over the kept rows (after the tail cut)
    const int* kblk_nrows;
    int n_kblk;
    const int* seq_slot;    // per sequence of the call: its slot, and the end (exclusive)
    const int* seq_conv;    //   of the positions whose attention operands come from the
                            //   cache: those before the call's first row when its rows are
                            //   consecutive positions (the QKV epilogue writes the rest),
                            //   else every position up to the largest
    int n_seq;
    int conv_tiles;         // max over the sequences of ceil(seq_conv / 64); 0: nothing to convert
};

// Positions of the attention operand buffers rounded up to whole 64-key tiles.
inline int att_ctx64(int n_ctx) { return (n_ctx + 63) & ~63; }

constexpr int kPrefillQB = 16;   // query rows per attention block

// ---- tensor-core path (prefill_tc.cu) --------------------------------------
// Encodes the TMA tensor maps and raises the GEMM shared-memory limits;
// needs ws.xn_h / o_h / mlp_h and the packed weights.
int tc_setup(Ctx& c, std::string& why);
// The four GEMMs of `layer` over the first M workspace rows.
cudaError_t tc_gemm_qkv(const Ctx& c, int layer, int M, const PrefillEpi& e, cudaStream_t st);
cudaError_t tc_gemm_o(const Ctx& c, int layer, int M, float* x, cudaStream_t st);
cudaError_t tc_gemm_gu(const Ctx& c, int layer, int M, cudaStream_t st);
cudaError_t tc_gemm_down(const Ctx& c, int layer, int M, float* x, cudaStream_t st);

// Causal GQA attention of the tensor-core path on tcgen05 MMAs into tensor
// memory (prefill_attn_tc.cu): writes a.o_h / a.o_l; grid (nkv, n_blk) over
// the 16-row query blocks; head_dim 64, at most 8 query heads per kv head.
// The f16 operand buffers it reads by TMA (Workspace::att_k / att_vt) hold
// the call's own keys (the QKV epilogue writes them); it first converts the
// positions below seq_conv from the f32 cache (keys an earlier call stored).
cudaError_t enqueue_attn_prefill_tc(const Ctx& c, const PrefillAttnArgs& a, const PrefillPlan& plan, int layer,
                                    cudaStream_t st);
cudaError_t prefill_attn_tc_set_smem();

// Final norm + LM head + argmax of the kept rows on tcgen05 (lm_head_tc.cu),
// up to 8 rows per launch; f16 LM head rows, hidden a multiple of 64.
cudaError_t lm_head_tc_setup(Ctx& c);
bool lm_head_tc_supported(const Ctx& c);
cudaError_t enqueue_lm_head_tc(Ctx& c, const float* xin, int B, float* logits, int* ids, cudaStream_t st);

cudaError_t enqueue_prefill(Ctx& c, int rows, int n_keep, const PrefillPlan& plan, float* logits_dev,
                            int* ids_dev, cudaStream_t st);
cudaError_t prefill_set_smem_limits();

}  // namespace qwen2
