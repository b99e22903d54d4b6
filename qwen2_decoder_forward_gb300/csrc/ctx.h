// Internal state of a libqwen2 context and the launchers the C ABI drives.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <map>
#include <string>
#include <vector>

#include "../../include/qwen2.h"

namespace qwen2 {

// One linear weight in device memory.  f16: `w` is [rows][k] halves.
// Q8_0: `q` is int8 [rows][k] and `d` the f16 scales [rows][k/32].
// Q4_0 (q4 set): `q` holds [rows][k/2] bytes of 4-bit codes (element 2j in
// the low nibble of byte j, code = value / scale + 8) and `d` the scales.
struct DevMat {
    const __half* w = nullptr;
    const int8_t* q = nullptr;
    const __half* d = nullptr;
    int rows = 0, k = 0;
    bool q4 = false;
};

// The block-quantised weight formats (Q8_0, Q4_0) run the batched product
// path; f16 runs the row-dot GEMV kernels and the persistent kernel.
inline bool block_quantised(const qwen2_config& g) { return g.weight_format != QWEN2_WEIGHTS_F16; }

// Packed layer.  Row orders (chosen so that an output pair an epilogue needs
// sits on adjacent rows):
//  wqkv: [(nh + 2 nkv) hd][H]; head slot s (q heads, then k, then v) holds
//        rows (s*hd + 2i, s*hd + 2i + 1) = original rows (s*hd + i,
//        s*hd + i + hd/2): the two halves a NeoX rotation pairs;
//  wgu:  [2I][H]; rows (2j, 2j+1) = (gate_proj row j, up_proj row j);
//  wo [H][nh hd] and wd [H][I] keep the HF order.
struct DevLayer {
    DevMat wqkv, wo, wgu, wd;
    const float* bqkv = nullptr;       // permuted like wqkv's rows
    const float* attn_norm = nullptr;
    const float* ffn_norm = nullptr;
};

// Columns of k per CTA of the Q8_0 down product (split-k chunk).
constexpr int kQ8DownKc = 448;
// Rows one quantised-activation prefill may send to the LM head.
constexpr int kQ8aMaxOut = 64;

struct Workspace {
    float* x = nullptr;        // [rows][H] residual stream
    float* xn = nullptr;       // [rows][max(H, I)] normed rows (unfused / prefill)
    float* q = nullptr;        // [rows][nh*hd] rotated queries
    float* o = nullptr;        // [rows][nh*hd] attention output (premix)
    float* mlp = nullptr;      // [rows][I] SiLU(gate) * up
    float* raw = nullptr;      // [max_seqs][max(NQKV, 2I)] unfused raw products
    float* att_part = nullptr; // decode split-K partials [max_seqs][nh][chunks][2+hd]
    int* att_count = nullptr;  // decode split-K arrival counters [max_seqs][nkv]
    float* am_val = nullptr;   // LM-head per-block argmax values [blocks][8]
    int* am_idx = nullptr;     // LM-head per-block argmax indices [blocks][8]
    int* am_count = nullptr;   // LM-head arrival counter
    float* lm_val = nullptr;   // Q8_0 LM-head per-CTA argmax values [ceil(V/256)][32]
    int* lm_idx = nullptr;     // Q8_0 LM-head per-CTA argmax indices
    __half* q8_ah = nullptr;   // Q8_0 product operand, f16 hi [32][H] (normed rows, attention output)
    __half* q8_al = nullptr;   //   and lo
    __half* q8_mh = nullptr;   // SiLU(gate) * up as f16 hi [32][I]
    __half* q8_ml = nullptr;   //   and lo
    float* q8_part = nullptr;  // down-product partials [ceil(I/kQ8DownKc)][32][H]
    int* q8_cnt = nullptr;     // down-product arrival counters, one per 64 output rows
    float* hidden = nullptr;   // [rows_out][H] final_norm_output
    float* logits = nullptr;   // [max_seqs][V] decode logits staging
    int* rows_tok = nullptr;   // prefill: per-row token
    int* rows_pos = nullptr;   // prefill: per-row position
    int* rows_slot = nullptr;  // prefill: per-row sequence slot
    int* keep_rows = nullptr;  // prefill: indices of the rows kept for the LM head
    int* keep_pos = nullptr;   // prefill: positions of the kept rows
    int* keep_slot = nullptr;  // prefill: slots of the kept rows
    int* blk = nullptr;        // prefill: attention query-block plan (4 arrays)
    float* x2 = nullptr;       // [rows][H] kept rows of the residual (tail cut)
    float* q2 = nullptr;       // [rows][nh*hd] kept rows of q (tail cut)
    __half* xn_h = nullptr;    // [rows][H] f16 normed rows (tensor prefill operand), and
    __half* xn_l = nullptr;    //   their f16 remainders x - f32(xn_h)
    __half* o_h = nullptr;     // [rows][nh*hd] f16 attention output (tensor prefill operand), and
    __half* o_l = nullptr;     //   its f16 remainders
    __half* mlp_h = nullptr;   // [rows][I] f16 SiLU(gate) * up (tensor prefill operand)
    __half* att_k = nullptr;   // tensor prefill attention operands of one layer, per slot and kv
    __half* att_vt = nullptr;  //   head: k as f16 [n_ctx64][hd], v transposed as f16 hi / lo [2][hd][n_ctx64]
    int* ids = nullptr;        // [rows] prefill ids staging
    int8_t* aq = nullptr;      // quantised prefill: activation codes [rows][max(H, I, nh*hd)]
    __half* ad = nullptr;      //   and their block scales [rows][max(H, I, nh*hd) / 32]
    float* q8a_lg = nullptr;   //   and the kept rows' logits [kQ8aMaxOut][V]
    float* out_logits = nullptr; // [rows_out][V] staging when the caller's logits are host memory
    size_t out_logits_rows = 0;
    int att_max_chunks = 0;
    int am_blocks = 0;
};

// Static device state the decode CUDA graphs read (their pointers are baked
// into the graphs).
constexpr int kIdsHist = 512;
struct DecodeState {
    int* tok = nullptr;      // [max_seqs] token fed this step
    int* pos = nullptr;      // [max_seqs] position of this step
    int* slot = nullptr;     // [max_seqs] KV slot (sequence id)
    int* step = nullptr;     // [1] index of the step within a decode_steps run
    int* ids_hist = nullptr; // [kIdsHist][max_seqs] ids per step
    int* stop_ids = nullptr;  // [kMaxStopIds] stop ids of a decode_steps_stop run
    int* stop_done = nullptr; // [max_seqs] 1 once the sequence generated a stop id
    int* n_gen = nullptr;     // [max_seqs] ids kept so far, the stop id included
};
constexpr int kMaxStopIds = 8;

// Per-layer weight pointers the persistent decode kernel reads.
struct PersistLayer {
    const __half *wqkv, *wo, *wgu, *wd;
    const float *bqkv, *attn_norm, *ffn_norm;
};

// State of the persistent batch-1 decode kernel.
struct PersistState {
    bool ok = false;                  // the kernel fits this shape and device
    const void* kernel = nullptr;     // the instantiation for this shape
    int grid = 0;                     // one CTA per SM
    size_t smem = 0;                  // dynamic shared memory per CTA
    int rows_h = 0, rows_i = 0;       // weight rows per ring stage (K = H, K = I)
    int act_floats = 0;               // activation / attention scratch floats
    int max_chunks = 0;               // attention chunks of 64 keys at n_ctx
    int merge_group = 0;              // chunks merged per shared-memory pass
    PersistLayer* layers = nullptr;   // [n_layer] on the device
    unsigned long long* pk = nullptr; // activation packets (value + epoch)
    unsigned* epoch = nullptr;        // completed launches (reset only after a device guard)
    unsigned long long* cnt = nullptr; // per-phase arrival counters
    size_t pk_bytes = 0, cnt_bytes = 0;
    long long* prof = nullptr;        // per-phase timestamps (QWEN2_FLAG_PROFILE)
    int prof_marks = 0;
    int test_stall = 0;               // the next launch waits on a counter nothing arrives at
    unsigned long long test_wait_ns = 0;  // and gives up after this many ns
    std::string why_not;              // why the kernel is unavailable, if it is
};

// TMA tensor maps of the tensor-core prefill GEMMs (encoded once; every
// pointer they hold is fixed for the context's lifetime).
struct TcLayerMaps {
    CUtensorMap wqkv, wo, wgu, wd;
};
// Every buffer dev_alloc makes has kCanaryBytes of kCanaryByte on each side.
constexpr size_t kCanaryBytes = 256;
constexpr unsigned char kCanaryByte = 0xA5;
struct CanaryRegion {
    unsigned char* user;  // first byte of the buffer proper
    size_t bytes;
};

struct TcState {
    bool ok = false;
    CUtensorMap a_xn, a_xn_lo, a_o, a_o_lo, a_mlp;   // activation operands [max_rows][K]
    CUtensorMap att_k, att_vt;                        // attention operands (Workspace::att_k / att_vt)
    CUtensorMap lm_e;                                 // LM head rows [V][H] in 128 x 64 boxes
    bool lm_ok = false;                               // lm_e encoded (the tensor-core LM head serves)
    std::vector<TcLayerMaps> layers;
};

struct Ctx {
    qwen2_config cfg{};
    int device = 0;
    int n_sm = 0;
    int nqkv = 0;                 // (nh + 2 nkv) * hd
    void* wblob = nullptr;        // all packed weights, one allocation
    size_t wbytes = 0;
    std::vector<DevLayer> layers;
    DevMat embed;                 // [V][H] token embedding
    DevMat lm_head;               // [V][H] readout: `embed` itself when tied, else its own matrix
    const float* final_norm = nullptr;
    float* kv = nullptr;          // [max_seqs][L][2][nkv][n_ctx][hd]
    size_t kv_floats = 0;
    CUtensorMap kvmap;            // kv as a [rows][64] f32 matrix, 32 x 64 boxes, 128-byte swizzle
    bool kvmap_ok = false;        // the map encoded (batched decode attention uses it)
    float2* rope = nullptr;       // [n_ctx][hd/2] (cos, sin), from double on the host
    int* err = nullptr;           // device guard word
    Workspace ws;
    DecodeState ds;
    PersistState pers;
    TcState tc;
    int max_rows = 0;             // rows the prefill workspace holds
    int max_rows_q8 = 32;         // rows one Q8_0 batched product carries
    int last_rows_out = 0;        // rows of the last call's final_norm_output
    cudaStream_t cap_stream = nullptr;
    std::map<int, cudaGraphExec_t> graphs;   // key: B | (want_logits << 16)
    std::vector<void*> allocs;    // device buffers freed at destroy
    std::vector<CanaryRegion> canaries;  // the same buffers' user regions, between guard words
    std::string last_error;
};

// ---- decode.cu ---------------------------------------------------------------
// Enqueue one decode step for the first B slots of DecodeState on `st`
// (B <= 8).  Logits go to ws.logits when want_logits.
cudaError_t enqueue_decode_step(Ctx& c, int B, bool want_logits, cudaStream_t st);
// Stop tokens over the first n_steps rows of the id history (one chunk of a
// decode_steps_stop run): ids after a sequence's first stop id become -1,
// and stop_done / n_gen carry over from the previous chunk unless first
// (n_stop may be 0: nothing is masked and n_gen counts every step).
cudaError_t enqueue_stop_mask(Ctx& c, int n_seq, int n_steps, int n_stop, bool first, cudaStream_t st);

// LM head + argmax over `B` rows of `xin` (f32 [B][H]); writes the hidden
// rows (ws.hidden), optional logits [B][V] and ids [B].  `decode` selects the
// decode-state update (next token, position advance, ids history; B <= 8).
cudaError_t enqueue_lm_head(Ctx& c, const float* xin, int B, float* logits, int* ids, bool decode,
                            cudaStream_t st);
cudaError_t decode_set_smem_limits(int max_bytes);
// o_proj + residual, RMSNorm + gate/up + SwiGLU and down + residual of
// `layer` on `rows` rows of x (f32 [rows][H]) with attention output o (f32
// [rows][nh*hd]), through the decode GEMV kernels (groups of 8 rows).
cudaError_t enqueue_rows_o_ffn(Ctx& c, int layer, float* x, const float* o, int rows, cudaStream_t st);

// ---- pack.cu -------------------------------------------------------------------
int pack_weights(Ctx& c, const qwen2_weights* w, std::string& err);
void quantize_q8_0_host(const uint16_t* w, int64_t rows, int64_t k, int8_t* q, uint16_t* d);
void quantize_q4_0_host(const uint16_t* w, int64_t rows, int64_t k, uint8_t* packed, uint16_t* d);
int build_rope_table(Ctx& c, std::string& err);

// Records the message of a failed call made without a context; read back
// with qwen2_last_error(NULL).
void set_thread_error(const std::string& msg);

}  // namespace qwen2
