// The C ABI of libqwen2: argument validation, context set-up (weight
// packing, KV cache, workspace, RoPE table), decode CUDA graphs, and the
// prefill / decode entry points declared in include/qwen2.h.
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <set>
#include <string>
#include <vector>

#include "ctx.h"
#include "persistent.h"
#include "prefill.h"
#include "tmap.h"

using namespace qwen2;

namespace qwen2 {
// decode.cu: write `code` into the device guard word from a one-thread
// kernel (the qwen2_test_raise_guard hook).
cudaError_t enqueue_raise_guard(Ctx& c, int code, cudaStream_t st);
}  // namespace qwen2

struct qwen2_ctx {
    Ctx c;
};

namespace {

thread_local std::string g_create_error;

int fail(Ctx* c, int code, const std::string& msg) {
    if (c) c->last_error = msg;
    else g_create_error = msg;
    return code;
}

int cuda_fail(Ctx* c, cudaError_t e, const char* what) {
    return fail(c, QWEN2_E_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

}  // namespace

// Message of a failed call that has no context (qwen2_last_error(NULL)).
void qwen2::set_thread_error(const std::string& msg) { g_create_error = msg; }

namespace {

#define Q2_CHECK(c, call)                                  \
    do {                                                   \
        cudaError_t e_ = (call);                           \
        if (e_ != cudaSuccess) return cuda_fail(c, e_, #call); \
    } while (0)

bool is_device_ptr(const void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

template <class T>
int dev_alloc(Ctx& c, T** p, size_t count, bool zero = true) {
    // The buffer sits between two guard regions of kCanaryBytes filled with
    // kCanaryByte; qwen2_check_canaries reads them back.
    void* v = nullptr;
    const size_t bytes = std::max<size_t>(count, 1) * sizeof(T);
    if (cudaMalloc(&v, bytes + 2 * kCanaryBytes) != cudaSuccess) {
        cudaGetLastError();
        return QWEN2_E_OOM;
    }
    unsigned char* user = static_cast<unsigned char*>(v) + kCanaryBytes;
    if (cudaMemset(v, kCanaryByte, kCanaryBytes) != cudaSuccess ||
        cudaMemset(user + bytes, kCanaryByte, kCanaryBytes) != cudaSuccess ||
        (zero && cudaMemset(user, 0, bytes) != cudaSuccess)) {
        cudaFree(v);
        return QWEN2_E_CUDA;
    }
    c.allocs.push_back(v);
    c.canaries.push_back({user, bytes});
    *p = reinterpret_cast<T*>(user);
    return QWEN2_OK;
}

int validate_config(const qwen2_config* g, std::string& msg) {
    if (g->n_layer < 1 || g->hidden < 1 || g->n_head < 1 || g->n_kv_head < 1 || g->head_dim < 1 ||
        g->intermediate < 1 || g->vocab < 2 || g->n_ctx < 1 || g->max_seqs < 1 || g->max_tokens < 1) {
        msg = "config sizes must be positive";
        return QWEN2_E_ARG;
    }
    if (!(g->rms_eps >= 0.f) || !(g->rope_theta > 0.0)) {
        msg = "rms_eps must be >= 0 and rope_theta > 0";
        return QWEN2_E_ARG;
    }
    if (g->head_dim != 64 && g->head_dim != 128) {
        msg = "head_dim " + std::to_string(g->head_dim) + " is not supported (64 or 128)";
        return QWEN2_E_UNSUPPORTED;
    }
    if (g->head_dim != 64 && g->prefill_mode == QWEN2_PREFILL_TENSOR) {
        msg = "the tensor-core prefill is built for head_dim 64; use QWEN2_PREFILL_F32";
        return QWEN2_E_UNSUPPORTED;
    }
    if (g->hidden != g->n_head * g->head_dim) {
        msg = "hidden must equal n_head * head_dim";
        return QWEN2_E_UNSUPPORTED;
    }
    if (g->hidden % 128 || g->intermediate % 128) {
        msg = "hidden and intermediate must be multiples of 128";
        return QWEN2_E_UNSUPPORTED;
    }
    if (g->n_head % g->n_kv_head || g->n_head / g->n_kv_head > 8) {
        msg = "n_head must be a multiple of n_kv_head with at most 8 query heads per kv head";
        return QWEN2_E_UNSUPPORTED;
    }
    if (g->weight_format != QWEN2_WEIGHTS_F16 && g->weight_format != QWEN2_WEIGHTS_Q8_0 &&
        g->weight_format != QWEN2_WEIGHTS_Q4_0) {
        msg = "weight_format " + std::to_string(g->weight_format) + " is not supported by this build";
        return QWEN2_E_UNSUPPORTED;
    }
    if (g->prefill_mode == QWEN2_PREFILL_Q8_ACT && g->weight_format != QWEN2_WEIGHTS_Q8_0) {
        msg = "QWEN2_PREFILL_Q8_ACT needs Q8_0 weights";
        return QWEN2_E_UNSUPPORTED;
    }
    if (block_quantised(*g) && g->prefill_mode == QWEN2_PREFILL_TENSOR) {
        msg = "Q8_0 and Q4_0 weights prefill on the f32 path (QWEN2_PREFILL_F32, or QWEN2_PREFILL_Q8_ACT)";
        return QWEN2_E_UNSUPPORTED;
    }
    if (block_quantised(*g) && g->hidden > 1024) {
        msg = "Q8_0 and Q4_0 weights need hidden <= 1024 (the batched product stages one activation chunk)";
        return QWEN2_E_UNSUPPORTED;
    }
    if (g->prefill_mode != QWEN2_PREFILL_F32 && g->prefill_mode != QWEN2_PREFILL_TENSOR &&
        g->prefill_mode != QWEN2_PREFILL_Q8_ACT) {
        msg = "prefill_mode " + std::to_string(g->prefill_mode) + " is not supported by this build";
        return QWEN2_E_UNSUPPORTED;
    }
    if ((int64_t)g->vocab * g->hidden > INT32_MAX * 8LL) {
        msg = "vocab * hidden too large";
        return QWEN2_E_UNSUPPORTED;
    }
    return QWEN2_OK;
}

int validate_weights(const qwen2_config* g, const qwen2_weights* w, std::string& msg) {
    if (!w->embed || !w->final_norm || !w->layers) {
        msg = "null weight pointer";
        return QWEN2_E_ARG;
    }
    for (int l = 0; l < g->n_layer; ++l) {
        const qwen2_layer_weights& L = w->layers[l];
        if (!L.wq || !L.wk || !L.wv || !L.wo || !L.wg || !L.wu || !L.wd || !L.bq || !L.bk || !L.bv ||
            !L.attn_norm || !L.ffn_norm) {
            msg = "null weight pointer in layer " + std::to_string(l);
            return QWEN2_E_ARG;
        }
    }
    return QWEN2_OK;
}

int setup_workspace(Ctx& c) {
    const qwen2_config& g = c.cfg;
    const int H = g.hidden, I = g.intermediate, nq = g.n_head * g.head_dim;
    const int R = std::max(g.max_tokens, g.max_seqs);
    const int S = g.max_seqs;
    c.max_rows = R;
    Workspace& w = c.ws;
    w.att_max_chunks = (g.n_ctx + 63) / 64;
    w.am_blocks = c.n_sm * 2;
    int r = QWEN2_OK;
    auto A = [&](auto** p, size_t n) {
        if (r == QWEN2_OK) r = dev_alloc(c, p, n);
    };
    A(&w.x, (size_t)R * H);
    A(&w.xn, (size_t)R * H);
    A(&w.q, (size_t)R * nq);
    A(&w.o, (size_t)R * nq);
    A(&w.mlp, (size_t)R * I);
    A(&w.raw, (size_t)S * std::max(c.nqkv, 2 * I));
    A(&w.att_part, (size_t)S * g.n_head * w.att_max_chunks * (g.head_dim + 2));
    A(&w.att_count, (size_t)S * g.n_kv_head);
    A(&w.am_val, (size_t)w.am_blocks * 8);
    A(&w.am_idx, (size_t)w.am_blocks * 8);
    A(&w.am_count, 1);
    A(&w.hidden, (size_t)R * H);
    A(&w.logits, (size_t)S * g.vocab);
    A(&w.rows_tok, R);
    A(&w.rows_pos, R);
    A(&w.rows_slot, R);
    A(&w.keep_rows, R);
    A(&w.keep_pos, R);
    A(&w.keep_slot, R);
    A(&w.blk, (size_t)6 * R);
    A(&w.x2, (size_t)R * H);
    A(&w.q2, (size_t)R * nq);
    A(&w.ids, R);
    if (block_quantised(g)) {
        const size_t blocks = ((size_t)g.vocab + 255) / 256;
        const size_t rq = (size_t)c.max_rows_q8;
        A(&w.lm_val, blocks * 32);
        A(&w.lm_idx, blocks * 32);
        A(&w.q8_ah, rq * std::max(H, nq));
        A(&w.q8_al, rq * std::max(H, nq));
        A(&w.q8_mh, rq * I);
        A(&w.q8_ml, rq * I);
        A(&w.q8_part, (size_t)((I + kQ8DownKc - 1) / kQ8DownKc) * rq * H);
        A(&w.q8_cnt, (size_t)(H + 63) / 64);
    }
    if (g.prefill_mode == QWEN2_PREFILL_Q8_ACT) {
        const size_t wmax = std::max({(size_t)H, (size_t)I, (size_t)nq});
        A(&w.aq, (size_t)R * wmax);
        A(&w.ad, (size_t)R * wmax / 32);
        A(&w.q8a_lg, (size_t)kQ8aMaxOut * g.vocab);
    }
    if (g.prefill_mode == QWEN2_PREFILL_TENSOR) {
        A(&w.xn_h, (size_t)R * H);
        A(&w.xn_l, (size_t)R * H);
        A(&w.o_h, (size_t)R * nq);
        A(&w.o_l, (size_t)R * nq);
        A(&w.mlp_h, (size_t)R * I);
        const size_t heads = (size_t)S * g.n_kv_head, n64 = (size_t)att_ctx64(g.n_ctx);
        A(&w.att_k, heads * n64 * g.head_dim);
        A(&w.att_vt, heads * 2 * g.head_dim * n64);
    }
    A(&c.ds.tok, S);
    A(&c.ds.pos, S);
    A(&c.ds.slot, S);
    A(&c.ds.step, 1);
    A(&c.ds.ids_hist, (size_t)kIdsHist * S);
    A(&c.ds.stop_ids, kMaxStopIds);
    A(&c.ds.stop_done, S);
    A(&c.ds.n_gen, S);
    A(&c.err, 1);
    return r;
}

// Sequence ids distinct and in range.
int check_seq_ids(Ctx& c, int n_seq, const int32_t* seq_ids) {
    std::set<int> seen;
    for (int i = 0; i < n_seq; ++i) {
        if (seq_ids[i] < 0 || seq_ids[i] >= c.cfg.max_seqs)
            return fail(&c, QWEN2_E_ARG, "sequence id " + std::to_string(seq_ids[i]) + " outside [0, max_seqs)");
        if (!seen.insert(seq_ids[i]).second)
            return fail(&c, QWEN2_E_ARG, "sequence id " + std::to_string(seq_ids[i]) + " repeated");
    }
    return QWEN2_OK;
}

int check_tokens(Ctx& c, int n, const int32_t* tokens) {
    for (int i = 0; i < n; ++i)
        if (tokens[i] < 0 || tokens[i] >= c.cfg.vocab)
            return fail(&c, QWEN2_E_ARG, "token " + std::to_string(tokens[i]) + " outside [0, vocab)");
    return QWEN2_OK;
}

int check_positions(Ctx& c, int n, const int32_t* pos, int extra) {
    for (int i = 0; i < n; ++i)
        if (pos[i] < 0 || (int64_t)pos[i] + extra > c.cfg.n_ctx - 1)
            return fail(&c, QWEN2_E_POS, "position " + std::to_string(pos[i]) +
                                             (extra ? " + " + std::to_string(extra) : std::string()) +
                                             " outside [0, n_ctx=" + std::to_string(c.cfg.n_ctx) + ")");
    return QWEN2_OK;
}

bool use_persistent(const Ctx& c, int B) {
    const uint32_t off = QWEN2_FLAG_NO_MEGAKERNEL | QWEN2_FLAG_NO_FUSE_QKV | QWEN2_FLAG_NO_FUSE_FFN;
    return B == 1 && c.pers.ok && !(c.cfg.flags & off);
}

// Sequences one decode step can carry: 8 with f16 weights (the row-dot
// GEMV kernels), 32 with Q8_0 weights (the batched tensor-core product).
int max_decode_batch(const Ctx& c) { return block_quantised(c.cfg) ? 32 : 8; }

cudaError_t enqueue_step(Ctx& c, int B, bool want_logits, cudaStream_t st) {
    if (use_persistent(c, B)) return enqueue_decode_persistent(c, want_logits, st);
    return enqueue_decode_step(c, B, want_logits, st);
}

int get_graph(Ctx& c, int B, bool want_logits, cudaGraphExec_t* out) {
    const int key = B | (want_logits ? 1 << 16 : 0) | (use_persistent(c, B) ? 1 << 17 : 0);
    auto it = c.graphs.find(key);
    if (it != c.graphs.end()) {
        *out = it->second;
        return QWEN2_OK;
    }
    cudaGraph_t graph = nullptr;
    Q2_CHECK(&c, cudaStreamBeginCapture(c.cap_stream, cudaStreamCaptureModeThreadLocal));
    cudaError_t e = enqueue_step(c, B, want_logits, c.cap_stream);
    cudaError_t e2 = cudaStreamEndCapture(c.cap_stream, &graph);
    if (e != cudaSuccess) return cuda_fail(&c, e, "decode step capture");
    if (e2 != cudaSuccess) return cuda_fail(&c, e2, "cudaStreamEndCapture");
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return cuda_fail(&c, e, "cudaGraphInstantiate");
    c.graphs[key] = exec;
    *out = exec;
    return QWEN2_OK;
}

int run_decode_step(Ctx& c, int B, bool want_logits, cudaStream_t st) {
    // A launch armed by qwen2_test_stall_decode carries its own arguments:
    // it runs outside the cached graphs (whose arguments are baked in).
    if ((c.cfg.flags & QWEN2_FLAG_NO_GRAPH) || (c.pers.test_stall && use_persistent(c, B))) {
        cudaError_t e = enqueue_step(c, B, want_logits, st);
        if (e != cudaSuccess) return cuda_fail(&c, e, "decode step launch");
        return QWEN2_OK;
    }
    cudaGraphExec_t exec;
    int r = get_graph(c, B, want_logits, &exec);
    if (r != QWEN2_OK) return r;
    Q2_CHECK(&c, cudaGraphLaunch(exec, st));
    return QWEN2_OK;
}

}  // namespace

extern "C" {

int qwen2_create(const qwen2_config* cfg, const qwen2_weights* weights, qwen2_ctx** out) {
    g_create_error.clear();
    if (!out) return fail(nullptr, QWEN2_E_ARG, "out is NULL");
    *out = nullptr;
    if (!cfg || !weights) return fail(nullptr, QWEN2_E_ARG, "cfg or weights is NULL");
    std::string msg;
    int r = validate_config(cfg, msg);
    if (r == QWEN2_OK) r = validate_weights(cfg, weights, msg);
    if (r != QWEN2_OK) return fail(nullptr, r, msg);

    qwen2_ctx* h = new qwen2_ctx();
    Ctx& c = h->c;
    c.cfg = *cfg;
    auto bail = [&](int code, const std::string& m) {
        g_create_error = m;
        qwen2_destroy(h);
        return code;
    };
    if (cudaGetDevice(&c.device) != cudaSuccess) return bail(QWEN2_E_CUDA, "no CUDA device");
    if (cudaDeviceGetAttribute(&c.n_sm, cudaDevAttrMultiProcessorCount, c.device) != cudaSuccess)
        return bail(QWEN2_E_CUDA, "cannot read the SM count");
    r = pack_weights(c, weights, msg);
    if (r != QWEN2_OK) return bail(r, msg);
    r = build_rope_table(c, msg);
    if (r != QWEN2_OK) return bail(r, msg);
    c.kv_floats = (size_t)cfg->max_seqs * qwen2_kv_bytes_per_seq(cfg) / 4;
    r = dev_alloc(c, &c.kv, c.kv_floats);
    if (r != QWEN2_OK) return bail(r, "KV cache allocation of " + std::to_string(c.kv_floats * 4) + " bytes failed");
    r = setup_workspace(c);
    if (r != QWEN2_OK) return bail(r, "workspace allocation failed");
    // The cache as a [rows][64] f32 matrix for the batched decode attention's
    // tensor copies (64-position tiles); if it cannot be encoded, that
    // attention falls back to its split-k kernel.
    if (cfg->head_dim == 64)
        c.kvmap_ok = encode_rows64_f32(&c.kvmap, c.kv, (uint64_t)(c.kv_floats / 64), 64);
    int max_smem = 0;
    cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, c.device);
    if (decode_set_smem_limits(max_smem) != cudaSuccess || prefill_set_smem_limits() != cudaSuccess)
        return bail(QWEN2_E_CUDA, "cannot set kernel shared-memory limits");
    if (persistent_setup(c) != cudaSuccess) return bail(QWEN2_E_CUDA, "persistent decode kernel set-up failed");
    if (cfg->prefill_mode == QWEN2_PREFILL_TENSOR) {
        r = tc_setup(c, msg);
        if (r != QWEN2_OK) return bail(r, "tensor-core prefill set-up failed: " + msg);
    }
    if (cudaStreamCreateWithFlags(&c.cap_stream, cudaStreamNonBlocking) != cudaSuccess)
        return bail(QWEN2_E_CUDA, "cannot create the capture stream");
    if (cudaDeviceSynchronize() != cudaSuccess) return bail(QWEN2_E_CUDA, "set-up failed on the device");
    if (!c.pers.ok) c.last_error = "note: persistent decode kernel unavailable: " + c.pers.why_not;
    *out = h;
    return QWEN2_OK;
}

void qwen2_destroy(qwen2_ctx* h) {
    if (!h) return;
    Ctx& c = h->c;
    cudaDeviceSynchronize();
    for (auto& kv : c.graphs) cudaGraphExecDestroy(kv.second);
    if (c.cap_stream) cudaStreamDestroy(c.cap_stream);
    for (void* p : c.allocs) cudaFree(p);
    if (c.ws.out_logits) cudaFree(c.ws.out_logits);
    if (c.rope) cudaFree(c.rope);
    if (c.wblob) cudaFree(c.wblob);
    cudaGetLastError();
    delete h;
}

const char* qwen2_last_error(const qwen2_ctx* h) {
    return h ? h->c.last_error.c_str() : g_create_error.c_str();
}

int qwen2_kv_cache(qwen2_ctx* h, float** base, int64_t dims[6]) {
    if (!h || !base || !dims) return h ? fail(&h->c, QWEN2_E_ARG, "null argument") : QWEN2_E_ARG;
    const qwen2_config& g = h->c.cfg;
    *base = h->c.kv;
    dims[0] = g.max_seqs;
    dims[1] = g.n_layer;
    dims[2] = 2;
    dims[3] = g.n_kv_head;
    dims[4] = g.n_ctx;
    dims[5] = g.head_dim;
    return QWEN2_OK;
}

int qwen2_prefill(qwen2_ctx* h, int32_t n_seq, const int32_t* seq_ids, const int32_t* n_tokens,
                  const int32_t* tokens, const int32_t* positions, int32_t n_out, float* logits, int32_t* ids,
                  void* stream) {
    if (!h) return QWEN2_E_ARG;
    Ctx& c = h->c;
    c.last_error.clear();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (n_seq < 1 || n_seq > c.cfg.max_seqs) return fail(&c, QWEN2_E_ARG, "n_seq outside [1, max_seqs]");
    if (!seq_ids || !n_tokens || !tokens || !positions) return fail(&c, QWEN2_E_ARG, "null input pointer");
    if (n_out < 1) return fail(&c, QWEN2_E_ARG, "n_out must be >= 1");
    int r = check_seq_ids(c, n_seq, seq_ids);
    if (r) return r;
    int64_t total = 0;
    for (int s = 0; s < n_seq; ++s) {
        if (n_tokens[s] < n_out) return fail(&c, QWEN2_E_ARG, "a sequence has fewer than n_out tokens");
        total += n_tokens[s];
    }
    if (total > c.cfg.max_tokens) return fail(&c, QWEN2_E_ARG, "more rows than max_tokens");
    if (c.cfg.prefill_mode == QWEN2_PREFILL_Q8_ACT && (int64_t)n_seq * n_out > kQ8aMaxOut)
        return fail(&c, QWEN2_E_ARG, "QWEN2_PREFILL_Q8_ACT sends at most 64 rows to the LM head per call");
    const int rows = (int)total;
    if ((r = check_tokens(c, rows, tokens))) return r;
    if ((r = check_positions(c, rows, positions, 0))) return r;

    // Row plan: per-row slot, kept rows, attention query blocks.
    std::vector<int> slot(rows), keep, plan;
    std::vector<int> b0, bn, kb0, kbn;
    int off = 0;
    for (int s = 0; s < n_seq; ++s) {
        const int n = n_tokens[s];
        for (int i = 0; i < n; ++i) slot[off + i] = seq_ids[s];
        for (int i = 0; i < n; i += kPrefillQB) {
            b0.push_back(off + i);
            bn.push_back(std::min(kPrefillQB, n - i));
        }
        const int k0 = (int)keep.size();
        for (int i = n - n_out; i < n; ++i) keep.push_back(off + i);
        for (int i = 0; i < n_out; i += kPrefillQB) {
            kb0.push_back(k0 + i);
            kbn.push_back(std::min(kPrefillQB, n_out - i));
        }
        off += n;
    }
    const int n_keep = (int)keep.size();
    {
        // Longest query blocks (most keys) first, so the causal attention's
        // heavy blocks do not form the tail of the grid.
        std::vector<int> ord(b0.size());
        for (size_t i = 0; i < ord.size(); ++i) ord[i] = (int)i;
        auto last_pos = [&](int i) {
            int m = 0;
            for (int r = 0; r < bn[i]; ++r) m = std::max(m, (int)positions[b0[i] + r]);
            return m;
        };
        std::vector<int> key(ord.size());
        for (size_t i = 0; i < ord.size(); ++i) key[i] = last_pos((int)i);
        std::stable_sort(ord.begin(), ord.end(), [&](int x, int y) { return key[x] > key[y]; });
        std::vector<int> s0(ord.size()), sn(ord.size());
        for (size_t i = 0; i < ord.size(); ++i) {
            s0[i] = b0[ord[i]];
            sn[i] = bn[ord[i]];
        }
        b0.swap(s0);
        bn.swap(sn);
    }
    plan.insert(plan.end(), b0.begin(), b0.end());
    plan.insert(plan.end(), bn.begin(), bn.end());
    plan.insert(plan.end(), kb0.begin(), kb0.end());
    plan.insert(plan.end(), kbn.begin(), kbn.end());
    // Per sequence: slot, and the end of the positions whose tensor-core
    // attention operands must be converted from the cache: the positions
    // before its first row when its rows are consecutive positions (the QKV
    // epilogue writes its own rows' operands), else all up to the largest.
    int conv_tiles = 0;
    {
        std::vector<int> ss(n_seq), se(n_seq);
        int o = 0;
        for (int s = 0; s < n_seq; ++s) {
            const int n = n_tokens[s];
            int m = 0;
            bool consecutive = true;
            for (int i = 0; i < n; ++i) {
                m = std::max(m, (int)positions[o + i]);
                if (i > 0 && positions[o + i] != positions[o + i - 1] + 1) consecutive = false;
            }
            ss[s] = seq_ids[s];
            se[s] = consecutive ? (int)positions[o] : m + 1;
            conv_tiles = std::max(conv_tiles, (se[s] + 63) / 64);
            o += n;
        }
        plan.insert(plan.end(), ss.begin(), ss.end());
        plan.insert(plan.end(), se.begin(), se.end());
    }
    Workspace& w = c.ws;
    Q2_CHECK(&c, cudaMemcpyAsync(w.rows_tok, tokens, rows * 4, cudaMemcpyHostToDevice, st));
    Q2_CHECK(&c, cudaMemcpyAsync(w.rows_pos, positions, rows * 4, cudaMemcpyHostToDevice, st));
    Q2_CHECK(&c, cudaMemcpyAsync(w.rows_slot, slot.data(), rows * 4, cudaMemcpyHostToDevice, st));
    Q2_CHECK(&c, cudaMemcpyAsync(w.keep_rows, keep.data(), n_keep * 4, cudaMemcpyHostToDevice, st));
    Q2_CHECK(&c, cudaMemcpyAsync(w.blk, plan.data(), plan.size() * 4, cudaMemcpyHostToDevice, st));
    PrefillPlan pp;
    const int nb = (int)b0.size(), nkb = (int)kb0.size();
    pp.blk_row0 = w.blk;
    pp.blk_nrows = w.blk + nb;
    pp.n_blk = nb;
    pp.kblk_row0 = w.blk + 2 * nb;
    pp.kblk_nrows = w.blk + 2 * nb + nkb;
    pp.n_kblk = nkb;
    pp.seq_slot = w.blk + 2 * nb + 2 * nkb;
    pp.seq_conv = pp.seq_slot + n_seq;
    pp.n_seq = n_seq;
    pp.conv_tiles = conv_tiles;

    const bool logits_dev = logits && is_device_ptr(logits);
    const bool ids_dev = ids && is_device_ptr(ids);
    float* lg = logits_dev ? logits : nullptr;
    if (logits && !logits_dev) {
        if (w.out_logits_rows < (size_t)n_keep) {
            if (w.out_logits) cudaFree(w.out_logits);
            w.out_logits = nullptr;
            w.out_logits_rows = 0;
            if (cudaMalloc(&w.out_logits, (size_t)n_keep * c.cfg.vocab * 4) != cudaSuccess) {
                cudaGetLastError();
                w.out_logits = nullptr;
                return fail(&c, QWEN2_E_OOM, "logits staging allocation failed");
            }
            w.out_logits_rows = n_keep;
        }
        lg = w.out_logits;
    }
    cudaError_t e = enqueue_prefill(c, rows, n_keep, pp, lg, ids ? (ids_dev ? ids : w.ids) : nullptr, st);
    if (e != cudaSuccess) return cuda_fail(&c, e, "prefill launch");
    if (logits && !logits_dev)
        Q2_CHECK(&c, cudaMemcpyAsync(logits, lg, (size_t)n_keep * c.cfg.vocab * 4, cudaMemcpyDeviceToHost, st));
    if (ids && !ids_dev) Q2_CHECK(&c, cudaMemcpyAsync(ids, w.ids, n_keep * 4, cudaMemcpyDeviceToHost, st));
    c.last_rows_out = n_keep;
    if ((logits && !logits_dev) || (ids && !ids_dev)) Q2_CHECK(&c, cudaStreamSynchronize(st));
    return QWEN2_OK;
}

int qwen2_decode_step(qwen2_ctx* h, int32_t n_seq, const int32_t* seq_ids, const int32_t* tokens,
                      const int32_t* positions, float* logits, int32_t* ids, void* stream) {
    if (!h) return QWEN2_E_ARG;
    Ctx& c = h->c;
    c.last_error.clear();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (n_seq < 1 || n_seq > c.cfg.max_seqs) return fail(&c, QWEN2_E_ARG, "n_seq outside [1, max_seqs]");
    if (n_seq > max_decode_batch(c))
        return fail(&c, QWEN2_E_UNSUPPORTED, "more than " + std::to_string(max_decode_batch(c)) +
                                                 " sequences per decode step with these weights");
    if (!seq_ids || !tokens || !positions) return fail(&c, QWEN2_E_ARG, "null input pointer");
    int r = check_seq_ids(c, n_seq, seq_ids);
    if (r) return r;
    if ((r = check_tokens(c, n_seq, tokens))) return r;
    if ((r = check_positions(c, n_seq, positions, 0))) return r;
    DecodeState& d = c.ds;
    Q2_CHECK(&c, cudaMemcpyAsync(d.tok, tokens, n_seq * 4, cudaMemcpyHostToDevice, st));
    Q2_CHECK(&c, cudaMemcpyAsync(d.pos, positions, n_seq * 4, cudaMemcpyHostToDevice, st));
    Q2_CHECK(&c, cudaMemcpyAsync(d.slot, seq_ids, n_seq * 4, cudaMemcpyHostToDevice, st));
    Q2_CHECK(&c, cudaMemsetAsync(d.step, 0, 4, st));
    if ((r = run_decode_step(c, n_seq, logits != nullptr, st))) return r;
    const bool host_out = (logits && !is_device_ptr(logits)) || (ids && !is_device_ptr(ids));
    if (logits)
        Q2_CHECK(&c, cudaMemcpyAsync(logits, c.ws.logits, (size_t)n_seq * c.cfg.vocab * 4, cudaMemcpyDefault, st));
    if (ids) Q2_CHECK(&c, cudaMemcpyAsync(ids, d.ids_hist, n_seq * 4, cudaMemcpyDefault, st));
    c.last_rows_out = n_seq;
    if (host_out) Q2_CHECK(&c, cudaStreamSynchronize(st));
    return QWEN2_OK;
}

// decode_steps with optional stop ids; with n_generated NULL (plain
// decode_steps) no stop handling runs at all.
static int decode_steps_impl(qwen2_ctx* h, int32_t n_seq, const int32_t* seq_ids, const int32_t* first_tokens,
                      const int32_t* start_positions, int32_t n_steps, const int32_t* stop_ids, int32_t n_stop,
                      int32_t* ids, int32_t* n_generated, void* stream) {
    if (!h) return QWEN2_E_ARG;
    Ctx& c = h->c;
    c.last_error.clear();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (n_seq < 1 || n_seq > c.cfg.max_seqs) return fail(&c, QWEN2_E_ARG, "n_seq outside [1, max_seqs]");
    if (n_seq > max_decode_batch(c))
        return fail(&c, QWEN2_E_UNSUPPORTED, "more than " + std::to_string(max_decode_batch(c)) +
                                                 " sequences per decode step with these weights");
    if (!seq_ids || !first_tokens || !start_positions || !ids) return fail(&c, QWEN2_E_ARG, "null pointer");
    if (n_steps < 1) return fail(&c, QWEN2_E_ARG, "n_steps must be >= 1");
    if (n_stop < 0 || n_stop > kMaxStopIds)
        return fail(&c, QWEN2_E_ARG, "n_stop outside [0, " + std::to_string(kMaxStopIds) + "]");
    const bool stops = n_generated != nullptr;
    if (n_stop > 0 && (!stop_ids || !stops)) return fail(&c, QWEN2_E_ARG, "null stop_ids or n_generated");
    for (int k = 0; k < n_stop; ++k)
        if (stop_ids[k] < 0 || stop_ids[k] >= c.cfg.vocab)
            return fail(&c, QWEN2_E_ARG, "stop id " + std::to_string(stop_ids[k]) + " outside [0, vocab)");
    int r = check_seq_ids(c, n_seq, seq_ids);
    if (r) return r;
    if ((r = check_tokens(c, n_seq, first_tokens))) return r;
    if ((r = check_positions(c, n_seq, start_positions, n_steps - 1))) return r;
    DecodeState& d = c.ds;
    Q2_CHECK(&c, cudaMemcpyAsync(d.tok, first_tokens, n_seq * 4, cudaMemcpyHostToDevice, st));
    Q2_CHECK(&c, cudaMemcpyAsync(d.pos, start_positions, n_seq * 4, cudaMemcpyHostToDevice, st));
    Q2_CHECK(&c, cudaMemcpyAsync(d.slot, seq_ids, n_seq * 4, cudaMemcpyHostToDevice, st));
    if (n_stop > 0) Q2_CHECK(&c, cudaMemcpyAsync(d.stop_ids, stop_ids, n_stop * 4, cudaMemcpyHostToDevice, st));
    Q2_CHECK(&c, cudaMemsetAsync(d.step, 0, 4, st));
    const bool host_out = !is_device_ptr(ids) || (stops && !is_device_ptr(n_generated));
    for (int s0 = 0; s0 < n_steps; s0 += kIdsHist) {
        const int n = std::min(kIdsHist, n_steps - s0);
        for (int s = 0; s < n; ++s)
            if ((r = run_decode_step(c, n_seq, false, st))) return r;
        if (stops) Q2_CHECK(&c, enqueue_stop_mask(c, n_seq, n, n_stop, s0 == 0, st));
        Q2_CHECK(&c, cudaMemcpy2DAsync(ids + (size_t)s0 * n_seq, n_seq * 4, d.ids_hist, c.cfg.max_seqs * 4,
                                       n_seq * 4, n, cudaMemcpyDefault, st));
    }
    if (stops) Q2_CHECK(&c, cudaMemcpyAsync(n_generated, d.n_gen, n_seq * 4, cudaMemcpyDefault, st));
    c.last_rows_out = n_seq;
    if (host_out) Q2_CHECK(&c, cudaStreamSynchronize(st));
    return QWEN2_OK;
}

int qwen2_decode_steps(qwen2_ctx* h, int32_t n_seq, const int32_t* seq_ids, const int32_t* first_tokens,
                       const int32_t* start_positions, int32_t n_steps, int32_t* ids, void* stream) {
    return decode_steps_impl(h, n_seq, seq_ids, first_tokens, start_positions, n_steps, nullptr, 0, ids, nullptr,
                             stream);
}

int qwen2_decode_steps_stop(qwen2_ctx* h, int32_t n_seq, const int32_t* seq_ids, const int32_t* first_tokens,
                            const int32_t* start_positions, int32_t n_steps, const int32_t* stop_ids,
                            int32_t n_stop, int32_t* ids, int32_t* n_generated, void* stream) {
    if (h && !n_generated) return fail(&h->c, QWEN2_E_ARG, "n_generated is NULL");
    return decode_steps_impl(h, n_seq, seq_ids, first_tokens, start_positions, n_steps, stop_ids, n_stop, ids,
                             n_generated, stream);
}

int qwen2_final_hidden(qwen2_ctx* h, float* dst, int32_t rows, void* stream) {
    if (!h) return QWEN2_E_ARG;
    Ctx& c = h->c;
    if (!dst || rows < 1 || rows > c.last_rows_out)
        return fail(&c, QWEN2_E_ARG, "rows outside [1, rows of the last call]");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Q2_CHECK(&c, cudaMemcpyAsync(dst, c.ws.hidden, (size_t)rows * c.cfg.hidden * 4, cudaMemcpyDefault, st));
    if (!is_device_ptr(dst)) Q2_CHECK(&c, cudaStreamSynchronize(st));
    return QWEN2_OK;
}

int qwen2_test_raise_guard(qwen2_ctx* h, int32_t code, void* stream) {
    if (!h) return QWEN2_E_ARG;
    Ctx& c = h->c;
    // The guard codes the kernels write: 1 position, 2 token, 3 shape, 4 timeout.
    if (code < 1 || code > 4) return fail(&c, QWEN2_E_ARG, "guard code outside [1, 4]");
    Q2_CHECK(&c, enqueue_raise_guard(c, code, static_cast<cudaStream_t>(stream)));
    return QWEN2_OK;
}

int qwen2_test_stall_decode(qwen2_ctx* h, int32_t wait_us) {
    if (!h) return QWEN2_E_ARG;
    Ctx& c = h->c;
    if (wait_us < 100 || wait_us > 2000000) return fail(&c, QWEN2_E_ARG, "wait_us outside [100, 2000000]");
    if (!c.pers.ok)
        return fail(&c, QWEN2_E_UNSUPPORTED, "no persistent decode kernel in this context: " + c.pers.why_not);
    if (c.cfg.flags & (QWEN2_FLAG_NO_MEGAKERNEL | QWEN2_FLAG_NO_FUSE_QKV | QWEN2_FLAG_NO_FUSE_FFN))
        return fail(&c, QWEN2_E_UNSUPPORTED, "the context's flags switch the persistent decode kernel off");
    c.pers.test_stall = 1;
    c.pers.test_wait_ns = (unsigned long long)wait_us * 1000ull;
    return QWEN2_OK;
}

int qwen2_check_canaries(qwen2_ctx* h) {
    if (!h) return QWEN2_E_ARG;
    Ctx& c = h->c;
    Q2_CHECK(&c, cudaDeviceSynchronize());
    std::vector<unsigned char> buf(kCanaryBytes);
    for (size_t i = 0; i < c.canaries.size(); ++i) {
        const CanaryRegion& k = c.canaries[i];
        for (int side = 0; side < 2; ++side) {
            const unsigned char* at = side ? k.user + k.bytes : k.user - kCanaryBytes;
            Q2_CHECK(&c, cudaMemcpy(buf.data(), at, kCanaryBytes, cudaMemcpyDeviceToHost));
            for (size_t j = 0; j < kCanaryBytes; ++j)
                if (buf[j] != kCanaryByte)
                    return fail(&c, QWEN2_E_DEVICE_GUARD,
                                std::string("canary ") + (side ? "after" : "before") + " device buffer #" +
                                    std::to_string(i) + " (" + std::to_string(k.bytes) + " bytes) overwritten at byte " +
                                    std::to_string(j));
        }
    }
    return QWEN2_OK;
}

int qwen2_synchronize(qwen2_ctx* h, void* stream) {
    if (!h) return QWEN2_E_ARG;
    Ctx& c = h->c;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Q2_CHECK(&c, cudaStreamSynchronize(st));
    int word = 0;
    Q2_CHECK(&c, cudaMemcpy(&word, c.err, 4, cudaMemcpyDeviceToHost));
    if (word) {
        Q2_CHECK(&c, cudaMemset(c.err, 0, 4));
        Q2_CHECK(&c, persistent_reset(c));
        static const char* names[] = {"none", "position outside [0, n_ctx)", "token outside [0, vocab)",
                                      "unexpected shape", "bounded wait timed out"};
        const char* nm = word > 0 && word < 5 ? names[word] : "unknown";
        return fail(&c, QWEN2_E_DEVICE_GUARD, std::string("device guard ") + std::to_string(word) + ": " + nm);
    }
    return QWEN2_OK;
}

int64_t qwen2_weight_bytes(const qwen2_ctx* h) { return h ? (int64_t)h->c.wbytes : 0; }

uint32_t qwen2_features(const qwen2_ctx* h) {
    if (!h) return 0;
    return (h->c.pers.ok ? QWEN2_FEATURE_PERSISTENT_DECODE : 0u) | (h->c.tc.ok ? QWEN2_FEATURE_TENSOR_PREFILL : 0u);
}

int qwen2_profile_marks(qwen2_ctx* h, int64_t* out, int64_t max_marks, int32_t* n_cta, int32_t* n_marks) {
    if (!h) return QWEN2_E_ARG;
    Ctx& c = h->c;
    if (!c.pers.prof || !out || !n_cta || !n_marks)
        return fail(&c, QWEN2_E_ARG, "profiling is off (create with QWEN2_FLAG_PROFILE) or null argument");
    *n_cta = c.pers.grid;
    *n_marks = c.pers.prof_marks;
    const int64_t n = std::min<int64_t>(max_marks, (int64_t)c.pers.grid * c.pers.prof_marks);
    Q2_CHECK(&c, cudaDeviceSynchronize());
    Q2_CHECK(&c, cudaMemcpy(out, c.pers.prof, n * 8, cudaMemcpyDeviceToHost));
    return QWEN2_OK;
}

int64_t qwen2_kv_bytes_per_seq(const qwen2_config* g) {
    if (!g) return 0;
    return (int64_t)g->n_layer * 2 * g->n_kv_head * g->n_ctx * g->head_dim * 4;
}

int qwen2_quantize_q8_0(const uint16_t* w, int64_t rows, int64_t k, int8_t* q, uint16_t* d) {
    if (!w || !q || !d || rows < 0 || k <= 0 || k % 32) return QWEN2_E_ARG;
    quantize_q8_0_host(w, rows, k, q, d);
    return QWEN2_OK;
}

int qwen2_quantize_q4_0(const uint16_t* w, int64_t rows, int64_t k, uint8_t* packed, uint16_t* d) {
    if (!w || !packed || !d || rows < 0 || k <= 0 || k % 32) return QWEN2_E_ARG;
    quantize_q4_0_host(w, rows, k, packed, d);
    return QWEN2_OK;
}

}  // extern "C"
