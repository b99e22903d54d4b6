/*
 * qwen2.h -- C ABI of libqwen2: a single-GPU (GB300, sm_103a) forward of the
 * Qwen2 / Qwen2.5 dense decoder.
 *
 * The forward each call runs is the layer of the minfer page "Qwen2 /
 * Qwen2.5 Architecture Support", section 1:
 *
 *   h - RMSNorm - WQ/WK/WV matmuls + bias - RoPE(Q, K) - KV store
 *     - GQA attention (Q K^T scale -> softmax -> V) - WO matmul - + residual
 *     - RMSNorm - gate/up matmuls - SiLU(gate) * up - down matmul - + residual
 *
 * repeated n_layer times, then the final RMSNorm and the tied LM head
 * (W_lm = E; Module 7 -- Qwen2 / Qwen2.5, section 7.3; nnterp encyclopedia
 * qwen2, "The readout is the plain projection") and a greedy argmax taken on
 * the device (Module 7 section 7.3, performance note: GPU argmax avoids
 * reading back the 151936 logits each step).
 *
 * Conventions for every entry point:
 *  - Return value: QWEN2_OK (0) or one of the QWEN2_E_* codes below.  On an
 *    argument, position or support error nothing has been enqueued on the
 *    stream and no output or cache slot has been written;
 *    qwen2_last_error() holds a message.
 *  - "host" pointers are ordinary CPU memory; they are read before the call
 *    returns and may be reused at once.  Output pointers (logits, ids,
 *    hidden) may be device memory or host memory: the library copies through
 *    the unified address space.  If any output pointer is host memory the
 *    call synchronises the stream before it returns; otherwise it does not
 *    block the host.
 *  - `stream` is a cudaStream_t passed as void* (NULL: the legacy default
 *    stream).  All device work of a call is ordered on that stream.
 *  - A context is single-threaded: no two calls on one context may run at
 *    the same time.
 */
#ifndef QWEN2_H
#define QWEN2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- error codes --------------------------------------------------------- */
#define QWEN2_OK                 0
#define QWEN2_E_ARG              1  /* null pointer, token outside [0, vocab), bad count or sequence id */
#define QWEN2_E_POS              2  /* a position outside [0, n_ctx): a hard error, never truncation
                                       (minfer page section 6: positions[i] < n_ctx is enforced with a
                                       hard Err in the KV-store arm; section 7 item 5) */
#define QWEN2_E_UNSUPPORTED      3  /* a config this build does not implement (e.g. head_dim 96) */
#define QWEN2_E_OOM              4  /* device allocation failed */
#define QWEN2_E_CUDA             5  /* a CUDA runtime call failed */
#define QWEN2_E_DEVICE_GUARD     6  /* a kernel's own guard tripped (found at qwen2_synchronize) */

/* ---- weight storage formats -------------------------------------------- */
#define QWEN2_WEIGHTS_F16        0  /* f16 linear weights and LM head, f32 biases and norm weights
                                       (Module 7 section 7.4) */
#define QWEN2_WEIGHTS_Q8_0       1  /* the seven linear weights and the tied embedding / LM head held as
                                       Q8_0 blocks: 32 int8 values along K plus one f16 scale per block;
                                       quantised by the library from the f16 weights given to create */
#define QWEN2_WEIGHTS_Q4_0       2  /* as Q8_0 with 4-bit codes: blocks of 32 along k, d = max|x| / 7,
                                       codes clamp(round-half-away(x / d), -7, 7) + 8, two per byte
                                       (element 2j in the low nibble), one f16 scale per block: 18
                                       bytes per 32 weights.  Named beside Q8_0 as the tied output
                                       matmul's format on the minfer page (section 3), never defined
                                       there: the four-bit counterpart of the Q8_0 reading.  Runs the
                                       same paths as Q8_0 (batched decode, f32 prefill) */

/* ---- prefill arithmetic -------------------------------------------------- */
#define QWEN2_PREFILL_F32        0  /* f32 activations, f32 accumulation on CUDA cores */
#define QWEN2_PREFILL_TENSOR     1  /* tensor-core (tcgen05) GEMMs on f16 operands with f32 accumulation;
                                       residual, norm statistics, softmax and the KV cache stay f32 */
#define QWEN2_PREFILL_Q8_ACT     2  /* Q8_0 weights only: every product of the prefill (Q/K/V, o_proj,
                                       gate/up, down, the LM head of the kept rows) quantises its f32
                                       activation rows to Q8_0 blocks as the packer quantises weights,
                                       sums each 32-block's int8 products exactly and scales the sum by
                                       the two f16 block scales (the minfer page, section 6: the CUDA
                                       prefill runs an int8 "MMQ" product; the details are this
                                       library's reading).  At most 64 rows per call reach the LM head.
                                       Decode steps keep f32 activations */

/* ---- flags ------------------------------------------------------------- */
#define QWEN2_FLAG_NO_FUSE_QKV   0x1u  /* separate norm, Q, K and V products and epilogue kernels instead of
                                          the fused QKV kernel (minfer page section 3, MINFER_NO_FUSE_QKV);
                                          results are bit-identical either way */
#define QWEN2_FLAG_NO_FUSE_FFN   0x2u  /* separate norm, gate, up and SiLU*up kernels (MINFER_NO_FUSE_FFN) */
#define QWEN2_FLAG_NO_GRAPH      0x4u  /* launch decode kernels one by one, without a CUDA graph */
#define QWEN2_FLAG_NO_MEGAKERNEL 0x8u  /* decode with one kernel per step of the layer instead of the
                                          persistent single-launch decode kernel */
#define QWEN2_FLAG_PROFILE       0x10u /* the persistent decode kernel records per-phase timestamps
                                          (qwen2_profile_marks); costs a few stores per phase */

/* ---- feature bits (qwen2_features) --------------------------------------- */
#define QWEN2_FEATURE_PERSISTENT_DECODE 0x1u  /* batch-1 decode runs the persistent single-launch kernel */
#define QWEN2_FEATURE_TENSOR_PREFILL    0x2u  /* prefill GEMMs run on the tcgen05 tensor cores */

typedef struct qwen2_config {
    int32_t n_layer;        /* num_hidden_layers (24 on Qwen2.5-0.5B) */
    int32_t hidden;         /* hidden_size H (896); must be n_head * head_dim and a multiple of 128 */
    int32_t n_head;         /* num_attention_heads (14) */
    int32_t n_kv_head;      /* num_key_value_heads (2); must divide n_head, n_head/n_kv_head <= 8 */
    int32_t head_dim;       /* H / n_head: 64 (0.5B) or 128 (every larger size, nnterp
                             * encyclopedia qwen2, "Grouped-query attention"); 128 runs the
                             * per-step decode kernels and the f32 prefill (the persistent
                             * batch-1 kernel and the tensor-core prefill are built for 64) */
    int32_t intermediate;   /* intermediate_size I (4864); a multiple of 128 */
    int32_t vocab;          /* vocab_size V (151936) */
    float   rms_eps;        /* rms_norm_eps (1e-6) */
    double  rope_theta;     /* rope_theta (1e6) */
    int32_t weight_format;  /* QWEN2_WEIGHTS_* */
    int32_t prefill_mode;   /* QWEN2_PREFILL_* */
    int32_t n_ctx;          /* KV positions per sequence; positions must lie in [0, n_ctx) */
    int32_t max_seqs;       /* number of sequence slots (KV caches) */
    int32_t max_tokens;     /* most rows one qwen2_prefill call may carry (sum over its sequences) */
    uint32_t flags;         /* QWEN2_FLAG_* */
} qwen2_config;

/* One decoder layer, host memory, HF layout [out_features][in_features]
 * (Module 7 Lab 7; nnterp "Printout").  f16 values are IEEE binary16 bit
 * patterns (uint16_t). */
typedef struct qwen2_layer_weights {
    const uint16_t *wq;   /* [n_head*head_dim][H]      q_proj.weight */
    const uint16_t *wk;   /* [n_kv_head*head_dim][H]   k_proj.weight */
    const uint16_t *wv;   /* [n_kv_head*head_dim][H]   v_proj.weight */
    const uint16_t *wo;   /* [H][n_head*head_dim]      o_proj.weight (no bias) */
    const uint16_t *wg;   /* [I][H]                    mlp.gate_proj.weight */
    const uint16_t *wu;   /* [I][H]                    mlp.up_proj.weight */
    const uint16_t *wd;   /* [H][I]                    mlp.down_proj.weight */
    const float *bq;      /* [n_head*head_dim]         q_proj.bias */
    const float *bk;      /* [n_kv_head*head_dim]      k_proj.bias */
    const float *bv;      /* [n_kv_head*head_dim]      v_proj.bias */
    const float *attn_norm;  /* [H] input_layernorm.weight */
    const float *ffn_norm;   /* [H] post_attention_layernorm.weight */
} qwen2_layer_weights;

typedef struct qwen2_weights {
    const uint16_t *embed;             /* [V][H] embed_tokens.weight; also the LM head when tied */
    const uint16_t *lm_head;           /* [V][H] lm_head.weight, or NULL for a tied head (the
                                        * embedding is the readout: 0.5B to 3B).  From 7B up the
                                        * embedding and unembedding are separate matrices (nnterp
                                        * encyclopedia qwen2, "The readout is the plain
                                        * projection"); the logits are then lm_head . final_norm(x). */
    const float *final_norm;           /* [H] model.norm.weight */
    const qwen2_layer_weights *layers; /* [n_layer] */
} qwen2_weights;

typedef struct qwen2_ctx qwen2_ctx;

/* Create a context on the current CUDA device from a config (the minfer
 * page "Qwen2 / Qwen2.5 Architecture Support", section 2: the HParams
 * fields -- layers, hidden, heads, KV heads, head_dim, intermediate,
 * vocabulary, rms_eps, rope_theta -- and the LayerWeights tensors, with the
 * tied embedding as the output projection) and host weight pointers:
 * validate `cfg`, pack and
 * upload the weights (the library keeps its own device copies; the host
 * arrays may be freed after the call), allocate the zeroed KV cache of
 * max_seqs sequences, the workspace and the RoPE table.  Synchronous.
 * Errors: QWEN2_E_ARG (null pointers, non-positive sizes), QWEN2_E_UNSUPPORTED
 * (head_dim not 64 or 128, head_dim 128 with QWEN2_PREFILL_TENSOR,
 * H != n_head*head_dim, H or I not a multiple of 128, n_head % n_kv_head
 * != 0, group > 8), QWEN2_E_OOM, QWEN2_E_CUDA.
 * On success *out receives the context; on failure *out is set to NULL and
 * qwen2_last_error(NULL) describes the failure. */
int qwen2_create(const qwen2_config *cfg, const qwen2_weights *weights, qwen2_ctx **out);

/* Free every device buffer of the context (synchronises the device first).
 * NULL is accepted. */
void qwen2_destroy(qwen2_ctx *ctx);

/* Message of the last failed call on `ctx` ("" if none); with ctx == NULL,
 * the calling thread's last qwen2_create failure.  The string stays valid
 * until the next call on the same context (or thread). */
const char *qwen2_last_error(const qwen2_ctx *ctx);

/* The KV cache (minfer page, section 6: an f32 K and V cache per layer,
 * sized by n_ctx when the context is created -- 24 KB per position on
 * Qwen2.5-0.5B -- whose slot is the token's position) as caller-visible
 * device memory: *base receives a device
 * pointer to f32 [max_seqs][n_layer][2][n_kv_head][n_ctx][head_dim]
 * (index 0 of the third axis holds rotated keys, 1 values; slot = position),
 * contiguous row-major; dims[0..5] receive those six sizes.  The memory is
 * owned by the context; the caller may read or write it between calls, in
 * stream order (e.g. to save and restore a conversation). */
int qwen2_kv_cache(qwen2_ctx *ctx, float **base, int64_t dims[6]);

/* Prefill: run the rows of n_seq sequences through the forward, storing
 * every row's key and value at its position in its sequence's cache.
 *   seq_ids   host int32 [n_seq], distinct, each in [0, max_seqs)
 *   n_tokens  host int32 [n_seq], each >= n_out; their sum <= max_tokens
 *   tokens    host int32 [sum n_tokens], sequence after sequence, in [0, V)
 *   positions host int32 [sum n_tokens], in [0, n_ctx)
 *   n_out     rows per sequence that reach the LM head: the last n_out rows
 *             of each sequence (minfer page, section 3, "G3 tail-row
 *             optimization": the other rows are cut before the last layer's
 *             attention output, since only the kept rows' results are used)
 *   logits    nullable; f32 [n_seq*n_out][V]
 *   ids       nullable; int32 [n_seq*n_out], the lowest index of each row's
 *             maximum logit
 * A row at position p attends to cache slots 0..p of its sequence; all
 * rows of a call are stored before any row attends. */
int qwen2_prefill(qwen2_ctx *ctx, int32_t n_seq, const int32_t *seq_ids,
                  const int32_t *n_tokens, const int32_t *tokens,
                  const int32_t *positions, int32_t n_out,
                  float *logits, int32_t *ids, void *stream);

/* One decode step: one row for each of n_seq sequences, the forward of
 * minfer page section 1 at one new position per sequence.  Positions are
 * data (minfer page, section 6): the row's key and value go to slot
 * `position` of its sequence's cache and it attends to slots 0..position;
 * a position outside [0, n_ctx) is QWEN2_E_POS with nothing enqueued (a
 * hard error, never a truncation).
 *   seq_ids, tokens, positions  host int32 [n_seq]
 *   logits  nullable; f32 [n_seq][V]
 *   ids     nullable; int32 [n_seq] greedy ids */
int qwen2_decode_step(qwen2_ctx *ctx, int32_t n_seq, const int32_t *seq_ids,
                      const int32_t *tokens, const int32_t *positions,
                      float *logits, int32_t *ids, void *stream);

/* n_steps greedy decode steps without a host round trip per step: step 0
 * feeds first_tokens at start_positions, each later step feeds the previous
 * step's ids at the next position (positions are data, minfer page section
 * 6).  ids: int32 [n_steps][n_seq].  Fails with QWEN2_E_POS (nothing run)
 * if any start_position + n_steps > n_ctx. */
int qwen2_decode_steps(qwen2_ctx *ctx, int32_t n_seq, const int32_t *seq_ids,
                       const int32_t *first_tokens, const int32_t *start_positions,
                       int32_t n_steps, int32_t *ids, void *stream);

/* Greedy decode that ends at stop tokens: generation stops at the
 * end-of-sequence id or the chat end-of-turn id (minfer page, section 5
 * "Tokenizer and chat", stop tokens eos and im_end; the nnterp
 * encyclopedia's qwen2 page names them: <|endoftext|> 151643 on base
 * models, <|im_end|> 151645 on instruct models).  Steps as
 * qwen2_decode_steps, and the same errors and position checks, plus:
 *   stop_ids     host int32 [n_stop], 0 <= n_stop <= 8, each in [0, vocab)
 *                (QWEN2_E_ARG otherwise); with n_stop = 0 no id is masked
 *   ids          int32 [n_steps][n_seq], host or device: the id each step
 *                produced, -1 after the sequence's first generated stop id
 *   n_generated  int32 [n_seq], host or device, not NULL: the ids kept per
 *                sequence, the stop id included (n_steps when none came)
 * The step graph has a fixed shape, so every step is still computed for
 * every sequence: KV entries past a sequence's stop hold the continuation,
 * which attention never reads before a later call writes those positions
 * again.  The stop ids of first_tokens (inputs, not generated) do not
 * count. */
int qwen2_decode_steps_stop(qwen2_ctx *ctx, int32_t n_seq, const int32_t *seq_ids,
                            const int32_t *first_tokens, const int32_t *start_positions,
                            int32_t n_steps, const int32_t *stop_ids, int32_t n_stop,
                            int32_t *ids, int32_t *n_generated, void *stream);

/* Copy the final-norm output rows (the input of the LM head,
 * "final_norm_output" in the nnterp names) of the last prefill or decode
 * step into dst: f32 [rows][H], rows <= n_seq*n_out of that call.  Device or
 * host dst. */
int qwen2_final_hidden(qwen2_ctx *ctx, float *dst, int32_t rows, void *stream);

/* Test hook for failure detection without a GPU fault: enqueue on `stream`
 * a one-thread kernel that writes `code` into the context's device guard
 * word the way a kernel does when one of its bounded waits gives up
 * (first code wins).  The next qwen2_synchronize then reports
 * QWEN2_E_DEVICE_GUARD with that code, clears the word and resets the
 * persistent decode kernel's exchange state.  code in [1, 4]
 * (position, token, shape, timeout); QWEN2_E_ARG otherwise. */
int qwen2_test_raise_guard(qwen2_ctx *ctx, int32_t code, void *stream);

/* Test hook for failure detection without a GPU fault: the next
 * persistent batch-1 decode launch of this context (one launch; the hook is
 * cleared by it) waits, after layer 0's Q/K/V, on an arrival counter that no
 * CTA ever arrives at, and every bounded wait of that launch gives up after
 * wait_us microseconds instead of 2 s.  The wait runs out, the CTAs stop
 * (each waits, bounded, for its weight copies in flight) and the launch
 * sets the guard word; the next qwen2_synchronize returns
 * QWEN2_E_DEVICE_GUARD ("bounded wait timed out") and resets the kernel's
 * exchange state.  The launch writes no ids; KV rows of layer 0 at its
 * position may be written.  Errors: QWEN2_E_ARG (wait_us outside [100,
 * 2000000]), QWEN2_E_UNSUPPORTED (the context has no persistent kernel). */
int qwen2_test_stall_decode(qwen2_ctx *ctx, int32_t wait_us);

/* Debug check for writes past the ends of device buffers: every buffer the
 * context allocates (KV cache, workspace, decode state) sits between two
 * 256-byte guard regions filled with 0xA5 at create.  Synchronises the
 * device, reads the guards back and returns QWEN2_E_DEVICE_GUARD (the
 * message names the buffer's index, size and the first changed byte) if a
 * kernel wrote into one, else QWEN2_OK.  Costs two small device-to-host
 * copies per buffer; meant for tests, not for every step. */
int qwen2_check_canaries(qwen2_ctx *ctx);

/* Synchronise `stream` and report any device-side guard that tripped since
 * the last check (QWEN2_E_DEVICE_GUARD, with the guard's code in the
 * message); clears the guard word. */
int qwen2_synchronize(qwen2_ctx *ctx, void *stream);

/* Bytes of packed weights resident on the device (linear weights, LM head,
 * biases, norm weights and, for Q8_0, scales), with 256-byte alignment
 * padding between tensors. */
int64_t qwen2_weight_bytes(const qwen2_ctx *ctx);

/* Feature bits of this context (QWEN2_FEATURE_*): which kernels its calls
 * will run on this device and shape.  0 for NULL. */
uint32_t qwen2_features(const qwen2_ctx *ctx);

/* Timestamps of the last persistent decode launch of a context created with
 * QWEN2_FLAG_PROFILE: out receives up to max_marks int64 values laid out
 * [cta][mark] (the GPU global timer in ns, 0 where a CTA did not pass a
 * mark).  Mark 0 is the launch start; layer l owns marks 1 + 16 l + k for
 * k = 0 input x gathered, 1 normed, 2 Q/K/V done, 3 queries ready
 * (attention CTAs only), 4 attention done, 5 attention partials counted,
 * 6 chunk merge done, 7 o_proj done, 8 x counted, 9 x gathered, 10 gate/up
 * done, 11 SwiGLU output counted, 12 gathered, 13 down done; marks
 * 1 + 16 L, 2 + 16 L and 3 + 16 L are the final x gathered, the LM head
 * done and the argmax done.  *n_cta and *n_marks receive the two sizes.
 * QWEN2_E_ARG if profiling is off.  Synchronises the device. */
int qwen2_profile_marks(qwen2_ctx *ctx, int64_t *out, int64_t max_marks, int32_t *n_cta, int32_t *n_marks);

/* Bytes one sequence's KV cache takes: n_layer * 2 * n_kv_head * n_ctx *
 * head_dim * 4 (24 KB per position on Qwen2.5-0.5B, minfer page section 6). */
int64_t qwen2_kv_bytes_per_seq(const qwen2_config *cfg);

/* Tied LM head and greedy argmax on already-normalised rows, with no device
 * allocation and no context.  Not an operation of its own in the Qwen2
 * description: it is the decode step's last stage (logits = E . h with the
 * embedding matrix E as the output projection, then the greedy id) offered
 * for callers that own every byte of device memory through their own
 * allocator and cannot let a library call cudaMalloc or hold a context.
 *   embed:  device, f16 bits [vocab][hidden_size], row-major (E itself).
 *   hidden: device, f32 [n_rows][hidden_size], the final RMSNorm output.
 *   logits: device, f32 [n_rows][vocab], or NULL to skip writing logits.
 *   ids:    device, int32 [n_rows]: the lowest index of each row's maximum
 *           (a NaN logit counts above every number, so a row of NaN logits
 *           gives its first index: every id is inside [0, vocab)).
 * Asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 * Limits: 1 <= n_rows <= 8; hidden_size a multiple of 8, at most 1024;
 * vocab >= 1; embed 16-byte aligned (rows are read with 16-byte vector
 * loads; sub-allocated pointers must keep that alignment).  Outside them:
 * QWEN2_E_ARG, nothing launched.
 * Scratch: a fixed static device array of the library (about 32 KB per
 * device).  The first call on a device looks up its address with that
 * device current, and so does the first call under any other context made
 * current on that device later; make that first call before any other use
 * that must not see a runtime call other than a kernel launch and a memset.
 * Each call zeroes the scratch's arrival counter on `stream` before its
 * kernel.  Two calls in flight at once on one device (other streams or
 * threads) share the scratch and race: order them.  The logits are bitwise
 * those of qwen2_decode_step for the same rows.  Errors: QWEN2_E_ARG,
 * QWEN2_E_CUDA; qwen2_last_error(NULL) describes the failure. */
int qwen2_lm_head_argmax_noalloc(const uint16_t *embed, const float *hidden, int32_t n_rows,
                                 int32_t hidden_size, int32_t vocab, float *logits, int32_t *ids,
                                 void *stream);

/* Host-only Q8_0 quantisation of an f16 matrix [rows][k] (k a multiple of
 * 32), as the library's packer does it: blocks of 32 along k;
 * d = max|x| / 127 in f32; q = clamp(round-half-away(x / d), -127, 127)
 * (q = 0 where d = 0); the stored scale is f16(d), round to nearest even.
 * q: int8 [rows][k]; d: f16 bits [rows][k/32].  Needs no GPU.  The format
 * is named, not defined, on the minfer page (sections 3 and 6). */
int qwen2_quantize_q8_0(const uint16_t *w, int64_t rows, int64_t k, int8_t *q, uint16_t *d);

/* Host-only Q4_0 quantisation of an f16 matrix [rows][k] (k a multiple of
 * 32), as the library's packer does it (QWEN2_WEIGHTS_Q4_0): packed:
 * uint8 [rows][k/2], element 2j in the low nibble of byte j; d: f16 bits
 * [rows][k/32].  Needs no GPU.  QWEN2_E_ARG for null pointers or a ragged
 * k. */
int qwen2_quantize_q4_0(const uint16_t *w, int64_t rows, int64_t k, uint8_t *packed, uint16_t *d);

#ifdef __cplusplus
}
#endif
#endif /* QWEN2_H */
