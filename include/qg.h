/*
 * qg.h -- C ABI of the batch-1 hybrid Gated-DeltaNet / full-attention decode
 * step with GGUF Q4_K / Q6_K weights, for NVIDIA GB300 (sm_103a).
 *
 * Every function returns QG_OK (0) or a negative QG_ERR_* code and never
 * throws; qg_last_error() gives a message for the calling thread.  Device
 * pointers ("_dev", "device") are CUDA global-memory addresses on the
 * library's current device; host pointers are plain CPU memory.  `qg_stream`
 * is a cudaStream_t (NULL = the legacy default stream).
 *
 * The operations and their order are those of forward_qwen35_cuda.rs
 * (aprender-serve 0.68.2): the Gated DeltaNet layer (deltanet_layer_inner),
 * the full-attention layer (attention_layer_inner) and the whole token
 * (forward_single), ending, as in aprender PR #4332 ("Greedy GPU argmax"), in
 * an on-device argmax that returns a 4-byte token id, first index on ties.
 */
#ifndef QG_H
#define QG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* qg_stream; /* == cudaStream_t */

/* ------------------------------------------------------------ status codes */
enum {
    QG_OK = 0,
    QG_ERR_SHAPE = -1,      /* a dimension the kernels cannot serve (e.g. k % 256 != 0,
                               n_v_heads % n_k_heads != 0, max_seq_len == 0, lm_head
                               shape != vocab x hidden) */
    QG_ERR_QTYPE = -2,      /* a tensor type with no kernel here */
    QG_ERR_EMPTY = -3,      /* an empty tensor (n == 0 or no data) */
    QG_ERR_POS = -4,        /* position >= the state's max_seq_len */
    QG_ERR_TOKEN = -5,      /* token id >= vocab */
    QG_ERR_LAYER_KIND = -6, /* layer index of the other kind, or out of range */
    QG_ERR_CUDA = -7,       /* a CUDA runtime call failed (message has the CUDA error) */
    QG_ERR_TIMEOUT = -8,    /* a bounded device-side wait gave up (kernel set the error word) */
    QG_ERR_ARG = -9,        /* NULL or misaligned pointer, negative size, bad argument */
    QG_ERR_OOM = -10        /* device or pinned host allocation failed */
};

/* GGML type ids of the supported k-quants. */
enum { QG_QTYPE_Q4_K = 12, QG_QTYPE_Q6_K = 14 };
/* Layer kinds (forward_qwen35_cuda.rs, enum CudaLayer). */
enum { QG_LAYER_DELTANET = 0, QG_LAYER_ATTENTION = 1 };

/* Shapes of the model (forward_qwen35_cuda.rs, struct Qwen35CudaDims).
 * conv_dim = 2 * n_k_heads * head_k_dim + n_v_heads * head_v_dim.
 * Served: hidden, ffn, n_v_heads*head_v_dim and n_heads*head_dim multiples of
 * 256; head_k_dim == 128; head_v_dim 32, 64 or 128; conv_kernel
 * 2..8; head_dim == 256;
 * n_rot even and <= head_dim; n_v_heads % n_k_heads == 0; n_heads % n_kv_heads
 * == 0 with at most 8 query heads per kv head. */
typedef struct qg_config {
    int32_t n_layers, hidden, ffn, vocab;
    int32_t n_k_heads, n_v_heads, head_k_dim, head_v_dim, conv_kernel;
    int32_t n_heads, n_kv_heads, head_dim, n_rot;
    float eps;                  /* every RMSNorm, per-head norm, gated norm and L2 norm */
    float rope_theta;           /* theta_scale = rope_theta^(-2/n_rot) is formed on the host */
    const int32_t* layer_kinds; /* host, n_layers entries of QG_LAYER_* */
} qg_config;

/* A quantized tensor in HOST memory, raw GGUF layout: n rows of k weights,
 * each row k/256 super-blocks (Q4_K 144 bytes, Q6_K 210 bytes). */
typedef struct qg_qtensor {
    const void* data;
    int32_t qtype; /* QG_QTYPE_* */
    int32_t n, k;
} qg_qtensor;

/* One layer's HOST weights (forward_qwen35_cuda.rs, CudaDeltaNetLayer and
 * CudaAttentionLayer).  Fields of the other kind are ignored.  Quantized
 * projections are Q4_K except ffn_down, which is Q6_K (QG_ERR_QTYPE otherwise). */
typedef struct qg_layer_weights {
    int32_t kind;
    const float* attn_norm;           /* [hidden] */
    const float* post_attention_norm; /* [hidden] */
    qg_qtensor ffn_gate, ffn_up;      /* [ffn x hidden] */
    qg_qtensor ffn_down;              /* [hidden x ffn] */
    /* Gated DeltaNet */
    const float* ssm_conv1d;  /* [conv_dim][conv_kernel] */
    const float* ssm_a_log;   /* [n_v_heads]: A_log; the decay rate a = -exp(A_log) is formed at create */
    const float* ssm_dt_bias; /* [n_v_heads] */
    const float* ssm_norm;    /* [head_v_dim], shared by the value heads */
    qg_qtensor attn_qkv;      /* [conv_dim x hidden] */
    qg_qtensor ssm_alpha, ssm_beta; /* [n_v_heads x hidden] */
    qg_qtensor attn_gate;     /* [n_v_heads*head_v_dim x hidden] */
    qg_qtensor ssm_out;       /* [hidden x n_v_heads*head_v_dim] */
    /* full attention */
    const float* attn_q_norm; /* [head_dim] */
    const float* attn_k_norm; /* [head_dim] */
    qg_qtensor attn_q;        /* [2*n_heads*head_dim x hidden], per head [q | gate] */
    qg_qtensor attn_k, attn_v;/* [n_kv_heads*head_dim x hidden] */
    qg_qtensor attn_output;   /* [hidden x n_heads*head_dim] */
} qg_layer_weights;

typedef struct qg_host_weights {
    const float* token_embd;  /* [vocab][hidden] f32 */
    const float* output_norm; /* [hidden] */
    qg_qtensor lm_head;       /* Q6_K [vocab x hidden], no bias */
    const qg_layer_weights* layers; /* n_layers entries */
} qg_host_weights;

typedef struct qg_model qg_model; /* device-resident weights (opaque) */
typedef struct qg_state qg_state; /* per-sequence decode state (opaque) */

/* Host-side counters of one state (aprender PR #4332 test counters:
 * device_allocs_total, device_to_host_bytes_total). */
typedef struct qg_stats {
    uint64_t device_allocs;   /* cudaMalloc/cudaHostAlloc calls made for this state */
    uint64_t h2d_bytes;       /* host-to-device bytes copied by decode calls */
    uint64_t d2h_bytes;       /* device-to-host bytes copied by decode calls */
    uint64_t graph_launches;  /* CUDA graph launches */
    uint64_t graph_captures;  /* CUDA graphs captured */
    uint64_t graph_kernel_nodes; /* kernel nodes of the per-token graph */
    uint64_t steps;           /* tokens decoded */
} qg_stats;

/* ---------------------------------------------------------- model / state */

/* Copies the host weights to `device` (the caller keeps its buffers):
 * fuses the projections that share an input, forms a = -exp(A_log) and
 * repacks every Q6_K tensor to the planar layout below
 * (forward_qwen35_cuda.rs, with_max_seq_len, build_layer).
 * Errors: QG_ERR_SHAPE, QG_ERR_QTYPE, QG_ERR_EMPTY, QG_ERR_ARG, QG_ERR_OOM, QG_ERR_CUDA. */
int qg_model_create(const qg_config* cfg, const qg_host_weights* w, int device, qg_model** out);
int qg_model_destroy(qg_model* m);

/* A fresh zeroed state (forward_qwen35_cuda.rs, new_state / build_state):
 * per DeltaNet layer a conv window [conv_dim][conv_kernel-1] (oldest first)
 * and a recurrent state [n_v_heads][head_v_dim][head_k_dim] with
 * s[j*head_k_dim + i] == S[i][j]; per attention layer f32 K and V caches
 * [max_seq_len][n_kv_heads*head_dim]; all scratch, the device token/position
 * slots, pinned host slots and its own CUDA stream.  Allocates everything a
 * decode needs up front.  Errors: QG_ERR_SHAPE (max_seq_len < 1), QG_ERR_OOM. */
int qg_state_create(const qg_model* m, int max_seq_len, qg_state** out);

/* KV cache formats.  QG_KV_F32: f32 rows, as qg_state_create makes them.
 * QG_KV_Q8_0_Q5_1: the decode session's quantized cache (forward_qwen35_cuda.rs,
 * full-attention layer: q8_0 K / q5_1 V, quantized on append by the attention
 * kernel, attention over the dequantized rows, this token's included).  Blocks
 * of 32 values with the GGUF block contents -- q8_0: f16 d, int8 q, x = d*q;
 * q5_1: f16 d, f16 m, 5-bit q, x = d*q + m -- stored per (kv head, position)
 * as one record with the 8 blocks' scales first (head_dim 256):
 *   K record, 272 bytes: d[8] (f16) | q[256] (int8)
 *   V record, 192 bytes: (d, m)[8] (f16 pairs) | qh[8] (u32, bit j = bit 4 of
 *     value j's code) | qs[8][16] (byte i: code i & 15 low, code i+16 & 15 high)
 * One layer's cache is [n_kv_heads][max_seq_len][record].  The quantizer: d from
 * the block's f32 statistics (q8_0: max|x|/127; q5_1: (max-min)/31, m = min),
 * code = roundf(x * (1/d)) (q5_1: roundf((x-min) * (1/d))), IEEE f32 operations,
 * clamped to the code range (zero codes when d is below FLT_MIN); d and m rounded
 * to f16 (nearest even), and every reader uses the stored f16 values. */
enum { QG_KV_F32 = 0, QG_KV_Q8_0_Q5_1 = 1 };
/* qg_state_create with the KV cache in `kv_format`.  A quantized cache holds
 * 464 bytes per (position, kv head) instead of 2048.  Errors: those of
 * qg_state_create, QG_ERR_ARG (unknown format). */
int qg_state_create_kv(const qg_model* m, int max_seq_len, int kv_format, qg_state** out);
int qg_state_kv_format(const qg_state* s, int* kv_format);
int qg_state_destroy(qg_state* s);
/* Zero every window, state and cache; kv_len = 0; clear the token mask: the
 * state a fresh forward_qwen35_cuda.rs new_state gives, without reallocating
 * (the captured graph and scratch are kept). */
int qg_state_reset(qg_state* s);

/* Teacher forcing (forward_qwen35_cuda.rs upload_layer, upload_attention_kv,
 * download_layer).  HOST buffers.  upload_layer: conv [conv_dim*(conv_kernel-1)]
 * and ssm [n_v_heads*head_v_dim*head_k_dim] of DeltaNet layer il.
 * upload_kv: `rows` whole K and V rows of attention layer il (f32,
 * [rows][n_kv_heads*head_dim]), sets kv_len = rows; a quantized cache stores
 * them through the append's quantizer on the device (it allocates and frees a
 * device staging buffer of 2*rows*kv_row floats).
 * download_layer: DeltaNet -> (conv, ssm), *n = max of the two lengths written
 * as (conv_len, ssm_len) into a and b; attention -> the kv_len*kv_row K and V
 * values written so far (*n = kv_len * n_kv_heads*head_dim; 0 on a fresh
 * state).  Pass a == b == NULL to query *n (DeltaNet: *n = ssm_len).
 * A quantized cache is read with qg_state_download_kv_records instead
 * (download_layer of its attention layers gives QG_ERR_ARG).
 * Errors: QG_ERR_LAYER_KIND, QG_ERR_SHAPE, QG_ERR_ARG, QG_ERR_CUDA. */
int qg_state_upload_layer(qg_state* s, int il, const float* conv, const float* ssm);
int qg_state_upload_kv(qg_state* s, int il, const float* k, const float* v, int rows);
int qg_state_download_layer(qg_state* s, int il, float* a, float* b, size_t* n);
/* Quantized cache of attention layer il as written so far: the first kv_len
 * K records of every kv head into k ([n_kv_heads][kv_len][272 bytes], HOST)
 * and the V records into v ([n_kv_heads][kv_len][192]); *k_bytes / *v_bytes
 * receive the sizes (pass k == v == NULL to query them).  Errors:
 * QG_ERR_LAYER_KIND, QG_ERR_ARG (NULL size pointers, or an f32 cache),
 * QG_ERR_CUDA. */
int qg_state_download_kv_records(qg_state* s, int il, void* k, void* v, size_t* k_bytes, size_t* v_bytes);
/* The residual stream after the last completed step ([hidden], host). */
int qg_state_download_hidden(qg_state* s, float* hidden_host);
int qg_state_kv_len(const qg_state* s, int* kv_len);
/* The CUDA stream every decode call of this state runs on (owned by the
 * state), e.g. to record timing events around qg_decode_greedy. */
int qg_state_stream(const qg_state* s, qg_stream* out);
int qg_state_stats(const qg_state* s, qg_stats* out);
/* Token mask of the whole-token calls (the decode session's grammar mask,
 * applied between the lm_head GEMV and the in-graph argmax): `allow` is a
 * packed bitset of ceil(vocab/32) words, HOST memory; token i may be chosen
 * iff bit (i & 31) of allow[i >> 5] is set.  The logit of every other token
 * is replaced by -FLT_MAX before the first-index argmax (so with every token
 * banned the result is 0).  The mask lives in the state at a fixed device
 * address that the captured step reads on every replay: setting it takes
 * effect from the next step, needs no recapture and allocates nothing; the
 * copy is ordered with the state's steps and complete when the call returns.
 * n_words = 0 (allow may be NULL) clears the mask; qg_state_create and
 * qg_state_reset start with no mask.  Errors: QG_ERR_SHAPE when n_words is
 * neither 0 nor ceil(vocab/32), QG_ERR_ARG for a NULL state or mask. */
int qg_state_set_token_mask(qg_state* s, const uint32_t* allow, int n_words);

/* Batched prompt prefill (the decode session's batched prefill,
 * forward_qwen35_cuda.rs): tokens[0..n_tokens) (HOST) at positions
 * pos0..pos0+n_tokens-1 go through the layers in chunks of up to 1024 tokens,
 * each projection one multi-token GEMM (weights read once per chunk), the conv
 * and delta-rule recurrences token by token inside one kernel per layer, and
 * causal attention over cache rows 0..pos for each token.  It leaves the state
 * a token-by-token decode of the same tokens leaves (conv windows, recurrent
 * states, K/V rows in the state's cache format, the residual stream of the
 * last token, kv_len >= pos0 + n_tokens) and writes to *next_token the argmax
 * of the last token's logits (under the state's token mask): the first
 * generated token, to be fed to qg_decode_token at position pos0 + n_tokens.
 * The first call on a state allocates its scratch, kept until
 * qg_state_destroy (later calls allocate nothing): about 1024 x (3 hidden +
 * ffn + max(ffn, w) + w + q_dim + 2 kv_dim + ...) floats plus the K-split
 * partial sums (per buffer, the largest split layout of the projections that
 * write it, from the split rule), w the widest fused input projection:
 * ~0.5 GB at the 4B shape.  Synchronous.
 * Errors: QG_ERR_ARG (NULL, or a state of another model), QG_ERR_SHAPE
 * (n_tokens < 1, head_k_dim != 128, a GQA group other than 1, 2, 4),
 * QG_ERR_POS (positions past the cache), QG_ERR_TOKEN, QG_ERR_OOM,
 * QG_ERR_CUDA, QG_ERR_TIMEOUT. */
int qg_prefill(qg_model* m, qg_state* s, const uint32_t* tokens, int n_tokens, int pos0, uint32_t* next_token);

/* Batched decode of n sequences in lockstep (the decode session's batched
 * decode, forward_qwen35_cuda.rs): token tokens[i] of the sequence held by
 * states[i] at position positions[i], for n distinct states of this model with
 * one KV cache format; writes each sequence's next token (the argmax of its
 * logits under its own token mask) to next_tokens[i] and leaves each state as
 * qg_decode_token would.  The projections read every weight once per step for
 * all n sequences (n <= 4: a small-batch dequantizing GEMV, 4 multiply-adds per
 * weight read; more: the prefill GEMM); the conv, delta rule and attention run
 * per sequence on its own state; the lm_head runs once per sequence.  Runs on
 * states[0]'s stream with its prefill scratch (made by the first call).
 * Synchronous.  Errors: QG_ERR_ARG (NULL, a state of another model, one state
 * twice, KV formats that differ), QG_ERR_SHAPE (n outside 1..16, head_k_dim !=
 * 128), QG_ERR_TOKEN, QG_ERR_POS, QG_ERR_OOM, QG_ERR_CUDA, QG_ERR_TIMEOUT. */
int qg_decode_batch(qg_model* m, qg_state* const* states, int n, const uint32_t* tokens, const int* positions,
                    uint32_t* next_tokens);

/* The same lockstep decode for a fixed set of sequences through one captured
 * CUDA graph: qg_batch_create records the states (n distinct states of m, one
 * KV format; they must outlive the batch, and their streams are not used
 * meanwhile by other calls); each qg_batch_step copies the n tokens and
 * positions in from pinned memory, replays the step (captured on the first
 * call; positions are read on the device, so any valid positions replay) and
 * copies the n tokens out.  Results are those of qg_decode_batch.  Errors: as
 * qg_decode_batch. */
typedef struct qg_batch qg_batch;
int qg_batch_create(qg_model* m, qg_state* const* states, int n, qg_batch** out);
int qg_batch_step(qg_batch* b, const uint32_t* tokens, const int* positions, uint32_t* next_tokens);
int qg_batch_destroy(qg_batch* b);


/* ------------------------------------------------------- building blocks
 * Device pointers, the caller's stream, no allocation, no synchronisation. */

/* y[n] = sum_k deq(W[n][k]) * x[k] (forward_qwen35_cuda.rs gemv_dispatch,
 * float variant).  x enters as a 24-bit block-fixed-point value: each element
 * to within 2^-23 of the largest magnitude of its 256-element block (the
 * precision of f32 for that largest element); sub-block sums are exact
 * integers, accumulated in f32.
 * w: Q4_K, raw GGUF layout, 16-byte aligned.  x: [k] f32.  y: [n] f32.
 * k a multiple of 256 up to 16384 else QG_ERR_SHAPE; n == 0 or k == 0 ->
 * QG_ERR_EMPTY. */
int qg_gemv_q4k(const void* w, const float* x, float* y, int n, int k, qg_stream stream);

/* Planar Q4_K, the layout the model's Q4_K projections are streamed from:
 * n8 = n rounded up to 8 rows, nb = k/256; for every 8-row group g and
 * super-block b one 1152-byte group-block holding the 8 rows' GGUF blocks of
 * super-block b in row order (144 bytes each; rows n..n8-1 zero), stored
 * slice-major as the planar Q6_K below: group-block (g, b) at
 * ((n8/8)*b0 + g*kb + (b - b0))*1152 for the slice [b0, b0 + kb) holding b.
 * qg_q4k_planar_bytes gives the size (n8*nb*144, 0 for a bad shape);
 * qg_q4k_to_planar repacks a raw GGUF tensor (both device pointers, dst
 * 16-byte aligned); qg_gemv_q4k_planar is qg_gemv_q4k on that layout, the
 * model's own GEMV path. */
size_t qg_q4k_planar_bytes(int n, int k);
int qg_q4k_to_planar(const void* src, void* dst, int n, int k, qg_stream stream);
int qg_gemv_q4k_planar(const void* w_planar, const float* x, float* y, int n, int k, qg_stream stream);

/* y[n] = sum_k deq(W[n][k]) * x[k] for Q6_K (forward_qwen35_cuda.rs
 * gemv_dispatch, float variant), straight from raw GGUF rows: w holds n rows
 * of k/256 210-byte blocks (ql[128], qh[64], int8 scales[16], fp16 d) exactly
 * as the file stores them, 2-byte aligned; x: [k] f32, 16-byte aligned; y:
 * [n] f32, 4-byte aligned.  Plain f32 arithmetic: every product w_k x_k
 * passes through at most k/256 + 13 roundings (an 8-term sum per sub-block
 * half, the block accumulation, the warp tree; d * scale is exact), so
 * |y - y_exact| <= (k/256 + 16) 2^-24 sum_k |w_k x_k|.
 * k a multiple of 256 else QG_ERR_SHAPE (no upper limit); n == 0 or k == 0
 * -> QG_ERR_EMPTY; NULL or misaligned pointers -> QG_ERR_ARG. */
int qg_gemv_q6k(const void* w, const float* x, float* y, int n, int k, qg_stream stream);

/* The same product on the library's planar Q6_K layout (made by
 * qg_q6k_to_planar), the model's own GEMV path: the GEMV engine with x in
 * 24-bit block fixed point, as qg_gemv_q4k.  w_planar 16-byte aligned; k a
 * multiple of 256 up to 16384 else QG_ERR_SHAPE. */
int qg_gemv_q6k_planar(const void* w_planar, const float* x, float* y, int n, int k, qg_stream stream);

/* Planar Q6_K (the layout the GEMV engine streams): n8 = n rounded up to 8
 * rows, nb = k/256.  For every 8-row group g and super-block b one 1680-byte
 * group-block holding exactly the GGUF bytes of those 8 blocks, rearranged:
 * for row rr (0..7) and 64-weight quarter cq = 2*half + part (0..3), u =
 * 4*rr + cq, a 48-byte record at 48*u: ql[64*half + 16*part .. +16],
 * ql[64*half + 32 + 16*part .. +16], qh[16*cq .. +16]; the quarter's four
 * int8 scales sc[8*half + part + 2*s], s = 0..3, at 1536 + 4*u; the row's
 * fp16 d at 1664 + 2*rr.  Group-blocks
 * are stored slice-major: K splits into slices of 8 super-blocks, then of 4,
 * 2 and 1 for the remainder (its binary digits, in that order); slice
 * [b0, b0 + kb) takes (n8/8)*kb group-blocks from offset (n8/8)*b0*1680, with
 * group-block (g, b) at ((n8/8)*b0 + g*kb + (b - b0))*1680.  Rows n..n8-1 are
 * zero.  qg_q6k_planar_bytes gives the size (n8*nb*210); src is the raw GGUF
 * tensor and both are device pointers, 16-byte aligned. */
size_t qg_q6k_planar_bytes(int n, int k);
int qg_q6k_to_planar(const void* src, void* dst, int n, int k, qg_stream stream);

/* Fused lm_head GEMV + argmax (forward_qwen35_cuda.rs forward_single tail;
 * aprender PR #4332 greedy argmax): *tok_dev = min{ i : l_i = max_j l_j },
 * l = W x, no bias, logits never stored.  NaN logits never win; if all are
 * NaN the result is 0.  w: planar Q6_K [n_vocab x k].  workspace: device,
 * qg_lmhead_argmax_workspace_bytes() bytes, zero-filled before the first
 * call; every call leaves it zero-filled; calls sharing a workspace must not
 * overlap on the GPU. */
size_t qg_lmhead_argmax_workspace_bytes(void);
int qg_lmhead_argmax(const void* w_planar, const float* x, int n_vocab, int k, void* workspace,
                     uint32_t* tok_dev, qg_stream stream);

/* qg_lmhead_argmax with its workspace in the library's static device memory
 * (16 of 256 bytes per device): no allocation of any kind, no workspace
 * argument; same arguments, result and errors otherwise.  For callers that
 * must not allocate (device memory reserved up front by a pool; a loop on a
 * latency budget, where an allocation call can synchronise the device).  The
 * first call on each device (the device current at the call) resolves the
 * scratch address (cudaGetSymbolAddress, which may load the library's device
 * code): make that first call before any stream capture.  The scratch is zero
 * when the library loads and every call leaves it zeroed, so no call clears it
 * first.  There is one scratch per device, so calls on one device must not
 * overlap on the GPU (two streams at once race on it).  The pages have no
 * counterpart of this entry point.  Errors: those of qg_lmhead_argmax,
 * QG_ERR_CUDA when the scratch cannot be resolved, QG_ERR_SHAPE if the
 * kernel's workspace ever outgrew the static area. */
int qg_lmhead_argmax_noalloc(const void* w_planar, const float* x, int n_vocab, int k, uint32_t* tok_dev,
                             qg_stream stream);

/* First index of the maximum of x[n] (NaN never wins; all NaN gives 0) ->
 * *idx_dev: the device argmax of aprender PR #4332 ("Greedy GPU argmax",
 * first index on ties) over logits the caller already holds.  x and idx_dev
 * 4-byte aligned device pointers.  Errors: QG_ERR_ARG, QG_ERR_EMPTY. */
int qg_argmax_f32(const float* x, int n, uint32_t* idx_dev, qg_stream stream);

/* One Gated DeltaNet layer (forward_qwen35_cuda.rs forward_deltanet_layer)
 * on hidden_dev [hidden], in place; the layer's conv window and recurrent
 * state advance one step.  No position: the caller feeds steps in order.
 * Errors: QG_ERR_LAYER_KIND, QG_ERR_ARG, QG_ERR_CUDA. */
int qg_deltanet_step(const qg_model* m, qg_state* s, int il, float* hidden_dev, qg_stream stream);

/* One full-attention layer (forward_qwen35_cuda.rs forward_attention_layer)
 * on hidden_dev at `pos`: K/V rows land at pos, attention covers rows
 * 0..pos, kv_len = max(kv_len, pos + 1).  Errors: QG_ERR_POS,
 * QG_ERR_LAYER_KIND, QG_ERR_ARG, QG_ERR_CUDA. */
int qg_attn_decode_step(const qg_model* m, qg_state* s, int il, float* hidden_dev, int pos,
                        qg_stream stream);

/* ----------------------------------------------------------- whole token */

/* One token at `pos` through every layer, the output norm and the fused
 * lm_head + argmax, replayed as one CUDA graph captured on the first call
 * (memra decode.rs GraphSession::step): 8 bytes host-to-device (token,
 * pos), 4 bytes device-to-host (the token id), no allocation after the first
 * call.  Blocks until *next_token is on the host.  Positions of DeltaNet
 * layers advance per call, so feed pos = 0, 1, 2, ... in order.
 * Errors: QG_ERR_TOKEN, QG_ERR_POS, QG_ERR_TIMEOUT, QG_ERR_CUDA. */
int qg_decode_token(qg_model* m, qg_state* s, uint32_t token, int pos, uint32_t* next_token);

/* The same step enqueued kernel by kernel without a graph (bit-identical). */
int qg_decode_token_eager(qg_model* m, qg_state* s, uint32_t token, int pos, uint32_t* next_token);

/* Greedy continuation kept on the device: n_steps tokens from pos0, each
 * step's input the previous step's argmax (the first: the token the last
 * decode call produced), the position advanced on the device.  One graph
 * replay per token, no host round trip between them; tokens_host[n_steps]
 * receives the ids at the end.  Errors as qg_decode_token. */
int qg_decode_greedy(qg_model* m, qg_state* s, int pos0, int n_steps, uint32_t* tokens_host);

/* ----------------------------------------------------------- measurement */

/* The kernels of the decode step, one launch each per layer of their kind
 * (the lm_head once per token). */
enum {
    QG_KERNEL_DN_IN = 0,     /* DeltaNet: RMSNorm + fused qkv/alpha/beta/gate GEMV + conv/gates */
    QG_KERNEL_DELTA = 1,     /* DeltaNet: per-head L2 norm + gated delta rule */
    QG_KERNEL_SSM_OUT = 2,   /* DeltaNet: gated RMSNorm + ssm_out GEMV */
    QG_KERNEL_ATTN_IN = 3,   /* attention: RMSNorm + fused q|gate/k/v GEMV + V append */
    QG_KERNEL_ATTN = 4,      /* attention: q/k norm, rope, K append, split-K GQA attention, gate */
    QG_KERNEL_ATTN_OUT = 5,  /* attention: attn_output GEMV */
    QG_KERNEL_FFN_UP = 6,    /* every layer: RMSNorm + ffn_gate/ffn_up dual GEMV + SwiGLU */
    QG_KERNEL_FFN_DOWN = 7,  /* every layer: ffn_down (Q6_K) GEMV */
    QG_KERNEL_LMHEAD = 8     /* output RMSNorm + lm_head GEMV + first-index argmax */
};

/* Measurement hook (the pages have no counterpart): enqueue `launches`
 * launches of one kernel kind of the decode step on `stream`, chained by
 * programmatic dependent launch as inside the step, walking the layers that
 * have that kernel in index order, so that consecutive launches stream
 * different layers' weights from HBM as the step does.  Each launch runs with
 * exactly the arguments it has inside the step; the state's buffers are its
 * inputs and outputs, so the state's contents (windows, recurrent states, the
 * cache rows at its position, scratch) are meaningless afterwards: reset or
 * re-prefill it before decoding again.  Allocates nothing and can be captured
 * in a CUDA graph, which is how a caller times one kernel with events on
 * `stream`.  Errors: QG_ERR_ARG (NULL, launches < 1, or a kind the model does
 * not have), QG_ERR_CUDA. */
int qg_bench_kernel(const qg_model* m, qg_state* s, int kind, int launches, qg_stream stream);

/* Error word of the building blocks on the current device: QG_OK, or
 * QG_ERR_TIMEOUT when a building-block kernel gave up on a bounded wait since
 * the last check (the word is cleared).  Synchronous.  The pages have no
 * counterpart: their kernels do not wait on device flags. */
int qg_device_status(void);

/* Message of the last failed call on this thread ("" if none). */
const char* qg_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* QG_H */
