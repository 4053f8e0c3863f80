// Internal layout of qg_model / qg_state and the per-layer launchers.
#pragma once
#include <cuda.h>

#include <vector>

#include "qg_host.cuh"

// Device-resident weights of one layer.
struct qg_layer_dev {
    int kind;
    float* attn_norm;
    float* post_norm;
    uint8_t* w_in;   // fused input projection, Q4_K rows: DeltaNet [qkv | alpha | beta | gate],
                     // attention [q|gate per head | k | v]
    int n_in;
    uint8_t* w_out;  // ssm_out / attn_output, Q4_K
    uint8_t* w_gate; // Q4_K [ffn x hidden]
    uint8_t* w_up;
    uint8_t* w_down; // Q6_K planar [hidden x ffn]
    // Gated DeltaNet
    float* conv_w;   // [conv_dim][conv_kernel]
    float* a;        // -exp(A_log) [n_v_heads]
    float* dt_bias;
    float* ssm_norm; // [head_v_dim]
    // full attention
    float* q_norm;
    float* k_norm;
};

struct qg_model {
    qg_config cfg;
    std::vector<int32_t> kinds;
    int device;
    int k_dim, v_dim, conv_dim, q_dim, kv_dim;
    float theta_scale;
    std::vector<qg_layer_dev> layers;
    float* embd;
    float* out_norm;
    uint8_t* lm_head;  // Q6_K planar [vocab x hidden]
    std::vector<void*> allocs;
};

struct qg_state {
    const qg_model* m;
    int max_seq;
    int kv_len;
    cudaStream_t stream;
    int kv_format;                          // QG_KV_F32 or QG_KV_Q8_0_Q5_1, fixed at creation
    std::vector<float*> conv, ssm, kc, vc;  // per layer, null for the other kind; with a quantized
                                            // cache kc / vc hold q8_0 / q5_1 records (bytes)
    std::vector<CUtensorMap> kmap, vmap;    // f32 cache: 2-D tensor maps of kc / vc (attention layers)
    // scratch; h: the residual stream after the last step (the lm_head input
    // plus the last pending y), hres: the residual stream between layers, y:
    // the output of the last GEMV, not yet added
    float *h, *hres, *y, *conv_out, *dt, *beta, *z, *o, *act, *qf, *kraw, *vraw, *attn;
    float *part_acc, *part_ml;
    unsigned* attn_count;       // [n_kv_heads] split arrivals (left at 0)
    float* kpart;               // split-K GEMV slice sums [max slices][hidden8]
    // the pending GEMV output y: ycur_parts vectors ycur_stride floats apart
    // (split-K slice sums), summed in order by its reader
    const float* ycur;
    int ycur_parts, ycur_stride;
    unsigned long long* am_ws;  // lm_head argmax workspace (left at 0)
    int* slots;                 // device: [0] token in, [1] position, [2] token out (bit 31: device error)
    uint32_t* hist;             // device: greedy token per position [max_seq]
    uint32_t* allow;            // device: token mask, ceil(vocab/32) words, bit set = allowed (all set: none)
    unsigned* err;              // device error word
    int* pinned;                // pinned host: [0] token, [1] position, [2] token out
    void* pf;                   // batched prefill scratch (made by the first qg_prefill call), or null
    int keys_per_split, max_splits;
    cudaGraphExec_t exec_step;
    cudaGraphExec_t exec_greedy;
    qg_stats stats;
    std::vector<void*> allocs;
};

namespace qg {

// Makes `dev` current for a scope and restores the caller's device after it.
struct DeviceGuard {
    int prev = -1;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) cudaSetDevice(dev);
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

// Residual-stream buffers of one layer: the layer reads a (+ the pending
// state y when y_pending, or the embedding row of slots[0] when embed), keeps
// its intermediate stream in b, and leaves the stream in a with its last
// GEMV's output pending in the state's y.
struct ResidualIO {
    float* a;
    float* b;
    bool y_pending;
    bool embed;
};

// Enqueue one layer on `st`; `pdl_first` allows its first kernel to overlap
// the previous kernel on the stream.
int run_deltanet_layer(const qg_model* m, qg_state* s, int il, const ResidualIO& io, cudaStream_t st, bool pdl_first);
int run_attention_layer(const qg_model* m, qg_state* s, int il, const ResidualIO& io, cudaStream_t st,
                        bool pdl_first);
// `launches` PDL-chained launches of one kernel kind of the step (QG_KERNEL_*),
// round robin over the layers that have it (measurement; the state's contents
// become meaningless).
int run_kernel_kind(const qg_model* m, qg_state* s, int kind, int launches, cudaStream_t st);
// h += the pending y (closes a layer run on its own).
int run_residual(qg_state* s, float* h, int n, cudaStream_t st);
// Output norm of a + y (stored to h_final) + fused lm_head GEMV + argmax ->
// slots[0] / slots[2]; `advance` also records hist[pos] and moves slots[1].
int run_lmhead(const qg_model* m, qg_state* s, const float* a, float* h_final, cudaStream_t st, bool advance);
// Output norm of a + fused lm_head GEMV + argmax, no pending y, no advance.
int run_lmhead_of(const qg_model* m, qg_state* s, const float* a, cudaStream_t st);
// Quantized-cache records of positions pos0..pos0+rows-1 (see kv_quantize_rows).
int kv_quantize_rows_at(const float* k, const float* v, int rows, int pos0, int n_kv, int max_seq, uint8_t* kq,
                        uint8_t* vq, cudaStream_t st);
// Free the batched-prefill scratch descriptor (its device buffers are in s->allocs).
void prefill_release(qg_state* s);
// The same with the first position read on the device (*pos0_dev; rows must be
// within the cache, which the caller checks on the host).
int kv_quantize_rows_dev(const float* k, const float* v, int rows, const int* pos0_dev, int n_kv, int max_seq,
                         uint8_t* kq, uint8_t* vq, cudaStream_t st);
// f32 cache: the 2-D tensor maps of every attention layer's K and V cache
// ([max_seq] rows of kv_dim floats; box: one head's 256 floats x the
// attention's keys per stage), for its tensor copies.
int encode_kv_maps(qg_state* s);
// Raw GGUF Q4_K rows -> the engine's grouped layout ((n+7)/8*8 x k/256 x 144 bytes).
int q4k_to_grouped(const void* src, void* dst, int n, int k, cudaStream_t st);
// Quantized-cache rows from f32 K/V rows ([rows][n_kv*256] each): the records
// of positions 0..rows-1 of every kv head, made by the append's quantizer.
int kv_quantize_rows(const float* k, const float* v, int rows, int n_kv, int max_seq, uint8_t* kq, uint8_t* vq,
                     cudaStream_t st);
// Bytes of one layer's K or V cache (which: 0 = K, 1 = V).
size_t kv_cache_bytes(const qg_state* s, int which);
// a = -exp(A_log) on the device.
int run_neg_exp(const float* src, float* dst, int n, cudaStream_t st);

}  // namespace qg
