// Parameters of the persistent whole-step kernel (step.cu): the geometry of
// its GEMV phases, per-layer weight and state pointers, and the step's
// scratch buffers.  Passed by value as one __grid_constant__ kernel argument.
#pragma once
#include <cstdint>

#include "qg_gemv.cuh"

namespace qg {

constexpr int kStepMaxLayers = 64;
constexpr int kSlotBytes = 16 * 1024;      // one ring slot = one stage
constexpr int kStepMaxSlots = 8;           // the ring's mbarriers (16 * kMaxStages bytes)
constexpr int kStepSmemPerCta = 112 * 1024;  // two CTAs per SM

enum StepGemv { SG_DN_IN, SG_ATTN_IN, SG_SSM_OUT, SG_ATTN_OUT, SG_FFN_UP, SG_FFN_DOWN, SG_LMHEAD, SG_COUNT };

struct StepLayer {
    const uint8_t* w_in;
    const uint8_t* w_out;
    const uint8_t* w_gate;
    const uint8_t* w_up;
    const uint8_t* w_down;
    const float* attn_norm;
    const float* post_norm;
    const float* conv_w;
    const float* a;
    const float* dt_bias;
    const float* ssm_norm;
    const float* q_norm;
    const float* k_norm;
    float* conv;
    float* ssm;
    float* kc;
    float* vc;
    int kind;
};

struct StepParams {
    GemvShape geo[SG_COUNT];  // geometry of each GEMV phase (weights per layer below)
    StepLayer L[kStepMaxLayers];
    int n_layers, hidden, ffn, vocab, conv_dim, conv_k, nv, nk, dv, k_dim, v_dim, q_dim, kv_dim;
    int gs, n_kv, n_rot, T, max_splits;
    float eps, theta_scale;
    const float* embd;
    const float* out_norm;
    const uint8_t* lm_head;
    float *h, *hres, *y, *conv_out, *dt, *beta, *z, *o, *act, *qf, *kraw, *attn, *part_acc, *part_ml;
    unsigned* attn_count;
    unsigned long long* am_ws;
    int* slots;
    uint32_t* hist;
    const uint32_t* allow;
    unsigned* err;
    unsigned* gbar;  // [0] barrier arrivals, [1] CTAs finished, [2] abort (all zero between steps)
    int advance;     // greedy: record hist[pos] and move the position slot
    int nslots;      // ring slots per CTA
    int ring_off;    // byte offset of the ring in dynamic shared memory
};

}  // namespace qg
