/*
 * CPU ORACLE for the batch-1 hybrid Gated-DeltaNet / full-attention decode
 * step.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the timed
 * CPU baseline of bench.py call it; the CUDA library never does.  It shares no
 * code, header or constant with the CUDA path.
 *
 * What it computes is the op order that forward_qwen35_cuda.rs (aprender-serve
 * 0.68.2, module documentation) states as the specification:
 *
 *   Gated DeltaNet layer: rms_norm -> attn_qkv GEMV -> causal_conv1d(+SiLU)
 *     -> split q|k|v -> per-head L2 on q,k -> ssm_alpha/ssm_beta GEMV
 *     -> dt/beta gates -> attn_gate GEMV -> delta rule -> gated rmsnorm
 *     -> ssm_out GEMV -> residual -> post_attention_norm -> SwiGLU FFN
 *     -> residual
 *   full-attention layer: rms_norm -> attn_q|attn_k|attn_v GEMV -> split
 *     q|gate -> per-head RMSNorm on q and k -> partial NEOX rope on q and k
 *     -> KV append at `position` -> GQA decode attention -> sigmoid gate
 *     -> attn_output GEMV -> residual -> post_attention_norm -> SwiGLU FFN
 *     -> residual
 *   token: embedding row -> every layer -> output rms_norm -> lm_head GEMV
 *     (no bias) -> argmax, first index of the maximum (aprender PR #4332, the
 *     greedy argmax on the GPU).
 *
 * Precision is the page's: weights dequantized to f32, f32 accumulation in
 * natural index order (the CPU reference of forward_qwen35_cuda.rs,
 * pin_reference_gemv, dequantizes to f32 and sums in f32).  An f64-accumulating
 * GEMV is kept for the error-bound pins (attn_q_gemv_of_host_input there).
 * Row loops may run on several OpenMP threads; each row's sum stays
 * sequential, so the thread count never changes a result.
 *
 * Readings taken where the pages are silent are listed beside each function.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ types */

enum { OR_Q4_K = 12, OR_Q6_K = 14 };
enum { OR_DELTANET = 0, OR_ATTENTION = 1 };

typedef struct {
    int n_layers, hidden, ffn, vocab;
    int n_k_heads, n_v_heads, head_k_dim, head_v_dim, conv_kernel;
    int n_heads, n_kv_heads, head_dim, n_rot;
    float eps, rope_theta;
    int max_seq_len;
} or_config;

typedef struct {
    const uint8_t* data; /* raw GGUF blocks, row-major */
    int qtype, n, k;
} or_qt;

typedef struct {
    int kind;
    const float *attn_norm, *post_norm;
    or_qt ffn_gate, ffn_up, ffn_down;
    /* Gated DeltaNet */
    const float *conv1d, *a_log, *dt_bias, *ssm_norm;
    or_qt qkv, alpha, beta, gate, ssm_out;
    /* full attention */
    const float *q_norm, *k_norm;
    or_qt wq, wk, wv, wo;
} or_layer;

typedef struct {
    or_config cfg;
    const float* embd;     /* [vocab][hidden] */
    const float* out_norm; /* [hidden] */
    or_qt lm_head;
    const or_layer* layers;
} or_model;

enum { OR_KV_F32 = 0, OR_KV_Q8_0_Q5_1 = 1 };

typedef struct {
    float** conv; /* per layer: [conv_dim][conv_kernel-1], or NULL */
    float** ssm;  /* per layer: [n_v_heads][head_v_dim][head_k_dim], or NULL */
    float** kc;   /* per layer: [max_seq_len][n_kv_heads*head_dim], or NULL; with a
                     quantized cache, the dequantized values of kq */
    float** vc;
    int kv_len;
    int kv_format; /* OR_KV_F32, or OR_KV_Q8_0_Q5_1 (q8_0 K, q5_1 V) */
    uint8_t** kq;  /* per layer, quantized cache only: [max_seq_len][kvd/32] q8_0 blocks */
    uint8_t** vq;  /* per layer, quantized cache only: [max_seq_len][kvd/32] q5_1 blocks */
} or_state;

void or_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int or_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------- k-quant decode */

/* IEEE 754 binary16 -> binary32. */
float or_f16(uint16_t h) {
    int sign = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
    float v;
    if (e == 0) v = ldexpf((float)m, -24);
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexpf((float)(1024 + m), e - 25);
    return sign ? -v : v;
}

static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/*
 * Q4_K super-block, 256 weights in 144 bytes (the GGUF k-quant layout; the
 * pages name the type, forward_qwen35_cuda.rs pin_float_gemv and aprender PR
 * #4332, and the layout is the public format's):
 *   bytes 0-1 fp16 d, 2-3 fp16 dmin, 4-15 eight 6-bit scales sc_j and eight
 *   6-bit mins m_j, 16-143 the 4-bit quants.
 *   Weight i of sub-block j (32 weights) = d*sc_j*q - dmin*m_j.
 *   Quant byte 32g+l holds weight 64g+l (low nibble, sub-block 2g) and weight
 *   64g+32+l (high nibble, sub-block 2g+1).
 *   Scale bytes s[0..11]: for j < 4, sc_j = s[j] & 63 and m_j = s[j+4] & 63;
 *   for j >= 4, sc_j = (s[j+4] & 15) | (s[j-4] >> 6) << 4 and
 *   m_j = (s[j+4] >> 4) | (s[j] >> 6) << 4.
 */
void or_q4k_scale_min(const uint8_t* s, int j, int* sc, int* m) {
    if (j < 4) {
        *sc = s[j] & 63;
        *m = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        *m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

void or_dequant_q4k_block(const uint8_t* b, float* out) {
    float d = or_f16(rd16(b)), dmin = or_f16(rd16(b + 2));
    const uint8_t* s = b + 4;
    const uint8_t* qs = b + 16;
    for (int g = 0; g < 4; g++) {
        int sc0, m0, sc1, m1;
        or_q4k_scale_min(s, 2 * g, &sc0, &m0);
        or_q4k_scale_min(s, 2 * g + 1, &sc1, &m1);
        float d0 = d * (float)sc0, mm0 = dmin * (float)m0;
        float d1 = d * (float)sc1, mm1 = dmin * (float)m1;
        for (int l = 0; l < 32; l++) {
            uint8_t q = qs[32 * g + l];
            out[64 * g + l] = d0 * (float)(q & 15) - mm0;
            out[64 * g + 32 + l] = d1 * (float)(q >> 4) - mm1;
        }
    }
}

/*
 * Q6_K super-block, 256 weights in 210 bytes (qualia resident_decode.rs pins
 * 2520 bytes for a 3072-wide Q6_K logits row, i.e. 210 per 256):
 *   bytes 0-127 low 4 bits, 128-191 high 2 bits, 192-207 sixteen int8
 *   scales (one per 16 weights), 208-209 fp16 d.
 *   Weight = d * scale * (q - 32), q = 6-bit.
 *   In half h (128 weights) and for l < 32: ql[64h+l] low nibble -> weight
 *   128h+l, ql[64h+32+l] low -> 128h+32+l, ql[64h+l] high -> 128h+64+l,
 *   ql[64h+32+l] high -> 128h+96+l; bit pair 2s of qh[32h+l] is the top of
 *   quarter s; weight 128h+32s+l uses scale 8h + l/16 + 2s.
 */
void or_dequant_q6k_block(const uint8_t* b, float* out) {
    const uint8_t* ql = b;
    const uint8_t* qh = b + 128;
    const int8_t* sc = (const int8_t*)(b + 192);
    float d = or_f16(rd16(b + 208));
    for (int h = 0; h < 2; h++) {
        for (int l = 0; l < 32; l++) {
            int is = l / 16;
            int q0 = (ql[64 * h + l] & 15) | (((qh[32 * h + l] >> 0) & 3) << 4);
            int q1 = (ql[64 * h + l + 32] & 15) | (((qh[32 * h + l] >> 2) & 3) << 4);
            int q2 = (ql[64 * h + l] >> 4) | (((qh[32 * h + l] >> 4) & 3) << 4);
            int q3 = (ql[64 * h + l + 32] >> 4) | (((qh[32 * h + l] >> 6) & 3) << 4);
            out[128 * h + l] = (d * (float)sc[8 * h + is + 0]) * (float)(q0 - 32);
            out[128 * h + l + 32] = (d * (float)sc[8 * h + is + 2]) * (float)(q1 - 32);
            out[128 * h + l + 64] = (d * (float)sc[8 * h + is + 4]) * (float)(q2 - 32);
            out[128 * h + l + 96] = (d * (float)sc[8 * h + is + 6]) * (float)(q3 - 32);
        }
    }
}

int or_block_bytes(int qtype) { return qtype == OR_Q4_K ? 144 : qtype == OR_Q6_K ? 210 : 0; }

void or_dequant_row(or_qt w, int r, float* out) {
    int nb = w.k / 256, bb = or_block_bytes(w.qtype);
    const uint8_t* row = w.data + (size_t)r * nb * bb;
    for (int b = 0; b < nb; b++) {
        if (w.qtype == OR_Q4_K) or_dequant_q4k_block(row + (size_t)b * bb, out + 256 * b);
        else or_dequant_q6k_block(row + (size_t)b * bb, out + 256 * b);
    }
}

/* ------------------------------------------------------------------ GEMV */

/* y[n] = sum_k deq(W[n,k]) * x[k], f32 accumulation in k order
 * (forward_qwen35_cuda.rs gemv_dispatch, float "mwv" variant). */
void or_gemv(or_qt w, const float* x, float* y) {
    #pragma omp parallel
    {
        float* row = (float*)malloc(sizeof(float) * (size_t)w.k);
        #pragma omp for schedule(static)
        for (int r = 0; r < w.n; r++) {
            or_dequant_row(w, r, row);
            float acc = 0.0f;
            for (int i = 0; i < w.k; i++) acc += row[i] * x[i];
            y[r] = acc;
        }
        free(row);
    }
}

/* The same product accumulated in f64 (attn_q_gemv_of_host_input: both
 * sides against an exact dequantized reference). */
void or_gemv_f64(or_qt w, const float* x, double* y) {
    #pragma omp parallel
    {
        float* row = (float*)malloc(sizeof(float) * (size_t)w.k);
        #pragma omp for schedule(static)
        for (int r = 0; r < w.n; r++) {
            or_dequant_row(w, r, row);
            double acc = 0.0;
            for (int i = 0; i < w.k; i++) acc += (double)row[i] * (double)x[i];
            y[r] = acc;
        }
        free(row);
    }
}

/* Rows [r0, r0 + cnt) only: the full-size parity tests sample rows. */
void or_gemv_rows(or_qt w, const float* x, const int* rows, int cnt, float* y) {
    #pragma omp parallel
    {
        float* row = (float*)malloc(sizeof(float) * (size_t)w.k);
        #pragma omp for schedule(static)
        for (int t = 0; t < cnt; t++) {
            or_dequant_row(w, rows[t], row);
            float acc = 0.0f;
            for (int i = 0; i < w.k; i++) acc += row[i] * x[i];
            y[t] = acc;
        }
        free(row);
    }
}

/* ------------------------------------------------------- elementwise ops */

float or_silu(float x) { return x / (1.0f + expf(-x)); }
float or_sigmoid(float x) { return 1.0f / (1.0f + expf(-x)); }
/* softplus in the overflow-free form max(x,0) + log1p(exp(-|x|)) (reading:
 * the gates see |x| of order 100 with random weights). */
float or_softplus(float x) { return fmaxf(x, 0.0f) + log1pf(expf(-fabsf(x))); }

/* y = x * rsqrt(mean(x^2) + eps) * w  (rmsnorm_into). */
void or_rmsnorm(const float* x, const float* w, float* y, int n, float eps) {
    float ss = 0.0f;
    for (int i = 0; i < n; i++) ss += x[i] * x[i];
    float r = 1.0f / sqrtf(ss / (float)n + eps);
    for (int i = 0; i < n; i++) y[i] = (x[i] * r) * w[i];
}

/* Per-head L2 norm on dk-wide heads, in place: x * rsqrt(sum x^2 + eps)
 * (gdn_per_head_l2_norm_into). */
void or_l2norm_heads(float* x, int dk, int nheads, float eps) {
    for (int h = 0; h < nheads; h++) {
        float* v = x + (size_t)h * dk;
        float ss = 0.0f;
        for (int i = 0; i < dk; i++) ss += v[i] * v[i];
        float r = 1.0f / sqrtf(ss + eps);
        for (int i = 0; i < dk; i++) v[i] = v[i] * r;
    }
}

/*
 * Causal depthwise conv1d + SiLU with the window rolled in place
 * (gdn_causal_conv1d_silu_into; memra ssm_conv1d_fused_decode assembles
 * [window | new column], convolves and rolls).  Reading: no conv bias (none is
 * uploaded); window stored [C][K-1], oldest first; tap K-1 multiplies the new
 * input.
 */
void or_conv1d_silu(const float* xin, float* win, const float* wconv, float* out, int C, int K) {
    for (int c = 0; c < C; c++) {
        float* wc = win + (size_t)c * (K - 1);
        const float* kw = wconv + (size_t)c * K;
        float acc = 0.0f;
        for (int t = 0; t < K - 1; t++) acc += kw[t] * wc[t];
        acc += kw[K - 1] * xin[c];
        out[c] = or_silu(acc);
        for (int t = 0; t < K - 2; t++) wc[t] = wc[t + 1];
        wc[K - 2] = xin[c];
    }
}

/* dt = softplus(alpha + dt_bias) * a, beta = sigmoid(beta_raw)
 * (gdn_gates_into).  a = -exp(A_log) is formed by the caller. */
void or_gates(const float* alpha, const float* dt_bias, const float* a, const float* beta_raw,
              float* dt, float* beta, int nv) {
    for (int h = 0; h < nv; h++) {
        dt[h] = or_softplus(alpha[h] + dt_bias[h]) * a[h];
        beta[h] = or_sigmoid(beta_raw[h]);
    }
}

/*
 * Gated delta rule, one decode step (gdn_delta_rule_into; memra
 * gdn_scan_s128 with scale = 1/sqrt(d_state)).  Value head h reads key head
 * h % nk (check_head_grouping).  State of head h: dv rows of dk,
 * s[j*dk + i] == S[i][j] (build_state).  For every row j:
 *   r = g * S[:, j],  g = exp(dt_h)          decay
 *   d = beta_h * (v_j - r . k)               read
 *   S[:, j] = r + k * d                      rank-1 update
 *   o_j = (S[:, j] . q) / sqrt(dk)           query of the updated state
 */
void or_delta_rule(const float* q, const float* k, const float* v, const float* beta,
                   const float* dt, float* S, float* o, int nk, int dk, int nv, int dv) {
    float scale = 1.0f / sqrtf((float)dk);
    float* r = (float*)malloc(sizeof(float) * (size_t)dk);
    for (int h = 0; h < nv; h++) {
        int kh = h % nk;
        const float* qh = q + (size_t)kh * dk;
        const float* kk = k + (size_t)kh * dk;
        float g = expf(dt[h]);
        for (int j = 0; j < dv; j++) {
            float* s = S + ((size_t)h * dv + j) * dk;
            for (int i = 0; i < dk; i++) r[i] = g * s[i];
            float dot = 0.0f;
            for (int i = 0; i < dk; i++) dot += r[i] * kk[i];
            float d = beta[h] * (v[(size_t)h * dv + j] - dot);
            for (int i = 0; i < dk; i++) s[i] = r[i] + kk[i] * d;
            float oq = 0.0f;
            for (int i = 0; i < dk; i++) oq += s[i] * qh[i];
            o[(size_t)h * dv + j] = oq * scale;
        }
    }
    free(r);
}

/* Per value head: u = rmsnorm(o_h) * w * silu(z_h), w shared by the heads
 * (gdn_gated_rmsnorm_into; memra gated_rmsnorm normalises each value-head row).  Reading:
 * the gate activation is SiLU. */
void or_gated_rmsnorm(const float* o, const float* z, const float* w, float* u, int dv, int nv,
                      float eps) {
    for (int h = 0; h < nv; h++) {
        const float* oh = o + (size_t)h * dv;
        float ss = 0.0f;
        for (int j = 0; j < dv; j++) ss += oh[j] * oh[j];
        float r = 1.0f / sqrtf(ss / (float)dv + eps);
        for (int j = 0; j < dv; j++)
            u[(size_t)h * dv + j] = ((oh[j] * r) * w[j]) * or_silu(z[(size_t)h * dv + j]);
    }
}

/* act = silu(gate) * up (fused_swiglu_into). */
void or_swiglu(const float* g, const float* up, float* act, int n) {
    for (int i = 0; i < n; i++) act[i] = or_silu(g[i]) * up[i];
}

/* Split the joint [q | gate] projection, per head 2*hd wide, q first
 * (gdn_split_interleaved_into). */
void or_split_q_gate(const float* qf, float* q, float* gate, int nh, int hd) {
    for (int h = 0; h < nh; h++)
        for (int d = 0; d < hd; d++) {
            q[(size_t)h * hd + d] = qf[(size_t)h * 2 * hd + d];
            gate[(size_t)h * hd + d] = qf[(size_t)h * 2 * hd + hd + d];
        }
}

/* Per-head RMSNorm with one hd-wide weight (per_head_rmsnorm_into). */
void or_rmsnorm_heads(const float* x, const float* w, float* y, int hd, int nheads, float eps) {
    for (int h = 0; h < nheads; h++)
        or_rmsnorm(x + (size_t)h * hd, w, y + (size_t)h * hd, hd, eps);
}

/* theta_scale = rope_theta^(-2/n_rot) in f32, on the host
 * (forward_qwen35_cuda.rs dims_of). */
float or_theta_scale(float rope_theta, int n_rot) {
    return powf(rope_theta, -2.0f / (float)n_rot);
}

/*
 * Partial NEOX rope, in place, on every hd-wide head (gdn_partial_neox_rope_into):
 * pair i < n_rot/2 is (x_i, x_{i+n_rot/2}) rotated by theta_i; dims >= n_rot
 * are untouched.  Reading: theta_0 = pos and theta_{i+1} = theta_i *
 * theta_scale, an f32 running product of the host-computed scale.
 */
void or_rope_neox(float* x, int nheads, int hd, int n_rot, int pos, float theta_scale) {
    int half = n_rot / 2;
    for (int h = 0; h < nheads; h++) {
        float* v = x + (size_t)h * hd;
        float theta = (float)pos;
        for (int i = 0; i < half; i++) {
            float c = cosf(theta), s = sinf(theta);
            float a = v[i], b = v[i + half];
            v[i] = a * c - b * s;
            v[i + half] = a * s + b * c;
            theta = theta * theta_scale;
        }
    }
}

/*
 * GQA decode attention over cache rows 0..t-1 (gdn_decode_attention_into):
 * head h uses kv group h / (nh / nkv) (reading: contiguous groups),
 * out_h = sum_t softmax_t(q_h . K[t] / sqrt(hd)) * V[t].
 */
void or_attention(const float* q, const float* kc, const float* vc, float* out, int nh, int nkv,
                  int hd, int t_len) {
    int kvd = nkv * hd, grp = nh / nkv;
    float scale = 1.0f / sqrtf((float)hd);
    float* sc = (float*)malloc(sizeof(float) * (size_t)(t_len > 0 ? t_len : 1));
    for (int h = 0; h < nh; h++) {
        int g = h / grp;
        const float* qh = q + (size_t)h * hd;
        float m = -INFINITY;
        for (int t = 0; t < t_len; t++) {
            const float* kr = kc + (size_t)t * kvd + (size_t)g * hd;
            float dot = 0.0f;
            for (int d = 0; d < hd; d++) dot += qh[d] * kr[d];
            sc[t] = dot * scale;
            if (sc[t] > m) m = sc[t];
        }
        float l = 0.0f;
        for (int t = 0; t < t_len; t++) {
            sc[t] = expf(sc[t] - m);
            l += sc[t];
        }
        for (int d = 0; d < hd; d++) {
            float acc = 0.0f;
            for (int t = 0; t < t_len; t++) acc += sc[t] * vc[(size_t)t * kvd + (size_t)g * hd + d];
            out[(size_t)h * hd + d] = acc / l;
        }
    }
    free(sc);
}

/* ---------------------------------------------------- quantized KV cache */
/*
 * The decode session's quantized KV cache (forward_qwen35_cuda.rs, full
 * attention layer: K as q8_0 blocks and V as q5_1 blocks, appended by a
 * quantize kernel on the device, the attention reading the quantized bytes).
 * That source names the two GGML block types and nothing more; their contents here are what those
 * names denote in GGUF (reading):
 *   q8_0, 34 bytes per 32 values: f16 d, int8 q[32];            x = d*q
 *   q5_1, 24 bytes per 32 values: f16 d, f16 m, u32 qh, u8 qs[16];
 *         q_j = (qs nibble) | (bit j of qh) << 4, the low nibble of qs[j]
 *         holding q_j and the high nibble q_{j+16};            x = d*q + m
 * The quantizer (reading): d from the block's f32 statistics (q8_0:
 * max|x| / 127; q5_1: (max - min) / 31 with m = min), each code
 * roundf(x * (1/d)) -- q5_1: roundf((x - min) * (1/d)) -- in f32 with the
 * f32 d (half away from zero), clamped to the code range; a d below the
 * smallest normal f32 gives zero codes.  d and m are stored as f16 (round to
 * nearest even) and dequantization uses the stored values.  Every row the
 * attention reads, the appended one included, is the dequantized row.
 */

/* IEEE 754 binary32 -> binary16, round to nearest, ties to even. */
uint16_t or_f32_to_f16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t sign = (u >> 16) & 0x8000u, a = u & 0x7fffffffu;
    if (a >= 0x7f800000u) return (uint16_t)(sign | (a > 0x7f800000u ? 0x7e00u : 0x7c00u));
    if (a >= 0x477ff000u) return (uint16_t)(sign | 0x7c00u); /* >= 65520: past the largest finite half */
    int e = (int)(a >> 23) - 127;
    uint32_t h, rem, half;
    if (e >= -14) { /* a normal half: keep 10 of the 23 fraction bits */
        h = ((uint32_t)(e + 15) << 10) | ((a & 0x7fffffu) >> 13);
        rem = a & 0x1fffu;
        half = 0x1000u;
    } else { /* a subnormal half (units of 2^-24), or zero */
        if (e < -25) return (uint16_t)sign;
        uint32_t m = (a & 0x7fffffu) | 0x800000u; /* value = m * 2^(e-23) */
        int shift = -e - 1;                       /* 14 .. 24 */
        h = m >> shift;
        rem = m & ((1u << shift) - 1u);
        half = 1u << (shift - 1);
    }
    if (rem > half || (rem == half && (h & 1u))) h++; /* a carry moves into the exponent correctly */
    return (uint16_t)(sign | h);
}

void or_f32_to_f16_n(const float* x, int n, uint16_t* out) {
    for (int i = 0; i < n; i++) out[i] = or_f32_to_f16(x[i]);
}

static void wr16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)(v & 0xff); p[1] = (uint8_t)(v >> 8); }

/* The f32 values each code rounds: x/d for q8_0, (x - min)/d for q5_1, both
 * taken as a product with the f32 reciprocal of the f32 d (0 when d is below
 * the smallest normal f32).  which: 0 = q8_0, 1 = q5_1.  n a multiple of 32. */
void or_kv_prescaled(const float* x, int n, int which, float* pre) {
    for (int b = 0; b < n / 32; b++) {
        const float* xb = x + 32 * b;
        float lo = xb[0], hi = xb[0], amax = 0.0f;
        for (int j = 0; j < 32; j++) {
            lo = fminf(lo, xb[j]);
            hi = fmaxf(hi, xb[j]);
            amax = fmaxf(amax, fabsf(xb[j]));
        }
        float d = which == 0 ? amax / 127.0f : (hi - lo) / 31.0f;
        float id = d >= FLT_MIN ? 1.0f / d : 0.0f;
        for (int j = 0; j < 32; j++) pre[32 * b + j] = which == 0 ? xb[j] * id : (xb[j] - lo) * id;
    }
}

/* n values (a multiple of 32) -> n/32 q8_0 blocks of 34 bytes. */
void or_quantize_q8_0(const float* x, int n, uint8_t* out) {
    float pre[32];
    for (int b = 0; b < n / 32; b++) {
        const float* xb = x + 32 * b;
        uint8_t* ob = out + 34 * (size_t)b;
        float amax = 0.0f;
        for (int j = 0; j < 32; j++) amax = fmaxf(amax, fabsf(xb[j]));
        wr16(ob, or_f32_to_f16(amax / 127.0f));
        or_kv_prescaled(xb, 32, 0, pre);
        for (int j = 0; j < 32; j++) {
            float v = roundf(pre[j]);
            int q = v >= 127.0f ? 127 : v <= -127.0f ? -127 : (int)v;
            ob[2 + j] = (uint8_t)(int8_t)q;
        }
    }
}

void or_dequantize_q8_0(const uint8_t* in, int n, float* x) {
    for (int b = 0; b < n / 32; b++) {
        const uint8_t* ib = in + 34 * (size_t)b;
        float d = or_f16(rd16(ib));
        for (int j = 0; j < 32; j++) x[32 * b + j] = d * (float)(int8_t)ib[2 + j];
    }
}

/* n values (a multiple of 32) -> n/32 q5_1 blocks of 24 bytes. */
void or_quantize_q5_1(const float* x, int n, uint8_t* out) {
    float pre[32];
    for (int b = 0; b < n / 32; b++) {
        const float* xb = x + 32 * b;
        uint8_t* ob = out + 24 * (size_t)b;
        float lo = xb[0], hi = xb[0];
        for (int j = 0; j < 32; j++) {
            lo = fminf(lo, xb[j]);
            hi = fmaxf(hi, xb[j]);
        }
        wr16(ob, or_f32_to_f16((hi - lo) / 31.0f));
        wr16(ob + 2, or_f32_to_f16(lo));
        or_kv_prescaled(xb, 32, 1, pre);
        uint8_t q[32];
        uint32_t qh = 0;
        for (int j = 0; j < 32; j++) {
            float v = roundf(pre[j]);
            q[j] = (uint8_t)(v >= 31.0f ? 31 : v <= 0.0f ? 0 : (int)v);
            qh |= (uint32_t)((q[j] >> 4) & 1) << j;
        }
        for (int i = 0; i < 4; i++) ob[4 + i] = (uint8_t)(qh >> (8 * i));
        for (int j = 0; j < 16; j++) ob[8 + j] = (uint8_t)((q[j] & 15) | ((q[j + 16] & 15) << 4));
    }
}

void or_dequantize_q5_1(const uint8_t* in, int n, float* x) {
    for (int b = 0; b < n / 32; b++) {
        const uint8_t* ib = in + 24 * (size_t)b;
        float d = or_f16(rd16(ib)), m = or_f16(rd16(ib + 2));
        uint32_t qh = (uint32_t)ib[4] | ((uint32_t)ib[5] << 8) | ((uint32_t)ib[6] << 16) | ((uint32_t)ib[7] << 24);
        for (int j = 0; j < 32; j++) {
            int nib = j < 16 ? (ib[8 + j] & 15) : (ib[8 + j - 16] >> 4);
            int q = nib | (int)(((qh >> j) & 1u) << 4);
            x[32 * b + j] = d * (float)q + m;
        }
    }
}

/* x *= sigmoid(gate) (gdn_sigmoid_gate_into). */
void or_sigmoid_gate(float* x, const float* gate, int n) {
    for (int i = 0; i < n; i++) x[i] = x[i] * or_sigmoid(gate[i]);
}

/* First index of the maximum (the CPU argmax of aprender PR #4332; qualia
 * merges candidates by value, the smaller index winning a tie).  NaN never
 * wins; an all-NaN vector gives 0. */
int or_argmax(const float* x, int n) {
    int best = -1;
    float bv = 0.0f;
    for (int i = 0; i < n; i++) {
        if (isnan(x[i])) continue;
        if (best < 0 || x[i] > bv) { best = i; bv = x[i]; }
    }
    return best < 0 ? 0 : best;
}

/* Top two values of a vector (the margin of a greedy decision). */
void or_top2(const float* x, int n, float* v1, float* v2) {
    float a = -INFINITY, b = -INFINITY;
    for (int i = 0; i < n; i++) {
        if (isnan(x[i])) continue;
        if (x[i] > a) { b = a; a = x[i]; }
        else if (x[i] > b) b = x[i];
    }
    *v1 = a;
    *v2 = b;
}

/* ------------------------------------------------------------ the layers */

static float* fbuf(size_t n) { return (float*)calloc(n ? n : 1, sizeof(float)); }

/* One Gated DeltaNet layer on hidden state h, in place
 * (forward_qwen35_cuda.rs deltanet_layer_inner). */
void or_deltanet_layer(const or_model* M, or_state* st, int il, float* h) {
    const or_config* c = &M->cfg;
    const or_layer* L = &M->layers[il];
    int H = c->hidden, nv = c->n_v_heads, nk = c->n_k_heads, dk = c->head_k_dim,
        dv = c->head_v_dim;
    int kdim = nk * dk, vdim = nv * dv, C = 2 * kdim + vdim;
    float *xn = fbuf(H), *qkv = fbuf(C), *conv = fbuf(C), *al = fbuf(nv), *br = fbuf(nv),
          *a = fbuf(nv), *dt = fbuf(nv), *be = fbuf(nv), *z = fbuf(vdim), *o = fbuf(vdim),
          *u = fbuf(vdim), *y = fbuf(H), *g = fbuf(c->ffn), *up = fbuf(c->ffn),
          *act = fbuf(c->ffn);

    or_rmsnorm(h, L->attn_norm, xn, H, c->eps);
    or_gemv(L->qkv, xn, qkv);
    or_conv1d_silu(qkv, st->conv[il], L->conv1d, conv, C, c->conv_kernel);
    float *q = conv, *k = conv + kdim, *v = conv + 2 * kdim;
    or_l2norm_heads(q, dk, nk, c->eps);
    or_l2norm_heads(k, dk, nk, c->eps);
    or_gemv(L->alpha, xn, al);
    or_gemv(L->beta, xn, br);
    /* a = -exp(A_log) (reading: the stored vector is A_log) */
    for (int i = 0; i < nv; i++) a[i] = -expf(L->a_log[i]);
    or_gates(al, L->dt_bias, a, br, dt, be, nv);
    or_gemv(L->gate, xn, z);
    or_delta_rule(q, k, v, be, dt, st->ssm[il], o, nk, dk, nv, dv);
    or_gated_rmsnorm(o, z, L->ssm_norm, u, dv, nv, c->eps);
    or_gemv(L->ssm_out, u, y);
    for (int i = 0; i < H; i++) h[i] = h[i] + y[i];
    or_rmsnorm(h, L->post_norm, xn, H, c->eps);
    or_gemv(L->ffn_gate, xn, g);
    or_gemv(L->ffn_up, xn, up);
    or_swiglu(g, up, act, c->ffn);
    or_gemv(L->ffn_down, act, y);
    for (int i = 0; i < H; i++) h[i] = h[i] + y[i];

    free(xn); free(qkv); free(conv); free(al); free(br); free(a); free(dt); free(be);
    free(z); free(o); free(u); free(y); free(g); free(up); free(act);
}

/* One full-attention layer on h at `pos`, appending K/V at row pos
 * (forward_qwen35_cuda.rs attention_layer_inner). */
void or_attention_layer(const or_model* M, or_state* st, int il, float* h, int pos) {
    const or_config* c = &M->cfg;
    const or_layer* L = &M->layers[il];
    int H = c->hidden, nh = c->n_heads, nkv = c->n_kv_heads, hd = c->head_dim;
    int qd = nh * hd, kvd = nkv * hd;
    float *xn = fbuf(H), *qf = fbuf(2 * (size_t)qd), *q = fbuf(qd), *qn = fbuf(qd),
          *gate = fbuf(qd), *kraw = fbuf(kvd), *att = fbuf(qd), *y = fbuf(H),
          *g = fbuf(c->ffn), *up = fbuf(c->ffn), *act = fbuf(c->ffn);
    float* krow = st->kc[il] + (size_t)pos * kvd;
    float* vrow = st->vc[il] + (size_t)pos * kvd;
    float ts = or_theta_scale(c->rope_theta, c->n_rot);

    or_rmsnorm(h, L->attn_norm, xn, H, c->eps);
    or_gemv(L->wq, xn, qf);
    or_gemv(L->wk, xn, kraw);
    or_gemv(L->wv, xn, vrow);
    or_split_q_gate(qf, q, gate, nh, hd);
    or_rmsnorm_heads(q, L->q_norm, qn, hd, nh, c->eps);
    or_rmsnorm_heads(kraw, L->k_norm, krow, hd, nkv, c->eps);
    or_rope_neox(qn, nh, hd, c->n_rot, pos, ts);
    or_rope_neox(krow, nkv, hd, c->n_rot, pos, ts);
    if (st->kv_format == OR_KV_Q8_0_Q5_1) {
        /* quantize-on-append: row pos becomes its q8_0 (K) / q5_1 (V) blocks, and
           the attention reads it, like every older row, dequantized */
        uint8_t* kb = st->kq[il] + (size_t)pos * (size_t)(kvd / 32) * 34;
        uint8_t* vb = st->vq[il] + (size_t)pos * (size_t)(kvd / 32) * 24;
        or_quantize_q8_0(krow, kvd, kb);
        or_dequantize_q8_0(kb, kvd, krow);
        or_quantize_q5_1(vrow, kvd, vb);
        or_dequantize_q5_1(vb, kvd, vrow);
    }
    or_attention(qn, st->kc[il], st->vc[il], att, nh, nkv, hd, pos + 1);
    or_sigmoid_gate(att, gate, qd);
    or_gemv(L->wo, att, y);
    for (int i = 0; i < H; i++) h[i] = h[i] + y[i];
    or_rmsnorm(h, L->post_norm, xn, H, c->eps);
    or_gemv(L->ffn_gate, xn, g);
    or_gemv(L->ffn_up, xn, up);
    or_swiglu(g, up, act, c->ffn);
    or_gemv(L->ffn_down, act, y);
    for (int i = 0; i < H; i++) h[i] = h[i] + y[i];
    if (st->kv_len < pos + 1) st->kv_len = pos + 1;

    free(xn); free(qf); free(q); free(qn); free(gate); free(kraw); free(att); free(y);
    free(g); free(up); free(act);
}

/*
 * One whole token (forward_qwen35_cuda.rs forward_single; greedy twin
 * forward_single_greedy of aprender PR #4332): embedding row, every layer in
 * order, output norm, lm_head without bias, first-index argmax.  Writes the
 * final residual stream to hidden_out and the logits to logits_out when those
 * are non-NULL.  Returns the token id, or -1 for a token or position out of
 * range.
 */
int or_forward_token(const or_model* M, or_state* st, int token, int pos, float* hidden_out,
                     float* logits_out) {
    const or_config* c = &M->cfg;
    if (token < 0 || token >= c->vocab || pos < 0 || pos >= c->max_seq_len) return -1;
    int H = c->hidden;
    float *h = fbuf(H), *xn = fbuf(H);
    float* logits = logits_out ? logits_out : fbuf(c->vocab);
    memcpy(h, M->embd + (size_t)token * H, sizeof(float) * (size_t)H);
    for (int il = 0; il < c->n_layers; il++) {
        if (M->layers[il].kind == OR_DELTANET) or_deltanet_layer(M, st, il, h);
        else or_attention_layer(M, st, il, h, pos);
    }
    if (hidden_out) memcpy(hidden_out, h, sizeof(float) * (size_t)H);
    or_rmsnorm(h, M->out_norm, xn, H, c->eps);
    or_gemv(M->lm_head, xn, logits);
    if (st->kv_len < pos + 1) st->kv_len = pos + 1;
    int tok = or_argmax(logits, c->vocab);
    free(h); free(xn);
    if (!logits_out) free(logits);
    return tok;
}
