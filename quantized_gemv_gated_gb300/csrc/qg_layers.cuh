// Device pieces shared by the per-layer kernels and the batched prefill: the
// epilogues of the fused input projections and of the lm_head argmax, the
// delta-rule row update, and the attention row helpers.
#pragma once
#include <cfloat>

#include "qg_internal.cuh"

namespace qg {

constexpr int kHd = 256;  // attention head_dim (the configs the kernels serve)

// ------------------------------------------------------------ epilogues
// DeltaNet input projection rows: [0, C) qkv -> conv; [C, C+nv) alpha;
// [C+nv, C+2nv) beta; [C+2nv, C+2nv+v_dim) z.  Each consumer thread owns rows
// r0 + tid, r0 + tid + 256, ...; the conv window and weights of its first row
// (state of the previous token, and constants) are loaded before the
// dependency wait.
constexpr int kMaxConvTaps = 8;
struct EpiDnIn : EpiBase {
    int C, nv, K;
    float* win;          // [C][K-1], oldest first
    const float* wconv;  // [C][K]
    float* conv_out;
    const float* dt_bias;
    const float* a;
    float* dt;
    float* beta;
    float* z;
    int pre_row;
    float pw[kMaxConvTaps], pwin[kMaxConvTaps], plast;
    __device__ void pre(int r0, int r1, int tid) {
        pre_row = r0 + tid;
        if (pre_row < r1 && pre_row < C) {
            const float* kw = wconv + static_cast<size_t>(pre_row) * K;
            const float* wc = win + static_cast<size_t>(pre_row) * (K - 1);
#pragma unroll
            for (int t = 0; t < kMaxConvTaps - 1; ++t) {
                if (t < K - 1) {
                    pw[t] = kw[t];
                    pwin[t] = __ldcg(wc + t);
                }
            }
            plast = kw[K - 1];
        }
    }
    __device__ void apply(int r0, int r1, const float* ys, const float*, int tid) {
        for (int r = r0 + tid; r < r1; r += kConsumers) row_out(r, ys[r - r0]);
    }
    __device__ void row_out(int r, float v) {
        if (r < C) {
            // causal conv1d + SiLU, then roll the window (gdn_causal_conv1d_silu_into)
            float* wc = win + static_cast<size_t>(r) * (K - 1);
            float acc = 0.0f;
            if (r == pre_row) {
#pragma unroll
                for (int t = 0; t < kMaxConvTaps - 1; ++t)
                    if (t < K - 1) acc += pw[t] * pwin[t];
#pragma unroll
                for (int t = 1; t < kMaxConvTaps - 1; ++t)
                    if (t < K - 1) wc[t - 1] = pwin[t];
                acc += plast * v;
            } else {
                const float* kw = wconv + static_cast<size_t>(r) * K;
                for (int t = 0; t < K - 1; ++t) {
                    const float wt = __ldcg(wc + t);
                    acc += kw[t] * wt;
                    if (t > 0) wc[t - 1] = wt;
                }
                acc += kw[K - 1] * v;
            }
            conv_out[r] = silu(acc);
            wc[K - 2] = v;
        } else if (r < C + nv) {
            const int h = r - C;  // dt = softplus(alpha + dt_bias) * a (gdn_gates_into)
            dt[h] = softplus(v + dt_bias[h]) * a[h];
        } else if (r < C + 2 * nv) {
            beta[r - C - nv] = sigmoid(v);
        } else {
            z[r - C - 2 * nv] = v;
        }
    }
};

// Attention input projection rows: [0, 2qd) [q | gate] per head; [2qd,
// 2qd+kvd) k before its norm; [2qd+kvd, 2qd+2kvd) v, straight into the V
// cache row at the position in slots[1] (the cache append), or, with a
// quantized cache, into a scratch row that the attention kernel quantizes.
struct EpiAttnIn : EpiBase {
    float* qf;
    float* kraw;
    float* vcache;  // f32 cache: the V row goes straight to row pos
    float* vraw;    // quantized cache: the V row goes here, the attention kernel quantizes it
    const int* slots;
    int qd2, kvd;
    int pos;
    __device__ void start() { pos = __ldcg(slots + 1); }
    __device__ void apply(int r0, int r1, const float* ys, const float*, int tid) {
        for (int r = r0 + tid; r < r1; r += kConsumers) {
            const float v = ys[r - r0];
            if (r < qd2) qf[r] = v;
            else if (r < qd2 + kvd) kraw[r - qd2] = v;
            else if (vraw) vraw[r - qd2 - kvd] = v;
            else vcache[static_cast<size_t>(pos) * kvd + (r - qd2 - kvd)] = v;
        }
    }
};

// lm_head argmax of the whole-token step: publishes the token to slots[0]
// (the next step's embedding input) and slots[2] (the host readback, with
// bit 31 set when any kernel of the step set the device error word).  allow:
// the token mask (bit i & 31 of word i >> 5 set = token i allowed); a banned
// token's logit is replaced by -FLT_MAX before the first-index argmax, as
// the decode session's grammar mask does before its in-graph argmax.
struct EpiArgmaxStep : EpiBase {
    unsigned long long* ws;
    int* slots;
    uint32_t* hist;
    const unsigned* err;
    const uint32_t* allow;
    int advance;
    unsigned long long best;
    __device__ void start() { best = 0ull; }
    __device__ void apply(int r0, int r1, const float* ys, const float*, int tid) {
        for (int r = r0 + tid; r < r1; r += kConsumers) {
            const bool ok = (__ldcg(allow + (r >> 5)) >> (r & 31)) & 1u;
            const unsigned long long key = argmax_key(ok ? ys[r - r0] : -FLT_MAX, static_cast<unsigned>(r));
            best = key > best ? key : best;
        }
    }
    __device__ void finish(float* sm, int tid) {
        unsigned long long* red = reinterpret_cast<unsigned long long*>(sm);
        best = warp_max_u64(best);
        if ((tid & 31) == 0) red[tid >> 5] = best;
        bar_sync(1, kConsumers);
        if (tid == 0) {
            unsigned long long m = 0ull;
            for (int i = 0; i < kConsumerWarps; ++i) m = red[i] > m ? red[i] : m;
            atomicMax(ws, m);
            __threadfence();
            const unsigned prev = atomicAdd(reinterpret_cast<unsigned*>(ws + 1), 1u);
            if (prev == gridDim.x - 1) {
                __threadfence();
                const unsigned long long key = atomicExch(ws, 0ull);
                atomicExch(reinterpret_cast<unsigned*>(ws + 1), 0u);
                const unsigned tok = key ? argmax_key_index(key) : 0u;
                const unsigned e = __ldcg(err);
                slots[0] = static_cast<int>(tok);
                slots[2] = static_cast<int>(tok | (e ? 0x80000000u : 0u));
                if (advance) {
                    const int pos = __ldcg(slots + 1);
                    hist[pos] = tok;
                    slots[1] = pos + 1;
                }
            }
        }
    }
};

// ------------------------------------------------------------ prologues
// x = gated RMSNorm of the delta-rule output (gdn_gated_rmsnorm_into):
// u_i = (o_i * rn_h) * w_j * silu(z_i), i = h dv + j, with rn_h = 1 /
// sqrt(mean_j o^2 + eps).  dv divides 256, so a super-block holds whole heads:
// the warp that turns a super-block into digits loads its o and z itself and
// the dv/8 lanes of a head (8 values each) reduce the head's sum of squares
// with an xor tree.  Only the norm weights are staged (before the wait).
struct ProGatedNorm {
    const float* o;
    const float* z;
    const float* w;
    int nv, dv;
    float eps;
    struct Raw {
        float4 oa, ob, za, zb;
    };
    static constexpr int kBatch = 2;
    __host__ __device__ int floats(int) const { return 128 + 16; }  // w (dv <= 128); scratch
    __device__ void pre(float* sm, int, int tid) {  // the norm weights: before the dependency wait
        for (int i = tid; i < dv; i += kConsumers) sm[i] = __ldg(w + i);
    }
    __device__ void prepare(float*, int, int) {}
    __device__ void load8(int i0, Raw& r) const {
        r.oa = ldcg4(o + i0);
        r.ob = ldcg4(o + i0 + 4);
        r.za = ldcg4(z + i0);
        r.zb = ldcg4(z + i0 + 4);
    }
    __device__ void value8(const float* sm, int i0, const Raw& r, float* v) const {
        const float ov[8] = {r.oa.x, r.oa.y, r.oa.z, r.oa.w, r.ob.x, r.ob.y, r.ob.z, r.ob.w};
        const float zv[8] = {r.za.x, r.za.y, r.za.z, r.za.w, r.zb.x, r.zb.y, r.zb.z, r.zb.w};
        float ss = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) ss = fmaf(ov[j], ov[j], ss);
        const int lanes = dv >> 3;  // lanes per head
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            if (off < lanes) ss += __shfl_xor_sync(FULL, ss, off);
        const float rn = 1.0f / sqrtf(ss / static_cast<float>(dv) + eps);
        const int j0 = i0 & (dv - 1);
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = ((ov[j] * rn) * sm[j0 + j]) * silu(zv[j]);
    }
};

// ------------------------------------------------------------ delta rule
// gdn_delta_rule_into: per value head a [dv x 128] state, s[j*128 + i] ==
// S[i][j]; the key head of value head h is h % n_k_heads.
constexpr int kDk = 128;

// Rows t = 0..3 of one value head, one warp (lane owns k-dims 4*lane..+3):
// decay by g, read S_t . k, rank-1 update S_t += k * beta * (v_t - S_t . k),
// write the rows back to Sg, query o_t = (S_t . q) / sqrt(128).  st: the rows
// in shared memory (row t at st + 128 t); lane vb + t holds v_t.  o[] comes
// out the same in every lane.
__device__ __forceinline__ void delta_rows4(const float* st, float* Sg, float4 kk, float4 qq, float v_lane, int vb,
                                            float g, float be, int lane, float* o) {
    float4 rr[4];
    float dot[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const float4 sv = *reinterpret_cast<const float4*>(st + t * kDk + 4 * lane);
        rr[t] = make_float4(g * sv.x, g * sv.y, g * sv.z, g * sv.w);  // decay
        float d = rr[t].x * kk.x;
        d = fmaf(rr[t].y, kk.y, d);
        d = fmaf(rr[t].z, kk.z, d);
        dot[t] = fmaf(rr[t].w, kk.w, d);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int t = 0; t < 4; ++t) dot[t] += __shfl_xor_sync(FULL, dot[t], off);  // read
    float oq[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const float d = be * (__shfl_sync(FULL, v_lane, vb + t) - dot[t]);
        const float4 sn = make_float4(fmaf(kk.x, d, rr[t].x), fmaf(kk.y, d, rr[t].y), fmaf(kk.z, d, rr[t].z),
                                      fmaf(kk.w, d, rr[t].w));  // rank-1 update
        *reinterpret_cast<float4*>(Sg + t * kDk + 4 * lane) = sn;
        float q = sn.x * qq.x;
        q = fmaf(sn.y, qq.y, q);
        q = fmaf(sn.z, qq.z, q);
        oq[t] = fmaf(sn.w, qq.w, q);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int t = 0; t < 4; ++t) oq[t] += __shfl_xor_sync(FULL, oq[t], off);  // query
    const float scale = 1.0f / sqrtf(static_cast<float>(kDk));
#pragma unroll
    for (int t = 0; t < 4; ++t) o[t] = oq[t] * scale;
}

// ------------------------------------------------------ GQA decode attention
// Grid (max_splits, n_kv_heads), CW consumer warps + 1 producer warp.  CTA
// (s, g) covers cache rows [s*T, min((s+1)*T, pos+1)) for the GS query heads
// of kv group g (contiguous groups).  The producer streams the split's K and V
// rows of head g (1 KB each) into a shared-memory ring, CW keys per stage as
// one 2-D tensor copy of K rows and one of V rows (f32 cache), or one bulk
// copy of K records and one of V records (quantized cache); rows older than
// pos are fetched before the dependency wait, V[pos] (written by the previous
// kernel) after it, and K[pos] is computed here.  head_dim = 256: lane owns
// dims 4*lane..+3 and 128+4*lane..+3.
constexpr int kAttnStages = 4;

__device__ __forceinline__ void row8(const float* p, int lane, float* v) {
    const float4 a = *reinterpret_cast<const float4*>(p + 4 * lane);
    const float4 b = *reinterpret_cast<const float4*>(p + 128 + 4 * lane);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load_row8(const float* p, int lane, float* v) {
    const float4 a = __ldcg(reinterpret_cast<const float4*>(p + 4 * lane));
    const float4 b = __ldcg(reinterpret_cast<const float4*>(p + 128 + 4 * lane));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ int dim8(int lane, int j) { return j < 4 ? 4 * lane + j : 128 + 4 * lane + j - 4; }

// ------------------------------------------------- quantized KV cache records
// The decode session's quantized cache (forward_qwen35_cuda.rs, full
// attention layer): K as q8_0 blocks, V as q5_1 blocks of 32 values, the GGUF
// block contents (q8_0: f16 d, int8 q, x = d*q; q5_1: f16 d, f16 m, 5-bit q
// as a nibble plus one bit of qh, x = d*q + m), laid out per (kv head,
// position) record with the 8 blocks' scales first:
//   K record, 272 bytes: d[8] (f16) | q[256] (int8)
//   V record, 192 bytes: (d, m)[8] (f16 pairs) | qh[8] (u32) | qs[8][16]
//   (qs byte i of a block: q_i & 15 in the low nibble, q_{i+16} & 15 high)
// The cache of one layer is [n_kv_heads][max_seq][record], so the keys of one
// head are contiguous and a stage of them is one bulk copy.
// Quantizer: the block's f32 statistics give d (q8_0: max|x| / 127; q5_1:
// (max - min) / 31, m = min); each code is roundf(x * (1/d)) (q5_1:
// roundf((x - min) * (1/d))) with IEEE-rounded f32 operations, clamped to the
// code range; d below the smallest normal float gives zero codes; d and m are
// stored as f16 (round to nearest even), and every reader uses the stored
// values.
constexpr int kKRec = 272;
constexpr int kVRec = 192;

// One warp quantizes one 32-value q8_0 block of a K record: lane holds value
// `lane` of block b.  Returns the lane's dequantized value.
__device__ __forceinline__ float kvq_put_q8_0(float x, int lane, int b, uint8_t* rec) {
    const float amax = warp_max(fabsf(x));
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = d >= FLT_MIN ? __frcp_rn(d) : 0.0f;
    const float r = fminf(fmaxf(roundf(__fmul_rn(x, id)), -127.0f), 127.0f);
    const int q = static_cast<int>(r);
    const __half dh = __float2half_rn(d);
    rec[16 + 32 * b + lane] = static_cast<uint8_t>(static_cast<int8_t>(q));
    if (lane == 0) *reinterpret_cast<uint16_t*>(rec + 2 * b) = __half_as_ushort(dh);
    return __fmul_rn(__half2float(dh), static_cast<float>(q));
}

// One warp quantizes one 32-value q5_1 block of a V record (lane = value).
__device__ __forceinline__ float kvq_put_q5_1(float x, int lane, int b, uint8_t* rec) {
    const float lo = -warp_max(-x), hi = warp_max(x);
    const float d = __fdiv_rn(__fsub_rn(hi, lo), 31.0f);
    const float id = d >= FLT_MIN ? __frcp_rn(d) : 0.0f;
    const float r = fminf(fmaxf(roundf(__fmul_rn(__fsub_rn(x, lo), id)), 0.0f), 31.0f);
    const int q = static_cast<int>(r);
    const unsigned qh = __ballot_sync(0xffffffffu, (q >> 4) & 1);
    const int q_hi = __shfl_down_sync(0xffffffffu, q, 16);
    const __half dh = __float2half_rn(d), mh = __float2half_rn(lo);
    if (lane < 16) rec[64 + 16 * b + lane] = static_cast<uint8_t>((q & 15) | ((q_hi & 15) << 4));
    if (lane == 0) {
        *reinterpret_cast<uint32_t*>(rec + 4 * b) =
            static_cast<uint32_t>(__half_as_ushort(dh)) | (static_cast<uint32_t>(__half_as_ushort(mh)) << 16);
        *reinterpret_cast<uint32_t*>(rec + 32 + 4 * b) = qh;
    }
    return __fadd_rn(__fmul_rn(__half2float(dh), static_cast<float>(q)), __half2float(mh));
}

// The lane's 8 dims (dim8 order) of a K record, dequantized.
__device__ __forceinline__ void kvq_k8(const uint8_t* rec, int lane, float* v) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int b = 4 * h + (lane >> 3);
        const float d = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(rec + 2 * b)));
        const uint32_t c = *reinterpret_cast<const uint32_t*>(rec + 16 + 128 * h + 4 * lane);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            v[4 * h + j] = __fmul_rn(d, static_cast<float>(static_cast<int8_t>((c >> (8 * j)) & 0xffu)));
    }
}

// The lane's 8 dims (dim8 order) of a V record, dequantized.
__device__ __forceinline__ void kvq_v8(const uint8_t* rec, int lane, float* v) {
    const int j0 = 4 * (lane & 7);  // the lane's first value inside its blocks
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int b = 4 * h + (lane >> 3);
        const uint32_t dm = *reinterpret_cast<const uint32_t*>(rec + 4 * b);
        const float d = __half2float(__ushort_as_half(static_cast<uint16_t>(dm & 0xffffu)));
        const float m = __half2float(__ushort_as_half(static_cast<uint16_t>(dm >> 16)));
        const uint32_t qh = *reinterpret_cast<const uint32_t*>(rec + 32 + 4 * b);
        const uint32_t qs = *reinterpret_cast<const uint32_t*>(rec + 64 + 16 * b + (j0 & 15));
        const int sh = j0 < 16 ? 0 : 4;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int q = static_cast<int>((qs >> (8 * j + sh)) & 15u) | static_cast<int>(((qh >> (j0 + j)) & 1u) << 4);
            v[4 * h + j] = __fadd_rn(__fmul_rn(d, static_cast<float>(q)), m);
        }
    }
}

}  // namespace qg
