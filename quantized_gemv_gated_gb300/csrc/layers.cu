// The two layer kinds of the hybrid decode step and the token tail, as fused
// GB300 kernels, in the op order of forward_qwen35_cuda.rs.
//
// Gated DeltaNet layer (deltanet_layer_inner), five launches:
//   1. RMSNorm prologue + one GEMV over the fused [attn_qkv | ssm_alpha |
//      ssm_beta | attn_gate] rows; the epilogue of each row does its own
//      causal conv1d + SiLU + window roll (qkv rows), dt/beta gates
//      (alpha/beta rows) or stores z (gate rows).
//   2. delta rule: per-head L2 norm of q and k, decay, read, rank-1 update,
//      query; the state tile of a CTA is loaded before the dependency wait.
//   3. gated-RMSNorm prologue + ssm_out GEMV + residual epilogue.
//   4. RMSNorm prologue + ffn_gate/ffn_up dual GEMV + SwiGLU epilogue.
//   5. ffn_down (Q6_K) GEMV + residual epilogue.
// Full-attention layer (attention_layer_inner), five launches:
//   1. RMSNorm prologue + GEMV over the fused [attn_q | attn_k | attn_v]
//      rows; v rows land in the V cache row at `pos`.
//   2. split-K GQA decode attention over rows 0..pos: q/k per-head RMSNorm,
//      partial NEOX rope and the K-cache append happen in the prologue; the
//      last CTA of each kv group combines the splits and applies the sigmoid
//      output gate.
//   3. attn_output GEMV + residual, 4.-5. the FFN as above.
// Token tail (forward_single): output-RMSNorm prologue + lm_head GEMV with an
// argmax epilogue (first index on ties).
#include "qg_internal.cuh"

namespace qg {

// ------------------------------------------------------------ epilogues
// DeltaNet input projection rows: [0, C) qkv -> conv; [C, C+nv) alpha;
// [C+nv, C+2nv) beta; [C+2nv, C+2nv+v_dim) z.
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
    __device__ void apply(int r0, int r1, const float* ys, const float*, int tid) {
        for (int r = r0 + tid; r < r1; r += kConsumers) row_out(r, ys[r - r0]);
    }
    __device__ void row_out(int r, float v) {
        if (r < C) {
            // causal conv1d + SiLU, then roll the window (gdn_causal_conv1d_silu_into)
            const float* kw = wconv + static_cast<size_t>(r) * K;
            float* wc = win + static_cast<size_t>(r) * (K - 1);
            float acc = 0.0f;
            for (int t = 0; t < K - 1; ++t) {
                const float wt = __ldcg(wc + t);
                acc += kw[t] * wt;
                if (t > 0) wc[t - 1] = wt;  // roll: shift left, append the new input
            }
            acc += kw[K - 1] * v;
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
// cache row at the position in slots[1] (the cache append).
struct EpiAttnIn : EpiBase {
    float* qf;
    float* kraw;
    float* vcache;
    const int* slots;
    int qd2, kvd;
    int pos;
    __device__ void start() { pos = __ldcg(slots + 1); }
    __device__ void apply(int r0, int r1, const float* ys, const float*, int tid) {
        for (int r = r0 + tid; r < r1; r += kConsumers) {
            const float v = ys[r - r0];
            if (r < qd2) qf[r] = v;
            else if (r < qd2 + kvd) kraw[r - qd2] = v;
            else vcache[static_cast<size_t>(pos) * kvd + (r - qd2 - kvd)] = v;
        }
    }
};

// lm_head argmax of the whole-token step: publishes the token to slots[0]
// (the next step's embedding input) and slots[2] (the host readback, with
// bit 31 set when any kernel of the step set the device error word).
struct EpiArgmaxStep : EpiBase {
    static constexpr bool kDeferred = false;
    unsigned long long* ws;
    int* slots;
    uint32_t* hist;
    const unsigned* err;
    int advance;
    unsigned long long best;
    __device__ void start() { best = 0ull; }
    __device__ void row(int r, float v) {
        const unsigned long long key = argmax_key(v, static_cast<unsigned>(r));
        best = key > best ? key : best;
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

// ------------------------------------------------------------ delta rule
// One CTA: 16 rows j of value head h (8 warps x 2 rows), head_k_dim = 128
// (4 per lane).  State row j of head h: s[(h*dv + j)*128 + i] == S[i][j].
constexpr int kDk = 128;

__global__ void __launch_bounds__(256) delta_kernel(const float* __restrict__ conv_out, const float* __restrict__ dt,
                                                    const float* __restrict__ beta, float* __restrict__ S,
                                                    float* __restrict__ o, int nk, int dv, int kdim, float eps) {
    __shared__ __align__(16) float qs[kDk];
    __shared__ __align__(16) float ks[kDk];
    const int h = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kh = h % nk;  // value head h reads key head h % nk (check_head_grouping)
    pdl_launch_dependents();
    // the state tile does not depend on the previous kernel: fetch it first
    float4 s[2];
    int js[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        js[r] = blockIdx.x * 16 + warp * 2 + r;
        s[r] = __ldcg(reinterpret_cast<const float4*>(S + (static_cast<size_t>(h) * dv + js[r]) * kDk + 4 * lane));
    }
    pdl_wait();
    if (warp < 2) {  // per-head L2 norm of q (warp 0) and k (warp 1) (gdn_per_head_l2_norm_into)
        const float4 v = ldcg4(conv_out + (warp ? kdim : 0) + kh * kDk + 4 * lane);
        float ss = v.x * v.x;
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
        ss = warp_sum(ss);
        const float r = 1.0f / sqrtf(ss + eps);
        float* dst = warp ? ks : qs;
        *reinterpret_cast<float4*>(dst + 4 * lane) = make_float4(v.x * r, v.y * r, v.z * r, v.w * r);
    }
    __syncthreads();
    const float g = expf(__ldcg(dt + h)), be = __ldcg(beta + h);
    const float scale = 1.0f / sqrtf(static_cast<float>(kDk));
    const float4 kk = *reinterpret_cast<const float4*>(ks + 4 * lane);
    const float4 qq = *reinterpret_cast<const float4*>(qs + 4 * lane);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const float4 rr = make_float4(g * s[r].x, g * s[r].y, g * s[r].z, g * s[r].w);  // decay
        float dot = rr.x * kk.x;
        dot = fmaf(rr.y, kk.y, dot);
        dot = fmaf(rr.z, kk.z, dot);
        dot = fmaf(rr.w, kk.w, dot);
        dot = warp_sum(dot);                                                     // read
        const float vj = __ldcg(conv_out + 2 * kdim + h * dv + js[r]);
        const float d = be * (vj - dot);
        const float4 sn = make_float4(fmaf(kk.x, d, rr.x), fmaf(kk.y, d, rr.y), fmaf(kk.z, d, rr.z),
                                      fmaf(kk.w, d, rr.w));  // rank-1 update
        *reinterpret_cast<float4*>(S + (static_cast<size_t>(h) * dv + js[r]) * kDk + 4 * lane) = sn;
        float oq = sn.x * qq.x;
        oq = fmaf(sn.y, qq.y, oq);
        oq = fmaf(sn.z, qq.z, oq);
        oq = fmaf(sn.w, qq.w, oq);
        oq = warp_sum(oq);  // query
        if (lane == 0) o[h * dv + js[r]] = oq * scale;
    }
}

// ------------------------------------------------------ GQA decode attention
// Grid (max_splits, n_kv_heads), 8 consumer warps + 1 producer warp.  CTA
// (s, g) covers cache rows [s*T, min((s+1)*T, pos+1)) for the GS query heads
// of kv group g (contiguous groups).  The producer streams the split's K and V
// rows of group g (1 KB each) into a shared-memory ring with bulk copies,
// 8 keys per stage; rows older than pos are fetched before the dependency
// wait, V[pos] (written by the previous kernel) after it, and K[pos] is
// computed here.  head_dim = 256: lane owns dims 4*lane..+3 and 128+4*lane..+3.
constexpr int kHd = 256;
constexpr int kAttnStages = 4;
constexpr int kKeysPerStage = 8;

struct AttnArgs {
    const float* qf;     // [nh][2*hd]: q then gate per head
    const float* kraw;   // [nkv*hd]
    float* kc;           // K cache [max_seq][kvd]
    const float* vc;     // V cache
    const float* q_norm;
    const float* k_norm;
    const int* slots;
    float* part_acc;     // [nkv][max_splits][GS][hd]
    float* part_ml;      // [nkv][max_splits][GS][2]
    unsigned* count;     // [nkv]
    float* out;          // [nh*hd], gated
    unsigned* err;
    int kvd, T, max_splits, n_rot;
    float theta_scale, eps;
};

template <int GS>
__host__ __device__ inline int attn_smem_floats() {
    return GS * kHd + kHd + kHd + 8 * GS * 2 + 8 * GS * kHd + 64 * GS * 2 + kAttnStages * kKeysPerStage * 2 * kHd;
}

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

template <int GS>
__global__ void __launch_bounds__(288) attn_kernel(const AttnArgs a) {
    extern __shared__ __align__(128) float sm[];
    __shared__ uint64_t full[kAttnStages], empty[kAttnStages];
    __shared__ int last_flag;
    float* ring = sm;                                        // [stages][8 keys][K row | V row]
    float* q_s = ring + kAttnStages * kKeysPerStage * 2 * kHd;  // [GS][hd]
    float* k_s = q_s + GS * kHd;                             // [hd]
    float* cs = k_s + kHd;                                   // [hd/2]
    float* sn = cs + kHd / 2;                                // [hd/2]
    float* wml = sn + kHd / 2;                               // [8][GS][2]
    float* wacc = wml + 8 * GS * 2;                          // [8][GS][hd]
    float* cml = wacc + 8 * GS * kHd;                        // [64][GS][2] split (m, l) of the combine

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s = blockIdx.x, g = blockIdx.y;
    pdl_launch_dependents();
    // the position is written before the first kernel of the step: safe to read now
    const int pos = __ldcg(a.slots + 1);
    const int t_len = pos + 1;
    const int n_act = (t_len + a.T - 1) / a.T;
    if (s >= n_act) return;
    const bool has_new = (s == n_act - 1);  // the split holding row pos
    const int t0 = s * a.T, t1 = min(t0 + a.T, t_len);
    const int nst = (t1 - t0 + kKeysPerStage - 1) / kKeysPerStage;
    const int half = a.n_rot / 2;

    if (tid == 0) {
        for (int i = 0; i < kAttnStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 8);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == 8) {
        // ----------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            bool waited = false, ok = true;
            int issued = 0;
            for (int st = 0; st < nst; ++st) {
                const int slot = st % kAttnStages;
                if (st >= kAttnStages && !mbar_wait(&empty[slot], ((st / kAttnStages) - 1) & 1)) {
                    atomicOr(a.err, DEVERR_EMPTY_WAIT);
                    ok = false;
                    break;
                }
                const int k0 = t0 + st * kKeysPerStage, k1 = min(k0 + kKeysPerStage, t1);
                if (!waited && k1 > pos) {
                    pdl_wait();  // V[pos] is written by the previous kernel
                    waited = true;
                }
                unsigned bytes = 0;
                for (int t = k0; t < k1; ++t) bytes += (t == pos ? 1u : 2u) * kHd * 4u;
                mbar_arrive_expect_tx(&full[slot], bytes);
                float* st_base = ring + static_cast<size_t>(slot) * kKeysPerStage * 2 * kHd;
                for (int t = k0; t < k1; ++t) {
                    float* dst = st_base + (t - k0) * 2 * kHd;
                    const size_t off = static_cast<size_t>(t) * a.kvd + g * kHd;
                    if (t != pos) bulk_g2s(dst, a.kc + off, kHd * 4, &full[slot], pol);
                    bulk_g2s(dst + kHd, a.vc + off, kHd * 4, &full[slot], pol);
                }
                issued = st + 1;
            }
            if (!ok)
                for (int st = max(0, issued - kAttnStages); st < issued; ++st)
                    if (!mbar_wait(&full[st % kAttnStages], (st / kAttnStages) & 1)) atomicOr(a.err, DEVERR_DRAIN_WAIT);
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    pdl_wait();
    // rope angles: theta_0 = pos, theta_{i+1} = theta_i * theta_scale (f32 running product)
    if (tid < half) {
        float th = static_cast<float>(pos);
        for (int i = 0; i < tid; ++i) th = th * a.theta_scale;
        float sv, cv;
        sincosf(th, &sv, &cv);
        cs[tid] = cv;
        sn[tid] = sv;
    }
    // per-head RMSNorm of q (and of this token's k) (per_head_rmsnorm_into)
    for (int job = warp; job < GS + (has_new ? 1 : 0); job += 8) {
        const float* src = job < GS ? a.qf + static_cast<size_t>(g * GS + job) * 2 * kHd : a.kraw + g * kHd;
        const float* w = job < GS ? a.q_norm : a.k_norm;
        float* dst = job < GS ? q_s + job * kHd : k_s;
        float v[8];
        load_row8(src, lane, v);
        float ss = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(v[i], v[i], ss);
        ss = warp_sum(ss);
        const float r = 1.0f / sqrtf(ss / static_cast<float>(kHd) + a.eps);
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[dim8(lane, i)] = (v[i] * r) * __ldg(w + dim8(lane, i));
    }
    bar_sync(1, 256);
    // partial NEOX rope on pairs (i, i + n_rot/2), i < n_rot/2 (gdn_partial_neox_rope_into)
    const int jobs = GS + (has_new ? 1 : 0);
    for (int p = tid; p < jobs * half; p += 256) {
        const int job = p / half, i = p - job * half;
        float* vec = job < GS ? q_s + job * kHd : k_s;
        const float x0 = vec[i], x1 = vec[i + half];
        vec[i] = x0 * cs[i] - x1 * sn[i];
        vec[i + half] = x0 * sn[i] + x1 * cs[i];
    }
    bar_sync(1, 256);
    if (has_new) a.kc[static_cast<size_t>(pos) * a.kvd + g * kHd + tid] = k_s[tid];  // K append at pos

    float q[GS][8];
#pragma unroll
    for (int i = 0; i < GS; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) q[i][j] = q_s[i * kHd + dim8(lane, j)];
    float m[GS], l[GS], acc[GS][8];
#pragma unroll
    for (int i = 0; i < GS; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
    }
    const float scale = 1.0f / sqrtf(static_cast<float>(kHd));
    for (int st = 0; st < nst; ++st) {
        const int slot = st % kAttnStages;
        if (!mbar_wait(&full[slot], (st / kAttnStages) & 1)) {
            atomicOr(a.err, DEVERR_FULL_WAIT);
            break;
        }
        const int t = t0 + st * kKeysPerStage + warp;
        if (t < t1) {
            const float* kv_row = ring + (static_cast<size_t>(slot) * kKeysPerStage + warp) * 2 * kHd;
            float kv[8], vv[8];
            row8(t == pos ? k_s : kv_row, lane, kv);
            row8(kv_row + kHd, lane, vv);
#pragma unroll
            for (int i = 0; i < GS; ++i) {
                float dot = 0.0f;
#pragma unroll
                for (int j = 0; j < 8; ++j) dot = fmaf(q[i][j], kv[j], dot);
                const float sc = warp_sum(dot) * scale;
                const float mn = fmaxf(m[i], sc);
                const float c = expf(m[i] - mn), p = expf(sc - mn);
                l[i] = fmaf(l[i], c, p);
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(acc[i][j], c, p * vv[j]);
                m[i] = mn;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }
#pragma unroll
    for (int i = 0; i < GS; ++i) {
        if (lane == 0) {
            wml[(warp * GS + i) * 2 + 0] = m[i];
            wml[(warp * GS + i) * 2 + 1] = l[i];
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) wacc[(warp * GS + i) * kHd + dim8(lane, j)] = acc[i][j];
    }
    bar_sync(1, 256);
    // combine the 8 warps: thread tid owns dim tid of every head
    const size_t pbase = (static_cast<size_t>(g) * a.max_splits + s) * GS;
    for (int i = 0; i < GS; ++i) {
        float M = -INFINITY;
        for (int w = 0; w < 8; ++w) M = fmaxf(M, wml[(w * GS + i) * 2]);
        float L = 0.0f, A = 0.0f;
        for (int w = 0; w < 8; ++w) {
            const float mw = wml[(w * GS + i) * 2];
            const float f = mw == -INFINITY ? 0.0f : expf(mw - M);
            L = fmaf(wml[(w * GS + i) * 2 + 1], f, L);
            A = fmaf(wacc[(w * GS + i) * kHd + tid], f, A);
        }
        a.part_acc[(pbase + i) * kHd + tid] = A;
        if (tid == 0) {
            a.part_ml[(pbase + i) * 2 + 0] = M;
            a.part_ml[(pbase + i) * 2 + 1] = L;
        }
    }
    __threadfence();
    bar_sync(1, 256);
    if (tid == 0) last_flag = (atomicAdd(a.count + g, 1u) == static_cast<unsigned>(n_act - 1));
    bar_sync(1, 256);
    if (!last_flag) return;
    __threadfence();
    // last CTA of group g: combine the splits in order, then the sigmoid gate
    const size_t hb = static_cast<size_t>(g) * a.max_splits * GS;
    for (int e = tid; e < n_act * GS * 2; e += 256) cml[e] = __ldcg(a.part_ml + hb * 2 + e);
    bar_sync(1, 256);
    for (int job = tid; job < GS * (kHd / 4); job += 256) {
        const int i = job / (kHd / 4), d4 = 4 * (job - i * (kHd / 4));
        float M = -INFINITY;
        for (int sp = 0; sp < n_act; ++sp) M = fmaxf(M, cml[(sp * GS + i) * 2]);
        float L = 0.0f;
        float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int sp0 = 0; sp0 < n_act; sp0 += 8) {
            float4 v[8];
            float f[8], lw[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const bool in = sp0 + u < n_act;
                const int sp = in ? sp0 + u : sp0;
                v[u] = __ldcg(reinterpret_cast<const float4*>(a.part_acc + (hb + sp * GS + i) * kHd + d4));
                f[u] = in ? expf(cml[(sp * GS + i) * 2] - M) : 0.0f;
                lw[u] = cml[(sp * GS + i) * 2 + 1];
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                L = fmaf(lw[u], f[u], L);
                A.x = fmaf(v[u].x, f[u], A.x);
                A.y = fmaf(v[u].y, f[u], A.y);
                A.z = fmaf(v[u].z, f[u], A.z);
                A.w = fmaf(v[u].w, f[u], A.w);
            }
        }
        const int h = g * GS + i;
        const float4 gt = __ldcg(reinterpret_cast<const float4*>(a.qf + static_cast<size_t>(h) * 2 * kHd + kHd + d4));
        float4 o;  // (A / L) * sigmoid(gate)  (gdn_sigmoid_gate_into)
        o.x = (A.x / L) * sigmoid(gt.x);
        o.y = (A.y / L) * sigmoid(gt.y);
        o.z = (A.z / L) * sigmoid(gt.z);
        o.w = (A.w / L) * sigmoid(gt.w);
        *reinterpret_cast<float4*>(a.out + h * kHd + d4) = o;
    }
    if (tid == 0) a.count[g] = 0u;
}

__global__ void neg_exp_kernel(const float* __restrict__ src, float* __restrict__ dst, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) dst[i] = -expf(src[i]);
}

int run_neg_exp(const float* src, float* dst, int n, cudaStream_t st) {
    neg_exp_kernel<<<(n + 255) / 256, 256, 0, st>>>(src, dst, n);
    QG_CUDA(cudaGetLastError());
    return QG_OK;
}

// --------------------------------------------------------------- launchers
static int ffn(const qg_model* m, qg_state* s, const qg_layer_dev& L, float* h, cudaStream_t st) {
    const qg_config& c = m->cfg;
    ProRmsNorm pn{};
    pn.h = h;
    pn.w = L.post_norm;
    pn.tok = nullptr;
    pn.h_out = nullptr;
    pn.eps = c.eps;
    pn.kdim = c.hidden;
    EpiSwiGlu sw{};
    sw.act = s->act;
    int rc = launch_gemv<QT_Q4K, true>(L.w_gate, L.w_up, c.ffn, c.hidden, pn, sw, st, true, s->err);
    if (rc) return rc;
    EpiResidual er{};
    er.h = h;
    return launch_gemv<QT_Q6K, false>(L.w_down, nullptr, c.hidden, c.ffn, ProPlain{s->act}, er, st, true, s->err);
}

static ProRmsNorm input_norm(const qg_model* m, qg_state* s, const qg_layer_dev& L, float* h, bool embed) {
    ProRmsNorm pn{};
    pn.h = embed ? m->embd : h;
    pn.w = L.attn_norm;
    pn.tok = embed ? s->slots : nullptr;
    pn.h_out = h;
    pn.eps = m->cfg.eps;
    pn.kdim = m->cfg.hidden;
    return pn;
}

int run_deltanet_layer(const qg_model* m, qg_state* s, int il, float* h, cudaStream_t st, bool embed,
                       bool pdl_first) {
    const qg_config& c = m->cfg;
    const qg_layer_dev& L = m->layers[il];
    EpiDnIn ei{};
    ei.C = m->conv_dim;
    ei.nv = c.n_v_heads;
    ei.K = c.conv_kernel;
    ei.win = s->conv[il];
    ei.wconv = L.conv_w;
    ei.conv_out = s->conv_out;
    ei.dt_bias = L.dt_bias;
    ei.a = L.a;
    ei.dt = s->dt;
    ei.beta = s->beta;
    ei.z = s->z;
    int rc = launch_gemv<QT_Q4K, false>(L.w_in, nullptr, L.n_in, c.hidden, input_norm(m, s, L, h, embed), ei, st,
                                        pdl_first, s->err);
    if (rc) return rc;
    rc = launch_pdl(delta_kernel, dim3(c.head_v_dim / 16, c.n_v_heads), dim3(256), 0, st, true, s->conv_out, s->dt,
                    s->beta, s->ssm[il], s->o, c.n_k_heads, c.head_v_dim, m->k_dim, c.eps);
    if (rc) return rc;
    ProGatedNorm pg{};
    pg.o = s->o;
    pg.z = s->z;
    pg.w = L.ssm_norm;
    pg.dv = c.head_v_dim;
    pg.eps = c.eps;
    pg.kdim = m->v_dim;
    EpiResidual er{};
    er.h = h;
    rc = launch_gemv<QT_Q4K, false>(L.w_out, nullptr, c.hidden, m->v_dim, pg, er, st, true, s->err);
    if (rc) return rc;
    return ffn(m, s, L, h, st);
}

template <int GS>
static int launch_attn(const qg_model* m, qg_state* s, const AttnArgs& a, cudaStream_t st) {
    const int smem = attn_smem_floats<GS>() * 4;
    static int configured = 0;
    if (smem > configured) {
        QG_CUDA(cudaFuncSetAttribute(attn_kernel<GS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
        configured = smem;
    }
    return launch_pdl(attn_kernel<GS>, dim3(s->max_splits, m->cfg.n_kv_heads), dim3(288), smem, st, true, a);
}

int run_attention_layer(const qg_model* m, qg_state* s, int il, float* h, cudaStream_t st, bool embed,
                        bool pdl_first) {
    const qg_config& c = m->cfg;
    const qg_layer_dev& L = m->layers[il];
    EpiAttnIn ea{};
    ea.qf = s->qf;
    ea.kraw = s->kraw;
    ea.vcache = s->vc[il];
    ea.slots = s->slots;
    ea.qd2 = 2 * m->q_dim;
    ea.kvd = m->kv_dim;
    int rc = launch_gemv<QT_Q4K, false>(L.w_in, nullptr, L.n_in, c.hidden, input_norm(m, s, L, h, embed), ea, st,
                                        pdl_first, s->err);
    if (rc) return rc;
    AttnArgs a{};
    a.qf = s->qf;
    a.kraw = s->kraw;
    a.kc = s->kc[il];
    a.vc = s->vc[il];
    a.q_norm = L.q_norm;
    a.k_norm = L.k_norm;
    a.slots = s->slots;
    a.part_acc = s->part_acc;
    a.part_ml = s->part_ml;
    a.count = s->attn_count;
    a.out = s->attn;
    a.err = s->err;
    a.kvd = m->kv_dim;
    a.T = s->keys_per_split;
    a.max_splits = s->max_splits;
    a.n_rot = c.n_rot;
    a.theta_scale = m->theta_scale;
    a.eps = c.eps;
    switch (c.n_heads / c.n_kv_heads) {
        case 1: rc = launch_attn<1>(m, s, a, st); break;
        case 2: rc = launch_attn<2>(m, s, a, st); break;
        case 4: rc = launch_attn<4>(m, s, a, st); break;
        case 8: rc = launch_attn<8>(m, s, a, st); break;
        default: return set_err(QG_ERR_SHAPE, "attention: %d query heads per kv head", c.n_heads / c.n_kv_heads);
    }
    if (rc) return rc;
    EpiResidual er{};
    er.h = h;
    rc = launch_gemv<QT_Q4K, false>(L.w_out, nullptr, c.hidden, m->q_dim, ProPlain{s->attn}, er, st, true, s->err);
    if (rc) return rc;
    return ffn(m, s, L, h, st);
}

int run_lmhead(const qg_model* m, qg_state* s, const float* h, cudaStream_t st, bool advance) {
    const qg_config& c = m->cfg;
    ProRmsNorm pn{};
    pn.h = h;
    pn.w = m->out_norm;
    pn.tok = nullptr;
    pn.h_out = nullptr;
    pn.eps = c.eps;
    pn.kdim = c.hidden;
    EpiArgmaxStep ea{};
    ea.ws = s->am_ws;
    ea.slots = s->slots;
    ea.hist = s->hist;
    ea.err = s->err;
    ea.advance = advance ? 1 : 0;
    return launch_gemv<QT_Q6K, false>(m->lm_head, nullptr, c.vocab, c.hidden, pn, ea, st, true, s->err);
}

}  // namespace qg
