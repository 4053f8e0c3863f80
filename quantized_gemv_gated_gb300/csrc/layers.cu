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
#include <algorithm>

#include "qg_layers.cuh"

namespace qg {

// ------------------------------------------------------------ delta rule
// gdn_delta_rule_into over items of 32 state rows of one value head (four
// rows per warp, head_k_dim = 128: 4 per lane): the item's 16 KB of state
// arrives in shared memory with one bulk copy issued before the dependency
// wait; each warp runs decay, read, rank-1 update and query on its rows
// (delta_rows4), writes them back and stores the rows' o (before the gated
// RMSNorm, which needs the whole head and is applied by the ssm_out GEMV's
// prologue, ProGatedNorm).
struct DeltaArgs {
    const float* conv_out;  // [q | k | v] after conv + SiLU
    const float* dt;        // log-decay per value head
    const float* beta;
    float* S;               // [nv][dv][128]
    float* o;               // [v_dim]
    unsigned* err;
    L2Prefetch next;
    int nk, dv, kdim;
    float eps;
};

constexpr int kDeltaRows = 32;  // state rows per CTA (one item)

__global__ void __launch_bounds__(256) delta_kernel(const DeltaArgs a) {
    __shared__ __align__(128) float st[kDeltaRows * kDk];
    __shared__ __align__(16) float qs[kDk];
    __shared__ __align__(16) float ks[kDk];
    __shared__ __align__(8) uint64_t bar;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int per_head = a.dv / kDeltaRows;
    const int h = blockIdx.x / per_head, jb = (blockIdx.x - h * per_head) * kDeltaRows;
    const int kh = h % a.nk;  // value head h reads key head h % nk (check_head_grouping)
    const int j = jb + 4 * warp;  // this warp's first row
    pdl_launch_dependents();
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {  // the state does not depend on the previous kernel
        const unsigned bytes = kDeltaRows * kDk * 4u;
        mbar_arrive_expect_tx(&bar, bytes);
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(st)),
            "l"(a.S + (static_cast<size_t>(h) * a.dv + jb) * kDk), "r"(bytes), "r"(smem_u32(&bar))
            : "memory");
        a.next.issue();
    }
    pdl_wait();
    if (warp < 2) {  // per-head L2 norm of q (warp 0) and k (warp 1) (gdn_per_head_l2_norm_into)
        const float4 v = ldcg4(a.conv_out + (warp ? a.kdim : 0) + kh * kDk + 4 * lane);
        float ss = v.x * v.x;
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
        ss = warp_sum(ss);
        const float r = 1.0f / sqrtf(ss + a.eps);
        float* dst = warp ? ks : qs;
        *reinterpret_cast<float4*>(dst + 4 * lane) = make_float4(v.x * r, v.y * r, v.z * r, v.w * r);
    }
    const float vl = lane < 4 ? __ldcg(a.conv_out + 2 * a.kdim + h * a.dv + j + lane) : 0.0f;
    const float g = expf(__ldcg(a.dt + h)), be = __ldcg(a.beta + h);
    __syncthreads();
    if (!mbar_wait(&bar, 0)) {
        atomicOr(a.err, DEVERR_FULL_WAIT);
        if (!mbar_wait(&bar, 0)) atomicOr(a.err, DEVERR_DRAIN_WAIT);
        return;
    }
    const float4 kk = *reinterpret_cast<const float4*>(ks + 4 * lane);
    const float4 qq = *reinterpret_cast<const float4*>(qs + 4 * lane);
    float o[4];
    delta_rows4(st + 4 * warp * kDk, a.S + (static_cast<size_t>(h) * a.dv + j) * kDk, kk, qq, vl, 0, g, be, lane, o);
    float mine = 0.0f;
#pragma unroll
    for (int t = 0; t < 4; ++t)
        if (lane == t) mine = o[t];
    if (lane < 4) a.o[h * a.dv + j + lane] = mine;
}

// h += y, y given as `parts` vectors `stride` floats apart added in order.
__global__ void residual_add_kernel(float* h, const float* y, int parts, int stride, int n) {
    pdl_launch_dependents();
    pdl_wait();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float v = __ldcg(y + i);
    for (int p = 1; p < parts; ++p) v += __ldcg(y + static_cast<size_t>(p) * stride + i);
    h[i] = __ldcg(h + i) + v;
}

struct AttnArgs {
    // f32 cache: 2-D tensor maps of the layer's K and V caches ([max_seq] rows
    // of kvd floats; box: 256 floats x the keys of a stage), so a stage of one
    // kv head's keys is one tensor copy for K and one for V
    CUtensorMap kmap, vmap;
    const float* qf;     // [nh][2*hd]: q then gate per head
    const float* kraw;   // [nkv*hd]
    float* kc;           // K cache: f32 [max_seq][kvd], or q8_0 records [nkv][max_seq][kKRec bytes]
    float* vc;           // V cache: f32 [max_seq][kvd], or q5_1 records [nkv][max_seq][kVRec bytes]
    const float* vraw;   // quantized cache: this token's V row [nkv*hd] (the input GEMV's output)
    const float* q_norm;
    const float* k_norm;
    const int* slots;
    float* part_acc;     // [nkv][max_splits][GS][hd]
    float* part_ml;      // [nkv][max_splits][GS][2]
    unsigned* count;     // [nkv]
    float* out;          // [nh*hd], gated
    unsigned* err;
    L2Prefetch next;
    int kvd, T, max_splits, n_rot, max_seq;
    float theta_scale, eps;
};

// Consumer warps CW of the attention kernel, which is also its keys per ring
// stage (one key per consumer warp per stage): 16 for up to 4 query heads per
// kv head, twice the keys in flight per SM of 8 warps (measured on the 4B
// step: 26 instead of ~35 us per launch at t ~ 8000, and no slower at t ~
// 900); 8 above that, where the per-warp accumulators of 8 heads need the
// registers.
inline int attn_warps(int gs) { return gs <= 4 ? 16 : 8; }

// Bytes of one ring stage: its keys' K rows then V rows (f32), or their K
// records then their V records (quantized cache).
template <bool KVQ, int CW>
__host__ __device__ constexpr int attn_stage_bytes() {
    return KVQ ? CW * (kKRec + kVRec) : CW * 2 * kHd * 4;
}

template <int GS, bool KVQ, int CW>
__host__ __device__ inline int attn_smem_floats() {
    return GS * kHd + kHd + kHd + kHd + CW * GS * 2 + CW * GS * kHd + 64 * GS * 2 +
           kAttnStages * attn_stage_bytes<KVQ, CW>() / 4;
}


// KVQ: the cache holds q8_0 K / q5_1 V records (the layout above kvq_put_q8_0):
// the split holding row pos quantizes this token's K (after its norm and
// rope) and V rows into the cache, and every key, this one included, is read
// back dequantized.
template <int GS, bool KVQ, int CW>
__global__ void __launch_bounds__(32 * (CW + 1)) attn_kernel(const __grid_constant__ AttnArgs a) {
    constexpr int KS = CW, NC = 32 * CW;  // keys per stage, consumer threads
    extern __shared__ __align__(128) float sm[];
    __shared__ uint64_t full[kAttnStages], empty[kAttnStages];
    __shared__ int last_flag;
    float* ring = sm;                                        // [stages][KS K rows | KS V rows] (f32), or
                                                             // [stages][KS K records | KS V records]
    float* q_s = ring + kAttnStages * attn_stage_bytes<KVQ, CW>() / 4;  // [GS][hd]
    float* k_s = q_s + GS * kHd;                             // [hd]
    float* v_s = k_s + kHd;                                  // [hd] this token's V, dequantized (KVQ)
    float* cs = v_s + kHd;                                   // [hd/2]
    float* sn = cs + kHd / 2;                                // [hd/2]
    float* wml = sn + kHd / 2;                               // [CW][GS][2]
    float* wacc = wml + CW * GS * 2;                         // [CW][GS][hd]
    float* cml = wacc + CW * GS * kHd;                       // [64][GS][2] split (m, l) of the combine

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
    const int nst = (t1 - t0 + KS - 1) / KS;
    const int half = a.n_rot / 2;

    if (tid == 0) {
        for (int i = 0; i < kAttnStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], CW);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == CW) {
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
                const int k0 = t0 + st * KS, k1 = min(k0 + KS, t1);
                if constexpr (KVQ) {
                    // rows before pos were written by earlier steps; row pos is made here
                    const int n_old = min(k1, pos) - k0;
                    const unsigned kb = static_cast<unsigned>(n_old > 0 ? n_old : 0) * kKRec;
                    const unsigned vb = static_cast<unsigned>(n_old > 0 ? n_old : 0) * kVRec;
                    mbar_arrive_expect_tx(&full[slot], kb + vb);
                    uint8_t* st_base = reinterpret_cast<uint8_t*>(ring) + static_cast<size_t>(slot) * attn_stage_bytes<true, CW>();
                    const size_t rec0 = static_cast<size_t>(g) * a.max_seq + k0;
                    if (kb) {
                        bulk_g2s(st_base, reinterpret_cast<const uint8_t*>(a.kc) + rec0 * kKRec, kb, &full[slot], pol);
                        bulk_g2s(st_base + KS * kKRec, reinterpret_cast<const uint8_t*>(a.vc) + rec0 * kVRec,
                                 vb, &full[slot], pol);
                    }
                } else {
                    if (!waited && k1 > pos) {
                        pdl_wait();  // V[pos] is written by the previous kernel
                        waited = true;
                    }
                    // one tensor copy of kv head g's K rows k0..k0+KS-1 and one of its V
                    // rows (K[pos] is replaced by this kernel's own row; rows past the
                    // split are read and not used, rows past the cache read as zeros)
                    constexpr unsigned box = KS * kHd * 4u;
                    mbar_arrive_expect_tx(&full[slot], 2u * box);
                    float* st_base = ring + static_cast<size_t>(slot) * KS * 2 * kHd;
                    tma_load_2d(st_base, &a.kmap, g * kHd, k0, &full[slot], pol);
                    tma_load_2d(st_base + KS * kHd, &a.vmap, g * kHd, k0, &full[slot], pol);
                }
                issued = st + 1;
                if (st == 0) a.next.issue();
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
    for (int job = warp; job < GS + (has_new ? 1 : 0); job += CW) {
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
    bar_sync(1, NC);
    // partial NEOX rope on pairs (i, i + n_rot/2), i < n_rot/2 (gdn_partial_neox_rope_into)
    const int jobs = GS + (has_new ? 1 : 0);
    for (int p = tid; p < jobs * half; p += NC) {
        const int job = p / half, i = p - job * half;
        float* vec = job < GS ? q_s + job * kHd : k_s;
        const float x0 = vec[i], x1 = vec[i + half];
        vec[i] = x0 * cs[i] - x1 * sn[i];
        vec[i + half] = x0 * sn[i] + x1 * cs[i];
    }
    bar_sync(1, NC);
    if constexpr (KVQ) {
        if (has_new) {  // quantize-on-append: warp w < 8 makes block w of the K and the V record at pos
            const size_t rec = static_cast<size_t>(g) * a.max_seq + pos;
            const int e = 32 * warp + lane;
            if (warp < 8) {
                k_s[e] = kvq_put_q8_0(k_s[e], lane, warp, reinterpret_cast<uint8_t*>(a.kc) + rec * kKRec);
                v_s[e] = kvq_put_q5_1(__ldcg(a.vraw + g * kHd + e), lane, warp,
                                      reinterpret_cast<uint8_t*>(a.vc) + rec * kVRec);
            }
            bar_sync(1, NC);
        }
    } else {
        if (has_new && tid < kHd) a.kc[static_cast<size_t>(pos) * a.kvd + g * kHd + tid] = k_s[tid];  // K append at pos
    }

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
        const int t = t0 + st * KS + warp;
        if (t < t1) {
            float kv[8], vv[8];
            if constexpr (KVQ) {
                const uint8_t* sb = reinterpret_cast<const uint8_t*>(ring) + static_cast<size_t>(slot) * attn_stage_bytes<true, CW>();
                if (t == pos) {
                    row8(k_s, lane, kv);
                    row8(v_s, lane, vv);
                } else {
                    kvq_k8(sb + warp * kKRec, lane, kv);
                    kvq_v8(sb + KS * kKRec + warp * kVRec, lane, vv);
                }
            } else {
                const float* k_row = ring + static_cast<size_t>(slot) * KS * 2 * kHd + warp * kHd;
                row8(t == pos ? k_s : k_row, lane, kv);
                row8(k_row + KS * kHd, lane, vv);
            }
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
    bar_sync(1, NC);
    // combine the CW warps in warp order: thread tid owns dim tid % 256 of
    // heads tid / 256, tid / 256 + NC / 256, ...
    const size_t pbase = (static_cast<size_t>(g) * a.max_splits + s) * GS;
    const int dd = tid & (kHd - 1);
    for (int i = tid / kHd; i < GS; i += NC / kHd) {
        float M = -INFINITY;
        for (int w = 0; w < CW; ++w) M = fmaxf(M, wml[(w * GS + i) * 2]);
        float L = 0.0f, A = 0.0f;
        for (int w = 0; w < CW; ++w) {
            const float mw = wml[(w * GS + i) * 2];
            const float f = mw == -INFINITY ? 0.0f : expf(mw - M);
            L = fmaf(wml[(w * GS + i) * 2 + 1], f, L);
            A = fmaf(wacc[(w * GS + i) * kHd + dd], f, A);
        }
        a.part_acc[(pbase + i) * kHd + dd] = A;
        if (dd == 0) {
            a.part_ml[(pbase + i) * 2 + 0] = M;
            a.part_ml[(pbase + i) * 2 + 1] = L;
        }
    }
    bar_sync(1, NC);  // every thread's partials are written ...
    if (tid == 0) {
        __threadfence();  // ... and released at gpu scope (cumulative over the barrier), before the arrival
        last_flag = (atomicAdd(a.count + g, 1u) == static_cast<unsigned>(n_act - 1));
    }
    bar_sync(1, NC);
    if (!last_flag) return;
    __threadfence();
    // last CTA of group g: combine the splits in order, then the sigmoid gate
    const size_t hb = static_cast<size_t>(g) * a.max_splits * GS;
    for (int e = tid; e < n_act * GS * 2; e += NC) cml[e] = __ldcg(a.part_ml + hb * 2 + e);
    bar_sync(1, NC);
    // one float4 of a head per job; when the CTA has two threads per job
    // (adjacent lanes), each folds every other split in split order and the
    // pair adds the two sums: half the dependent L2 round trips per thread
    constexpr int JOBS = GS * (kHd / 4);
    constexpr int R = NC >= 2 * JOBS ? 2 : 1;
    for (int jt = tid; jt < R * JOBS; jt += NC) {
        const int job = jt / R, half = jt % R;
        const int i = job / (kHd / 4), d4 = 4 * (job - i * (kHd / 4));
        float M = -INFINITY;
        for (int sp = 0; sp < n_act; ++sp) M = fmaxf(M, cml[(sp * GS + i) * 2]);
        float L = 0.0f;
        float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int sp0 = half; sp0 < n_act; sp0 += 8 * R) {
            float4 v[8];
            float f[8], lw[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int spu = sp0 + R * u;
                const bool in = spu < n_act;
                const int sp = in ? spu : 0;  // split 0 always exists; its term is weighted 0
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
        if constexpr (R == 2) {  // the pair's two sums (every lane of the warp takes part)
            L += __shfl_xor_sync(FULL, L, 1);
            A.x += __shfl_xor_sync(FULL, A.x, 1);
            A.y += __shfl_xor_sync(FULL, A.y, 1);
            A.z += __shfl_xor_sync(FULL, A.z, 1);
            A.w += __shfl_xor_sync(FULL, A.w, 1);
            if (half) continue;
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
static size_t q4_bytes(int n, int k) { return static_cast<size_t>((n + 7) & ~7) * (k / 256) * 144; }
static size_t q6_bytes(int n, int k) { return static_cast<size_t>((n + 7) & ~7) * (k / 256) * 210; }
static L2Prefetch prefetch_of(const void* p0, size_t b0, const void* p1 = nullptr, size_t b1 = 0) {
    L2Prefetch pf{};
    pf.p[0] = static_cast<const uint8_t*>(p0);
    pf.bytes[0] = b0;
    pf.p[1] = static_cast<const uint8_t*>(p1);
    pf.bytes[1] = b1;
    return pf;
}
// Operands of the first kernel of layer il + 1 (or of the lm_head), for the
// L2 prefetch issued by the last kernel of layer il.
static L2Prefetch next_layer_prefetch(const qg_model* m, const qg_state* s, int il) {
    const qg_config& c = m->cfg;
    if (il + 1 >= c.n_layers)  // the lm_head: its first 8 MB
        return prefetch_of(m->lm_head, std::min<size_t>(q6_bytes(c.vocab, c.hidden), 8u << 20));
    const qg_layer_dev& N = m->layers[il + 1];
    if (N.kind == QG_LAYER_DELTANET)
        return prefetch_of(N.w_in, q4_bytes(N.n_in, c.hidden), N.conv_w, sizeof(float) * m->conv_dim * c.conv_kernel);
    return prefetch_of(N.w_in, q4_bytes(N.n_in, c.hidden));
}
// Residual stream: a layer maps (A, pending y) -> (A, pending y') with B as
// the temporary: its first kernel stores A + y (or the embedding row) to B,
// its ffn_up stores B + y_mixer to A; the output GEMVs only store y.
static ProRmsNorm norm_pro(const float* h, const qg_state* s, bool with_y, const float* w, const int* tok,
                           float* h_out, float eps, int k) {
    ProRmsNorm pn{};
    pn.h = h;
    pn.y = with_y ? s->ycur : nullptr;
    pn.y_parts = s->ycur_parts;
    pn.y_stride = s->ycur_stride;
    pn.w = w;
    pn.tok = tok;
    pn.h_out = h_out;
    pn.eps = eps;
    pn.kdim = k;
    return pn;
}

// y = W x for the projections back to the hidden size (ssm_out, attn_output,
// ffn_down): split-K over (slice, 8-row group) tasks when K has several
// slices (the same floats as the one-CTA-per-row path), else the plain engine.
template <int QT, class Pro>
static int out_gemv(qg_state* s, const uint8_t* w, int n, int k, const Pro& pro, cudaStream_t st,
                    const L2Prefetch& next) {
    if (gemv_slices(k) > 1) {
        s->ycur = s->kpart;
        s->ycur_parts = gemv_slices(k);
        s->ycur_stride = (n + 7) & ~7;
        return launch_gemv_split<QT>(w, n, k, pro, st, true, s->err, s->kpart, next);
    }
    s->ycur = s->y;
    s->ycur_parts = 1;
    s->ycur_stride = 0;
    EpiStore ey{};
    ey.y = s->y;
    return launch_gemv<QT, false>(w, nullptr, n, k, pro, ey, st, true, s->err, next);
}

// The pending output of a projection back to the hidden size (ssm_out,
// attn_output, ffn_down) of k inputs, as out_gemv leaves it for the next
// reader: split-K slice sums, or one vector.
static void pending_y(qg_state* s, int n, int k) {
    if (gemv_slices(k) > 1) {
        s->ycur = s->kpart;
        s->ycur_parts = gemv_slices(k);
        s->ycur_stride = (n + 7) & ~7;
    } else {
        s->ycur = s->y;
        s->ycur_parts = 1;
        s->ycur_stride = 0;
    }
}

// ----------------------------------------------- the kernels of one layer
// FFN gate/up: RMSNorm prologue of io.b + the pending y (the mixer's output),
// storing the stream to io.a; dual GEMV with the SwiGLU epilogue.
static int launch_ffn_up(const qg_model* m, qg_state* s, int il, const ResidualIO& io, cudaStream_t st) {
    const qg_config& c = m->cfg;
    const qg_layer_dev& L = m->layers[il];
    EpiSwiGlu sw{};
    sw.act = s->act;
    return launch_gemv<QT_Q4K, true>(L.w_gate, L.w_up, c.ffn, c.hidden,
                                     norm_pro(io.b, s, true, L.post_norm, nullptr, io.a, c.eps, c.hidden), sw, st, true,
                                     s->err, prefetch_of(L.w_down, q6_bytes(c.hidden, c.ffn)));
}

// FFN down (Q6_K, split-K over the hidden rows): y pending for the next layer.
static int launch_ffn_down(const qg_model* m, qg_state* s, int il, cudaStream_t st) {
    const qg_config& c = m->cfg;
    return out_gemv<QT_Q6K>(s, m->layers[il].w_down, c.hidden, c.ffn, ProPlainG{s->act}, st,
                            next_layer_prefetch(m, s, il));
}

static ProRmsNorm input_norm(const qg_model* m, qg_state* s, const qg_layer_dev& L, const ResidualIO& io) {
    if (io.embed) return norm_pro(m->embd, s, false, L.attn_norm, s->slots, io.b, m->cfg.eps, m->cfg.hidden);
    return norm_pro(io.a, s, io.y_pending, L.attn_norm, nullptr, io.b, m->cfg.eps, m->cfg.hidden);
}

// DeltaNet input: RMSNorm prologue + the fused [qkv | alpha | beta | gate]
// GEMV with the conv / gates / z epilogue.
static int launch_dn_in(const qg_model* m, qg_state* s, int il, const ResidualIO& io, cudaStream_t st, bool pdl) {
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
    return launch_gemv<QT_Q4K, false>(L.w_in, nullptr, L.n_in, c.hidden, input_norm(m, s, L, io), ei, st, pdl, s->err,
                                      prefetch_of(s->ssm[il], sizeof(float) * c.n_v_heads * c.head_v_dim * kDk));
}

static int launch_delta(const qg_model* m, qg_state* s, int il, cudaStream_t st) {
    const qg_config& c = m->cfg;
    const qg_layer_dev& L = m->layers[il];
    DeltaArgs da{};
    da.conv_out = s->conv_out;
    da.dt = s->dt;
    da.beta = s->beta;
    da.S = s->ssm[il];
    da.o = s->o;
    da.err = s->err;
    da.next = prefetch_of(L.w_out, q4_bytes(c.hidden, m->v_dim));
    da.nk = c.n_k_heads;
    da.dv = c.head_v_dim;
    da.kdim = m->k_dim;
    da.eps = c.eps;
    return launch_pdl(delta_kernel, dim3(c.n_v_heads * (c.head_v_dim / kDeltaRows)), dim3(256), 0, st, true, da);
}

// ssm_out: gated-RMSNorm prologue (per value head, on o and z) + GEMV.
static int launch_ssm_out(const qg_model* m, qg_state* s, int il, cudaStream_t st) {
    const qg_config& c = m->cfg;
    const qg_layer_dev& L = m->layers[il];
    ProGatedNorm gn{};
    gn.o = s->o;
    gn.z = s->z;
    gn.w = L.ssm_norm;
    gn.nv = c.n_v_heads;
    gn.dv = c.head_v_dim;
    gn.eps = c.eps;
    return out_gemv<QT_Q4K>(s, L.w_out, c.hidden, m->v_dim, gn, st,
                            prefetch_of(L.w_gate, q4_bytes(c.ffn, c.hidden), L.w_up, q4_bytes(c.ffn, c.hidden)));
}

int run_deltanet_layer(const qg_model* m, qg_state* s, int il, const ResidualIO& io, cudaStream_t st, bool pdl_first) {
    int rc;
    if ((rc = launch_dn_in(m, s, il, io, st, pdl_first)) || (rc = launch_delta(m, s, il, st)) ||
        (rc = launch_ssm_out(m, s, il, st)) || (rc = launch_ffn_up(m, s, il, io, st)))
        return rc;
    return launch_ffn_down(m, s, il, st);
}

// Grid (rows, n_kv): one CTA per (position, kv head), warp w makes block w
// of its K and V records with the append's quantizer.
__global__ void __launch_bounds__(256) kv_quantize_kernel(const float* __restrict__ k, const float* __restrict__ v,
                                                          int n_kv, int max_seq, int pos0, const int* pos0_dev,
                                                          uint8_t* kq, uint8_t* vq) {
    const int t = blockIdx.x, g = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t src = (static_cast<size_t>(t) * n_kv + g) * kHd + 32 * warp + lane;
    const int base = pos0_dev ? *pos0_dev : pos0;  // first position: an argument, or read on the device
    const size_t rec = static_cast<size_t>(g) * max_seq + base + t;
    kvq_put_q8_0(k[src], lane, warp, kq + rec * kKRec);
    kvq_put_q5_1(v[src], lane, warp, vq + rec * kVRec);
}

int kv_quantize_rows(const float* k, const float* v, int rows, int n_kv, int max_seq, uint8_t* kq, uint8_t* vq,
                     cudaStream_t st) {
    return kv_quantize_rows_at(k, v, rows, 0, n_kv, max_seq, kq, vq, st);
}

int kv_quantize_rows_at(const float* k, const float* v, int rows, int pos0, int n_kv, int max_seq, uint8_t* kq,
                        uint8_t* vq, cudaStream_t st) {
    if (rows <= 0) return QG_OK;
    if (pos0 < 0 || pos0 + rows > max_seq) return set_err(QG_ERR_POS, "kv_quantize: rows past the cache");
    kv_quantize_kernel<<<dim3(rows, n_kv), 256, 0, st>>>(k, v, n_kv, max_seq, pos0, nullptr, kq, vq);
    QG_CUDA(cudaGetLastError());
    return QG_OK;
}

int kv_quantize_rows_dev(const float* k, const float* v, int rows, const int* pos0_dev, int n_kv, int max_seq,
                         uint8_t* kq, uint8_t* vq, cudaStream_t st) {
    if (rows <= 0) return QG_OK;
    kv_quantize_kernel<<<dim3(rows, n_kv), 256, 0, st>>>(k, v, n_kv, max_seq, 0, pos0_dev, kq, vq);
    QG_CUDA(cudaGetLastError());
    return QG_OK;
}

size_t kv_cache_bytes(const qg_state* s, int which) {
    const qg_model* m = s->m;
    if (s->kv_format == QG_KV_Q8_0_Q5_1)
        return static_cast<size_t>(m->cfg.n_kv_heads) * s->max_seq * (which == 0 ? kKRec : kVRec);
    return sizeof(float) * static_cast<size_t>(s->max_seq) * m->kv_dim;
}

template <int GS, bool KVQ, int CW>
static int launch_attn_as(const qg_model* m, qg_state* s, const AttnArgs& a, cudaStream_t st) {
    const int smem = attn_smem_floats<GS, KVQ, CW>() * 4;
    if (int rc = grant_smem(reinterpret_cast<const void*>(attn_kernel<GS, KVQ, CW>), smem)) return rc;
    return launch_pdl(attn_kernel<GS, KVQ, CW>, dim3(s->max_splits, m->cfg.n_kv_heads), dim3(32 * (CW + 1)), smem, st,
                      true, a);
}

template <int GS, bool KVQ>
static int launch_attn_w(const qg_model* m, qg_state* s, const AttnArgs& a, cudaStream_t st) {
    if constexpr (GS <= 4) return launch_attn_as<GS, KVQ, 16>(m, s, a, st);
    else return launch_attn_as<GS, KVQ, 8>(m, s, a, st);
}

template <int GS>
static int launch_attn(const qg_model* m, qg_state* s, const AttnArgs& a, cudaStream_t st) {
    return s->kv_format == QG_KV_Q8_0_Q5_1 ? launch_attn_w<GS, true>(m, s, a, st) : launch_attn_w<GS, false>(m, s, a, st);
}

// Attention input: RMSNorm prologue + the fused [q|gate | k | v] GEMV; v rows
// land in the V cache row at the step's position.
static int launch_attn_in(const qg_model* m, qg_state* s, int il, const ResidualIO& io, cudaStream_t st, bool pdl) {
    const qg_config& c = m->cfg;
    const qg_layer_dev& L = m->layers[il];
    EpiAttnIn ea{};
    ea.qf = s->qf;
    ea.kraw = s->kraw;
    ea.vcache = s->vc[il];
    ea.vraw = s->kv_format == QG_KV_Q8_0_Q5_1 ? s->vraw : nullptr;
    ea.slots = s->slots;
    ea.qd2 = 2 * m->q_dim;
    ea.kvd = m->kv_dim;
    return launch_gemv<QT_Q4K, false>(L.w_in, nullptr, L.n_in, c.hidden, input_norm(m, s, L, io), ea, st, pdl, s->err);
}

static int launch_attention(const qg_model* m, qg_state* s, int il, cudaStream_t st) {
    const qg_config& c = m->cfg;
    const qg_layer_dev& L = m->layers[il];
    AttnArgs a{};
    a.kmap = s->kmap[il];
    a.vmap = s->vmap[il];
    a.next = prefetch_of(L.w_out, q4_bytes(c.hidden, m->q_dim));
    a.qf = s->qf;
    a.kraw = s->kraw;
    a.kc = s->kc[il];
    a.vc = s->vc[il];
    a.vraw = s->vraw;
    a.max_seq = s->max_seq;
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
        case 1: return launch_attn<1>(m, s, a, st);
        case 2: return launch_attn<2>(m, s, a, st);
        case 4: return launch_attn<4>(m, s, a, st);
        case 8: return launch_attn<8>(m, s, a, st);
        default: return set_err(QG_ERR_SHAPE, "attention: %d query heads per kv head", c.n_heads / c.n_kv_heads);
    }
}

static int launch_attn_out(const qg_model* m, qg_state* s, int il, cudaStream_t st) {
    const qg_config& c = m->cfg;
    const qg_layer_dev& L = m->layers[il];
    return out_gemv<QT_Q4K>(s, L.w_out, c.hidden, m->q_dim, ProPlainG{s->attn}, st,
                            prefetch_of(L.w_gate, q4_bytes(c.ffn, c.hidden), L.w_up, q4_bytes(c.ffn, c.hidden)));
}

int encode_kv_maps(qg_state* s) {
    const qg_model* m = s->m;
    const int n = m->cfg.n_layers;
    s->kmap.assign(n, CUtensorMap{});
    s->vmap.assign(n, CUtensorMap{});
    if (s->kv_format != QG_KV_F32) return QG_OK;
    using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    static Encode encode = nullptr;
    if (!encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        QG_CUDA(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q));
        if (q != cudaDriverEntryPointSuccess || !fn)
            return set_err(QG_ERR_CUDA, "the driver has no cuTensorMapEncodeTiled");
        encode = reinterpret_cast<Encode>(fn);
    }
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(m->kv_dim), static_cast<cuuint64_t>(s->max_seq)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(m->kv_dim) * sizeof(float)};
    const int gs = m->cfg.n_kv_heads > 0 ? m->cfg.n_heads / m->cfg.n_kv_heads : 1;
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kHd), static_cast<cuuint32_t>(attn_warps(gs))};
    const cuuint32_t estr[2] = {1, 1};
    for (int il = 0; il < n; ++il) {
        if (m->kinds[il] != QG_LAYER_ATTENTION) continue;
        for (int which = 0; which < 2; ++which) {
            CUtensorMap* map = which ? &s->vmap[il] : &s->kmap[il];
            const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, which ? s->vc[il] : s->kc[il], dims,
                                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) return set_err(QG_ERR_CUDA, "cuTensorMapEncodeTiled: error %d (layer %d)", r, il);
        }
    }
    return QG_OK;
}

int run_attention_layer(const qg_model* m, qg_state* s, int il, const ResidualIO& io, cudaStream_t st,
                        bool pdl_first) {
    int rc;
    if ((rc = launch_attn_in(m, s, il, io, st, pdl_first)) || (rc = launch_attention(m, s, il, st)) ||
        (rc = launch_attn_out(m, s, il, st)) || (rc = launch_ffn_up(m, s, il, io, st)))
        return rc;
    return launch_ffn_down(m, s, il, st);
}

// Measurement: `launches` launches of one kernel kind, PDL-chained on st,
// walking the layers that have it (for kernels that read the previous
// kernel's pending output, the bookkeeping of that predecessor is set first,
// so every launch runs exactly the configuration it has inside the step).
int run_kernel_kind(const qg_model* m, qg_state* s, int kind, int launches, cudaStream_t st) {
    const qg_config& c = m->cfg;
    std::vector<int> layers;
    for (int il = 0; il < c.n_layers; ++il) {
        const bool dn = m->kinds[il] == QG_LAYER_DELTANET;
        const bool has = kind == QG_KERNEL_FFN_UP || kind == QG_KERNEL_FFN_DOWN ||
                         ((kind == QG_KERNEL_DN_IN || kind == QG_KERNEL_DELTA || kind == QG_KERNEL_SSM_OUT) && dn) ||
                         ((kind == QG_KERNEL_ATTN_IN || kind == QG_KERNEL_ATTN || kind == QG_KERNEL_ATTN_OUT) && !dn);
        if (has) layers.push_back(il);
    }
    if (kind == QG_KERNEL_LMHEAD) layers.push_back(c.n_layers - 1);
    if (layers.empty() || kind < 0 || kind > QG_KERNEL_LMHEAD)
        return set_err(QG_ERR_ARG, "bench_kernel: kernel kind %d does not occur in this model", kind);
    const ResidualIO io{s->hres, s->h, true, false};
    for (int i = 0; i < launches; ++i) {
        const int il = layers[static_cast<size_t>(i) % layers.size()];
        const bool dn = m->kinds[il] == QG_LAYER_DELTANET;
        int rc = QG_OK;
        switch (kind) {
            case QG_KERNEL_DN_IN:
            case QG_KERNEL_ATTN_IN:
                pending_y(s, c.hidden, c.ffn);  // after the previous layer's ffn_down
                rc = dn ? launch_dn_in(m, s, il, io, st, true) : launch_attn_in(m, s, il, io, st, true);
                break;
            case QG_KERNEL_DELTA: rc = launch_delta(m, s, il, st); break;
            case QG_KERNEL_SSM_OUT: rc = launch_ssm_out(m, s, il, st); break;
            case QG_KERNEL_ATTN: rc = launch_attention(m, s, il, st); break;
            case QG_KERNEL_ATTN_OUT: rc = launch_attn_out(m, s, il, st); break;
            case QG_KERNEL_FFN_UP:
                pending_y(s, c.hidden, dn ? m->v_dim : m->q_dim);  // after the mixer's output projection
                rc = launch_ffn_up(m, s, il, io, st);
                break;
            case QG_KERNEL_FFN_DOWN: rc = launch_ffn_down(m, s, il, st); break;
            default:
                pending_y(s, c.hidden, c.ffn);
                rc = run_lmhead(m, s, s->hres, s->h, st, false);
                break;
        }
        if (rc) return rc;
    }
    return QG_OK;
}

int run_residual(qg_state* s, float* h, int n, cudaStream_t st) {
    return launch_pdl(residual_add_kernel, dim3((n + 255) / 256), dim3(256), 0, st, true, h, s->ycur, s->ycur_parts,
                      s->ycur_stride, n);
}

int run_lmhead(const qg_model* m, qg_state* s, const float* a, float* h_final, cudaStream_t st, bool advance) {
    const qg_config& c = m->cfg;
    EpiArgmaxStep ea{};
    ea.ws = s->am_ws;
    ea.slots = s->slots;
    ea.hist = s->hist;
    ea.err = s->err;
    ea.allow = s->allow;
    ea.advance = advance ? 1 : 0;
    return launch_gemv<QT_Q6K, false>(m->lm_head, nullptr, c.vocab, c.hidden,
                                      norm_pro(a, s, true, m->out_norm, nullptr, h_final, c.eps, c.hidden), ea, st, true,
                                      s->err);
}

// Output norm of a (no pending y; stored to s->h) + fused lm_head GEMV + argmax
// -> slots[0] / slots[2]; no history, no position move (the end of a prefill).
int run_lmhead_of(const qg_model* m, qg_state* s, const float* a, cudaStream_t st) {
    const qg_config& c = m->cfg;
    EpiArgmaxStep ea{};
    ea.ws = s->am_ws;
    ea.slots = s->slots;
    ea.hist = s->hist;
    ea.err = s->err;
    ea.allow = s->allow;
    ea.advance = 0;
    return launch_gemv<QT_Q6K, false>(m->lm_head, nullptr, c.vocab, c.hidden,
                                      norm_pro(a, s, false, m->out_norm, nullptr, s->h, c.eps, c.hidden), ea, st,
                                      false, s->err);
}

}  // namespace qg
