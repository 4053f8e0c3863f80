// The whole decode step as one persistent kernel: the GB300 form of
// forward_qwen35_cuda.rs forward_single / forward_single_greedy.
//
// One cooperative launch per token.  Every CTA (two per SM: 8 consumer warps
// + 1 producer warp each, as in the GEMV engine) stays resident for the whole
// step, which is a fixed sequence of phases -- per layer: input projection,
// mixer (delta rule or attention), output projection, ffn gate/up, ffn down;
// then the lm_head GEMV + argmax -- separated by grid-wide barriers: every
// phase needs all of its predecessor's output (a GEMV reads its whole input
// vector), so nothing finer than a barrier would do.
//
// Weights do not depend on the activations.  The producer warp of each CTA
// walks the same phase sequence ahead of its consumers and streams the CTA's
// share of every phase -- weight rows, DeltaNet state rows, K/V cache rows of
// earlier positions -- into a ring of 16 KB shared-memory slots with bulk
// copies, without waiting for any barrier: HBM keeps streaming while the grid
// synchronises, and a phase's weights are mostly on chip when it starts.
//
// The consumers run each phase with the arithmetic of the per-layer kernels
// (same lane partition of every dot product, same reduction orders), so a
// step here is bit-identical to the kernel-by-kernel step.
#include <algorithm>
#include <cstring>

#include "qg_layers.cuh"
#include "qg_step.cuh"

namespace qg {

__device__ __forceinline__ bool aborted(const StepParams& P) { return __ldcg(P.gbar + 2) != 0u; }

__device__ __forceinline__ void raise_abort(const StepParams& P, unsigned bit) {
    atomicOr(P.err, bit);
    atomicExch(P.gbar + 2, 1u);
}

// ============================================================== producer
// The whole producer warp runs these (lane-uniform control flow); the pipe's
// lane 0 owns the mbarrier protocol, the lanes issue a stage's copies in
// parallel.  Weight stages come from the GEMV engine's gemv_produce.

// DeltaNet state rows: item = (value head h, 32 rows), one 16 KB stage.
__device__ bool produce_delta(Pipe& pr, const StepParams& P, const StepLayer& L) {
    const int per_head = P.dv / 32, items = P.nv * per_head;
    for (int it = blockIdx.x; it < items; it += gridDim.x) {
        const int h = it / per_head, jb = (it - h * per_head) * 32;
        if (!pr.acquire()) return false;
        pr.expect(32u * kDk * 4u);
        if (pr.lane == 0) pr.copy(pr.cur(), L.ssm + (static_cast<size_t>(h) * P.dv + jb) * kDk, 32u * kDk * 4u);
        pr.commit();
    }
    return true;
}

// K/V rows of earlier positions: item = (kv group, split), 8 keys per stage;
// row pos (appended by this step) is read by the consumers themselves.
__device__ bool produce_attn(Pipe& pr, const StepParams& P, const StepLayer& L, int pos) {
    const int n_act = (pos + P.T) / P.T, items = P.n_kv * n_act;
    for (int it = blockIdx.x; it < items; it += gridDim.x) {
        const int g = it % P.n_kv, s = it / P.n_kv;
        const int t0 = s * P.T, t1 = min(t0 + P.T, pos + 1);
        for (int k0 = t0; k0 < t1; k0 += kKeysPerStage) {
            const int k1 = min(k0 + kKeysPerStage, t1);
            if (!pr.acquire()) return false;
            const int nk = k1 - k0 - ((pos >= k0 && pos < k1) ? 1 : 0);
            pr.expect(static_cast<unsigned>(nk) * 2u * kHd * 4u);
            float* st = reinterpret_cast<float*>(pr.cur());
            for (int i = pr.lane; i < 2 * (k1 - k0); i += 32) {
                const int t = k0 + (i >> 1), which = i & 1;
                if (t == pos) continue;
                const size_t off = static_cast<size_t>(t) * P.kv_dim + g * kHd;
                pr.copy(st + (t - k0) * 2 * kHd + which * kHd, (which ? L.vc : L.kc) + off, kHd * 4u);
            }
            pr.commit();
        }
    }
    return true;
}

template <int QT, bool DUAL>
__device__ bool produce_gemv(Pipe& pr, const GemvShape& g, const uint8_t* w0, const uint8_t* w1) {
    int r0, r1;
    cta_rows(g.units, g.n, r0, r1);
    return gemv_produce<QT, LAYOUT_GROUPED, DUAL>(pr, g, w0, w1, r0, r1, nullptr);
}

__device__ void producer_main(Pipe& pr, const StepParams& P, int pos) {
    bool ok = true;
    for (int il = 0; il < P.n_layers && ok; ++il) {
        const StepLayer& L = P.L[il];
        if (L.kind == QG_LAYER_DELTANET) {
            ok = produce_gemv<QT_Q4K, false>(pr, P.geo[SG_DN_IN], L.w_in, nullptr) && produce_delta(pr, P, L) &&
                 produce_gemv<QT_Q4K, false>(pr, P.geo[SG_SSM_OUT], L.w_out, nullptr);
        } else {
            ok = produce_gemv<QT_Q4K, false>(pr, P.geo[SG_ATTN_IN], L.w_in, nullptr) && produce_attn(pr, P, L, pos) &&
                 produce_gemv<QT_Q4K, false>(pr, P.geo[SG_ATTN_OUT], L.w_out, nullptr);
        }
        ok = ok && produce_gemv<QT_Q4K, true>(pr, P.geo[SG_FFN_UP], L.w_gate, L.w_up) &&
             produce_gemv<QT_Q6K, false>(pr, P.geo[SG_FFN_DOWN], L.w_down, nullptr);
    }
    if (ok) ok = produce_gemv<QT_Q6K, false>(pr, P.geo[SG_LMHEAD], P.lm_head, nullptr);
    if (!ok) pr.drain();
}

// ============================================================== consumers
// Control flow stays uniform across the consumer warps whatever happens: a
// failed wait raises the step-wide abort flag and the phase runs on (every
// later wait then returns at once) up to the next grid barrier, which every
// CTA leaves through its abort exit.
struct Consumer {
    Pipe R;
    uint8_t* smem;  // dynamic shared memory base (scratch at off_dig())
    int tid, warp, lane;
    int* flag;      // shared int for CTA-wide decisions
    bool ok;        // false once the step is aborted (uniform after a grid barrier)
    __device__ void wait_full() const { R.wait_full(); }
    __device__ void release() { R.release(); }
};

// Grid-wide barrier number `nbar` (1-based) among the consumer groups.
__device__ bool grid_sync(Consumer& c, const StepParams& P, unsigned nbar) {
    bar_sync(1, kConsumers);
    if (c.tid == 0) {
        int good = aborted(P) ? 0 : 1;
        if (good) {
            red_release_add_gpu(P.gbar, 1u);  // orders this CTA's phase output before the arrival
            const unsigned target = nbar * gridDim.x;
            if (ld_relaxed_gpu(P.gbar) < target) {
                const long long t0 = clock64();
                int n = 0;
                while (ld_relaxed_gpu(P.gbar) < target) {
                    if ((n++ & 63) == 0 && aborted(P)) {
                        good = 0;
                        break;
                    }
                    if (clock64() - t0 > kWaitCycles) {
                        raise_abort(P, DEVERR_GRID_WAIT);
                        good = 0;
                        break;
                    }
                }
            }
            fence_acq_rel_gpu();  // the other CTAs' phase output is visible from here on
        }
        *c.flag = good;
    }
    bar_sync(1, kConsumers);
    c.ok = *c.flag != 0;
    return c.ok;
}

template <int QT, bool DUAL, class Pro, class Epi>
__device__ void consume_gemv(Consumer& c, const GemvShape& g, Pro pro, Epi epi) {
    int r0, r1;
    cta_rows(g.units, g.n, r0, r1);
    epi.pre(r0, r1, c.tid);
    pro.pre(reinterpret_cast<float*>(c.smem + off_pro(QT, g.k)), g.k, c.tid);
    gemv_consume<QT, LAYOUT_GROUPED, DUAL>(c.R, g, r0, r1, pro, epi, c.smem, c.tid);
}

// Delta rule, item = (value head h, rows jb..jb+31), four rows per warp; the
// rows' o (before the gated norm, which the ssm_out prologue applies) go to P.o.
__device__ void consume_delta(Consumer& c, const StepParams& P, const StepLayer& L) {
    float* qs = reinterpret_cast<float*>(c.smem + off_dig());
    float* ks = qs + kDk;
    const int per_head = P.dv / 32, items = P.nv * per_head;
    for (int it = blockIdx.x; it < items; it += gridDim.x) {
        const int h = it / per_head, jb = (it - h * per_head) * 32;
        const int kh = h % P.nk;
        if (c.warp < 2) {  // per-head L2 norm of q (warp 0) and k (warp 1) (gdn_per_head_l2_norm_into)
            const float4 v = ldcg4(P.conv_out + (c.warp ? P.k_dim : 0) + kh * kDk + 4 * c.lane);
            float ss = v.x * v.x;
            ss = fmaf(v.y, v.y, ss);
            ss = fmaf(v.z, v.z, ss);
            ss = fmaf(v.w, v.w, ss);
            ss = warp_sum(ss);
            const float r = 1.0f / sqrtf(ss + P.eps);
            float* dst = c.warp ? ks : qs;
            *reinterpret_cast<float4*>(dst + 4 * c.lane) = make_float4(v.x * r, v.y * r, v.z * r, v.w * r);
        }
        const int j = jb + 4 * c.warp;  // this warp's first row
        const float vl = c.lane < 4 ? __ldcg(P.conv_out + 2 * P.k_dim + h * P.dv + j + c.lane) : 0.0f;
        const float g = expf(__ldcg(P.dt + h)), be = __ldcg(P.beta + h);
        bar_sync(1, kConsumers);
        c.wait_full();
        const float* st = reinterpret_cast<const float*>(c.R.cur());
        const float4 kk = *reinterpret_cast<const float4*>(ks + 4 * c.lane);
        const float4 qq = *reinterpret_cast<const float4*>(qs + 4 * c.lane);
        float o[4];
        delta_rows4(st + 4 * c.warp * kDk, L.ssm + (static_cast<size_t>(h) * P.dv + j) * kDk, kk, qq, vl, 0, g, be,
                    c.lane, o);
        float mine = 0.0f;
#pragma unroll
        for (int t = 0; t < 4; ++t)
            if (c.lane == t) mine = o[t];
        if (c.lane < 4) P.o[h * P.dv + j + c.lane] = mine;
        c.release();
        bar_sync(1, kConsumers);  // qs / ks are rewritten by the next item
    }
}

// Split-K GQA decode attention, item = (kv group g, split s): the arithmetic
// of attn_kernel (q/k RMSNorm, partial NEOX rope, K append, online softmax per
// warp, warp combine, split partials, last-CTA split combine + sigmoid gate).
template <int GS>
__device__ void consume_attn(Consumer& c, const StepParams& P, const StepLayer& L, int pos) {
    float* q_s = reinterpret_cast<float*>(c.smem + off_dig());  // [GS][hd]
    float* k_s = q_s + GS * kHd;                                // [hd]
    float* cs = k_s + kHd;
    float* sn = cs + kHd / 2;
    float* wml = sn + kHd / 2;       // [8][GS][2]
    float* wacc = wml + 8 * GS * 2;  // [8][GS][hd]
    float* cml = wacc + 8 * GS * kHd;  // [64][GS][2]
    const int tid = c.tid, warp = c.warp, lane = c.lane;
    const int t_len = pos + 1, n_act = (t_len + P.T - 1) / P.T, items = P.n_kv * n_act;
    const int half = P.n_rot / 2;
    for (int it = blockIdx.x; it < items; it += gridDim.x) {
        const int g = it % P.n_kv, s = it / P.n_kv;
        const bool has_new = (s == n_act - 1);
        const int t0 = s * P.T, t1 = min(t0 + P.T, t_len);
        const int nst = (t1 - t0 + kKeysPerStage - 1) / kKeysPerStage;
        if (tid < half) {  // theta_0 = pos, theta_{i+1} = theta_i * theta_scale
            float th = static_cast<float>(pos);
            for (int i = 0; i < tid; ++i) th = th * P.theta_scale;
            float sv, cv;
            sincosf(th, &sv, &cv);
            cs[tid] = cv;
            sn[tid] = sv;
        }
        for (int job = warp; job < GS + (has_new ? 1 : 0); job += 8) {  // per_head_rmsnorm_into
            const float* src = job < GS ? P.qf + static_cast<size_t>(g * GS + job) * 2 * kHd : P.kraw + g * kHd;
            const float* w = job < GS ? L.q_norm : L.k_norm;
            float* dst = job < GS ? q_s + job * kHd : k_s;
            float v[8];
            load_row8(src, lane, v);
            float ss = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) ss = fmaf(v[i], v[i], ss);
            ss = warp_sum(ss);
            const float r = 1.0f / sqrtf(ss / static_cast<float>(kHd) + P.eps);
#pragma unroll
            for (int i = 0; i < 8; ++i) dst[dim8(lane, i)] = (v[i] * r) * __ldg(w + dim8(lane, i));
        }
        bar_sync(1, kConsumers);
        const int jobs = GS + (has_new ? 1 : 0);
        for (int p = tid; p < jobs * half; p += kConsumers) {  // gdn_partial_neox_rope_into
            const int job = p / half, i = p - job * half;
            float* vec = job < GS ? q_s + job * kHd : k_s;
            const float x0 = vec[i], x1 = vec[i + half];
            vec[i] = x0 * cs[i] - x1 * sn[i];
            vec[i + half] = x0 * sn[i] + x1 * cs[i];
        }
        bar_sync(1, kConsumers);
        if (has_new) L.kc[static_cast<size_t>(pos) * P.kv_dim + g * kHd + tid] = k_s[tid];  // K append at pos

        float m[GS], l[GS], acc[GS][8];
#pragma unroll
        for (int i = 0; i < GS; ++i) {
            m[i] = -INFINITY;
            l[i] = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
        }
        const float scale = 1.0f / sqrtf(static_cast<float>(kHd));
        for (int stg = 0; stg < nst; ++stg) {
            c.wait_full();
            const int t = t0 + stg * kKeysPerStage + warp;
            if (t < t1) {
                const float* kv_row = reinterpret_cast<const float*>(c.R.cur()) + warp * 2 * kHd;
                float kv[8], vv[8];
                row8(t == pos ? k_s : kv_row, lane, kv);
                if (t == pos) load_row8(L.vc + static_cast<size_t>(pos) * P.kv_dim + g * kHd, lane, vv);
                else row8(kv_row + kHd, lane, vv);
#pragma unroll
                for (int i = 0; i < GS; ++i) {
                    float dot = 0.0f;
#pragma unroll
                    for (int j = 0; j < 8; ++j) dot = fmaf(q_s[i * kHd + dim8(lane, j)], kv[j], dot);
                    const float sc = warp_sum(dot) * scale;
                    const float mn = fmaxf(m[i], sc);
                    const float cc = expf(m[i] - mn), p = expf(sc - mn);
                    l[i] = fmaf(l[i], cc, p);
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(acc[i][j], cc, p * vv[j]);
                    m[i] = mn;
                }
            }
            c.release();
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
        bar_sync(1, kConsumers);
        const size_t pbase = (static_cast<size_t>(g) * P.max_splits + s) * GS;
        for (int i = 0; i < GS; ++i) {
            float M = -INFINITY;
            for (int w = 0; w < 8; ++w) M = fmaxf(M, wml[(w * GS + i) * 2]);
            float Lsum = 0.0f, A = 0.0f;
            for (int w = 0; w < 8; ++w) {
                const float mw = wml[(w * GS + i) * 2];
                const float f = mw == -INFINITY ? 0.0f : expf(mw - M);
                Lsum = fmaf(wml[(w * GS + i) * 2 + 1], f, Lsum);
                A = fmaf(wacc[(w * GS + i) * kHd + tid], f, A);
            }
            P.part_acc[(pbase + i) * kHd + tid] = A;
            if (tid == 0) {
                P.part_ml[(pbase + i) * 2 + 0] = M;
                P.part_ml[(pbase + i) * 2 + 1] = Lsum;
            }
        }
        __threadfence();
        bar_sync(1, kConsumers);
        if (tid == 0) *c.flag = (atomicAdd(P.attn_count + g, 1u) == static_cast<unsigned>(n_act - 1));
        bar_sync(1, kConsumers);
        const bool last = *c.flag != 0;
        if (last) {  // combine the splits of group g in order, then the sigmoid gate
            __threadfence();
            const size_t hb = static_cast<size_t>(g) * P.max_splits * GS;
            for (int e = tid; e < n_act * GS * 2; e += kConsumers) cml[e] = __ldcg(P.part_ml + hb * 2 + e);
            bar_sync(1, kConsumers);
            for (int job = tid; job < GS * (kHd / 4); job += kConsumers) {
                const int i = job / (kHd / 4), d4 = 4 * (job - i * (kHd / 4));
                float M = -INFINITY;
                for (int sp = 0; sp < n_act; ++sp) M = fmaxf(M, cml[(sp * GS + i) * 2]);
                float Lsum = 0.0f;
                float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int sp0 = 0; sp0 < n_act; sp0 += 8) {
                    float4 v[8];
                    float f[8], lw[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const bool in = sp0 + u < n_act;
                        const int sp = in ? sp0 + u : sp0;
                        v[u] = __ldcg(reinterpret_cast<const float4*>(P.part_acc + (hb + sp * GS + i) * kHd + d4));
                        f[u] = in ? expf(cml[(sp * GS + i) * 2] - M) : 0.0f;
                        lw[u] = cml[(sp * GS + i) * 2 + 1];
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        Lsum = fmaf(lw[u], f[u], Lsum);
                        A.x = fmaf(v[u].x, f[u], A.x);
                        A.y = fmaf(v[u].y, f[u], A.y);
                        A.z = fmaf(v[u].z, f[u], A.z);
                        A.w = fmaf(v[u].w, f[u], A.w);
                    }
                }
                const int h = g * GS + i;
                const float4 gt =
                    __ldcg(reinterpret_cast<const float4*>(P.qf + static_cast<size_t>(h) * 2 * kHd + kHd + d4));
                float4 o;  // (A / L) * sigmoid(gate)  (gdn_sigmoid_gate_into)
                o.x = (A.x / Lsum) * sigmoid(gt.x);
                o.y = (A.y / Lsum) * sigmoid(gt.y);
                o.z = (A.z / Lsum) * sigmoid(gt.z);
                o.w = (A.w / Lsum) * sigmoid(gt.w);
                *reinterpret_cast<float4*>(P.attn + h * kHd + d4) = o;
            }
            if (tid == 0) P.attn_count[g] = 0u;
        }
        bar_sync(1, kConsumers);  // q_s / k_s / cml are rewritten by the next item
    }
}

__device__ ProRmsNorm step_norm(const float* h, const float* y, const float* w, const int* tok, float* h_out,
                                const StepParams& P) {
    ProRmsNorm pn{};
    pn.h = h;
    pn.y = y;
    pn.w = w;
    pn.tok = tok;
    pn.h_out = h_out;
    pn.eps = P.eps;
    pn.kdim = P.hidden;
    pn.y_parts = 1;
    pn.y_stride = 0;
    return pn;
}

__device__ void consumer_main(Consumer& c, const StepParams& P, int pos) {
    unsigned nbar = 0;
    // residual stream: layer maps (A = hres, pending y) -> (A, pending y'),
    // with B = h as its temporary; the first layer reads the embedding row
    float* A = P.hres;
    float* B = P.h;
    for (int il = 0; il < P.n_layers; ++il) {
        const StepLayer& L = P.L[il];
        const ProRmsNorm in_norm = il == 0 ? step_norm(P.embd, nullptr, L.attn_norm, P.slots, B, P)
                                           : step_norm(A, P.y, L.attn_norm, nullptr, B, P);
        if (L.kind == QG_LAYER_DELTANET) {
            EpiDnIn ei{};
            ei.C = P.conv_dim;
            ei.nv = P.nv;
            ei.K = P.conv_k;
            ei.win = L.conv;
            ei.wconv = L.conv_w;
            ei.conv_out = P.conv_out;
            ei.dt_bias = L.dt_bias;
            ei.a = L.a;
            ei.dt = P.dt;
            ei.beta = P.beta;
            ei.z = P.z;
            consume_gemv<QT_Q4K, false>(c, P.geo[SG_DN_IN], in_norm, ei);
            if (!grid_sync(c, P, ++nbar)) return;
            consume_delta(c, P, L);
            if (!grid_sync(c, P, ++nbar)) return;
            ProGatedNorm gn{};
            gn.o = P.o;
            gn.z = P.z;
            gn.w = L.ssm_norm;
            gn.nv = P.nv;
            gn.dv = P.dv;
            gn.eps = P.eps;
            EpiStore ey{};
            ey.y = P.y;
            consume_gemv<QT_Q4K, false>(c, P.geo[SG_SSM_OUT], gn, ey);
        } else {
            EpiAttnIn ea{};
            ea.qf = P.qf;
            ea.kraw = P.kraw;
            ea.vcache = L.vc;
            ea.slots = P.slots;
            ea.qd2 = 2 * P.q_dim;
            ea.kvd = P.kv_dim;
            consume_gemv<QT_Q4K, false>(c, P.geo[SG_ATTN_IN], in_norm, ea);
            if (!grid_sync(c, P, ++nbar)) return;
            switch (P.gs) {
                case 1: consume_attn<1>(c, P, L, pos); break;
                case 2: consume_attn<2>(c, P, L, pos); break;
                default: consume_attn<4>(c, P, L, pos); break;
            }
            if (!grid_sync(c, P, ++nbar)) return;
            EpiStore ey{};
            ey.y = P.y;
            consume_gemv<QT_Q4K, false>(c, P.geo[SG_ATTN_OUT], ProPlainG{P.attn}, ey);
        }
        if (!grid_sync(c, P, ++nbar)) return;
        EpiSwiGlu sw{};
        sw.act = P.act;
        consume_gemv<QT_Q4K, true>(c, P.geo[SG_FFN_UP], step_norm(B, P.y, L.post_norm, nullptr, A, P), sw);
        if (!grid_sync(c, P, ++nbar)) return;
        EpiStore ey{};
        ey.y = P.y;
        consume_gemv<QT_Q6K, false>(c, P.geo[SG_FFN_DOWN], ProPlainG{P.act}, ey);
        if (!grid_sync(c, P, ++nbar)) return;
    }
    EpiArgmaxStep ea{};
    ea.ws = P.am_ws;
    ea.slots = P.slots;
    ea.hist = P.hist;
    ea.err = P.err;
    ea.allow = P.allow;
    ea.advance = P.advance;
    consume_gemv<QT_Q6K, false>(c, P.geo[SG_LMHEAD], step_norm(A, P.y, P.out_norm, nullptr, P.h, P), ea);
    // the last CTA out re-arms the barrier words for the next step
    bar_sync(1, kConsumers);
    if (c.tid == 0) {
        __threadfence();
        if (atomicAdd(P.gbar + 1, 1u) == gridDim.x - 1) {
            atomicExch(P.gbar, 0u);
            atomicExch(P.gbar + 1, 0u);
        }
    }
}

__global__ void __launch_bounds__(kThreads, 2) step_kernel(const __grid_constant__ StepParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int flag;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kMaxStages;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (__ldcg(P.gbar + 2)) return;  // an earlier step aborted: the host resets the words
    const int pos = __ldcg(P.slots + 1);
    if (tid == 0) {
        for (int s = 0; s < P.nslots; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();
    Pipe R{full, empty, smem + P.ring_off, P.nslots, kSlotBytes, 0u, P.err, P.gbar + 2, lane, 0ull};
    if (warp == kConsumerWarps) {
        R.pol = policy_evict_first();
        producer_main(R, P, pos);
        return;
    }
    Consumer c{R, smem, tid, warp, lane, &flag, true};
    consumer_main(c, P, pos);
}

// ================================================================== host
static_assert(stage_bytes_of(QT_Q6K) <= kSlotBytes && stage_bytes_of(QT_Q4K) <= kSlotBytes,
              "a GEMV stage must fit one ring slot");

static int make_geo(GemvShape* g, int qt, bool dual, int n, int k, int pro_floats, int grid, int* scratch) {
    if (!gemv_k_served(k)) return set_err(QG_ERR_SHAPE, "step kernel: k=%d", k);
    int used = 0;
    *g = gemv_geometry(qt, dual, nullptr, nullptr, n, k, pro_floats, grid, nullptr, &used, 1);  // stage = one slot
    // every CTA of the step runs every phase: rows split over the whole grid
    g->rows_cta = 8 * ((g->units + grid - 1) / grid);
    const int need = off_ring(qt, k, pro_floats, (dual ? 2 : 1) * g->rows_cta);
    *scratch = std::max(*scratch, need);
    return QG_OK;
}

int step_setup(const qg_model* m, qg_state* s) {
    const qg_config& c = m->cfg;
    StepParams& P = *s->step;
    std::memset(&P, 0, sizeof P);
    if (c.n_layers > kStepMaxLayers) return set_err(QG_ERR_SHAPE, "step kernel: %d layers (at most %d)", c.n_layers, kStepMaxLayers);
    const int gs = c.n_kv_heads > 0 ? c.n_heads / c.n_kv_heads : 1;
    bool has_attn = false, has_dn = false;
    for (int il = 0; il < c.n_layers; ++il) (m->kinds[il] == QG_LAYER_DELTANET ? has_dn : has_attn) = true;
    if (has_attn && gs != 1 && gs != 2 && gs != 4)
        return set_err(QG_ERR_SHAPE, "step kernel: %d query heads per kv head (served: 1, 2, 4)", gs);
    int dev = 0, sms = 0, coop = 0;
    QG_CUDA(cudaGetDevice(&dev));
    QG_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    QG_CUDA(cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev));
    if (!coop) return set_err(QG_ERR_CUDA, "step kernel: the device has no cooperative launch");

    // scratch = the largest phase's needs, then as many ring slots as fit
    int scratch = off_dig() + 4 * (2 * kDk);  // delta: q and k of one head
    if (has_attn)
        scratch = std::max(scratch, off_dig() + 4 * (gs * kHd + kHd + kHd + 8 * gs * 2 + 8 * gs * kHd + 64 * gs * 2));
    const int H = c.hidden;
    int grid = 2 * sms;
    for (int pass = 0; pass < 2; ++pass) {
        int sc = scratch, rc = QG_OK;
        ProRmsNorm pn{};
        if (has_dn) {
            const qg_layer_dev* L = nullptr;
            for (const auto& l : m->layers) if (l.kind == QG_LAYER_DELTANET) { L = &l; break; }
            if ((rc = make_geo(&P.geo[SG_DN_IN], QT_Q4K, false, L->n_in, H, pn.floats(H), grid, &sc)) ||
                (rc = make_geo(&P.geo[SG_SSM_OUT], QT_Q4K, false, H, m->v_dim, ProGatedNorm{}.floats(m->v_dim), grid, &sc)))
                return rc;
        }
        if (has_attn) {
            const qg_layer_dev* L = nullptr;
            for (const auto& l : m->layers) if (l.kind == QG_LAYER_ATTENTION) { L = &l; break; }
            if ((rc = make_geo(&P.geo[SG_ATTN_IN], QT_Q4K, false, L->n_in, H, pn.floats(H), grid, &sc)) ||
                (rc = make_geo(&P.geo[SG_ATTN_OUT], QT_Q4K, false, H, m->q_dim, ProPlainG{}.floats(0), grid, &sc)))
                return rc;
        }
        if ((rc = make_geo(&P.geo[SG_FFN_UP], QT_Q4K, true, c.ffn, H, pn.floats(H), grid, &sc)) ||
            (rc = make_geo(&P.geo[SG_FFN_DOWN], QT_Q6K, false, H, c.ffn, ProPlainG{}.floats(0), grid, &sc)) ||
            (rc = make_geo(&P.geo[SG_LMHEAD], QT_Q6K, false, c.vocab, H, pn.floats(H), grid, &sc)))
            return rc;
        P.ring_off = (sc + 127) & ~127;
        const int per_cta = kStepSmemPerCta;
        P.nslots = std::min(kStepMaxSlots, (per_cta - P.ring_off) / kSlotBytes);
        if (P.nslots < 2) return set_err(QG_ERR_SHAPE, "step kernel: %d bytes of phase scratch leave no ring", sc);
        s->step_smem = P.ring_off + P.nslots * kSlotBytes;
        if ((rc = grant_smem(reinterpret_cast<const void*>(step_kernel), kStepSmemPerCta))) return rc;
        int per_sm = 0;
        QG_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, step_kernel, kThreads, s->step_smem));
        if (per_sm < 1) return set_err(QG_ERR_SHAPE, "step kernel: no CTA fits an SM");
        const int g2 = std::min(per_sm, 2) * sms;
        if (g2 == grid) break;
        grid = g2;  // fewer CTAs per SM: redo the row split
    }
    s->step_grid = grid;

    P.n_layers = c.n_layers;
    P.hidden = H;
    P.ffn = c.ffn;
    P.vocab = c.vocab;
    P.conv_dim = m->conv_dim;
    P.conv_k = c.conv_kernel;
    P.nv = c.n_v_heads;
    P.nk = c.n_k_heads;
    P.dv = c.head_v_dim;
    P.k_dim = m->k_dim;
    P.v_dim = m->v_dim;
    P.q_dim = m->q_dim;
    P.kv_dim = m->kv_dim;
    P.gs = gs;
    P.n_kv = c.n_kv_heads;
    P.n_rot = c.n_rot;
    P.T = s->keys_per_split;
    P.max_splits = s->max_splits;
    P.eps = c.eps;
    P.theta_scale = m->theta_scale;
    P.embd = m->embd;
    P.out_norm = m->out_norm;
    P.lm_head = m->lm_head;
    for (int il = 0; il < c.n_layers; ++il) {
        const qg_layer_dev& D = m->layers[il];
        StepLayer& L = P.L[il];
        L.kind = D.kind;
        L.w_in = D.w_in;
        L.w_out = D.w_out;
        L.w_gate = D.w_gate;
        L.w_up = D.w_up;
        L.w_down = D.w_down;
        L.attn_norm = D.attn_norm;
        L.post_norm = D.post_norm;
        L.conv_w = D.conv_w;
        L.a = D.a;
        L.dt_bias = D.dt_bias;
        L.ssm_norm = D.ssm_norm;
        L.q_norm = D.q_norm;
        L.k_norm = D.k_norm;
        L.conv = s->conv[il];
        L.ssm = s->ssm[il];
        L.kc = s->kc[il];
        L.vc = s->vc[il];
    }
    P.h = s->h;
    P.hres = s->hres;
    P.y = s->y;
    P.conv_out = s->conv_out;
    P.dt = s->dt;
    P.beta = s->beta;
    P.z = s->z;
    P.o = s->o;
    P.act = s->act;
    P.qf = s->qf;
    P.kraw = s->kraw;
    P.attn = s->attn;
    P.part_acc = s->part_acc;
    P.part_ml = s->part_ml;
    P.attn_count = s->attn_count;
    P.am_ws = s->am_ws;
    P.slots = s->slots;
    P.hist = s->hist;
    P.allow = s->allow;
    P.err = s->err;
    P.gbar = s->gbar;
    return QG_OK;
}

int run_step(qg_state* s, cudaStream_t st, bool advance) {
    StepParams& P = *s->step;
    P.advance = advance ? 1 : 0;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(s->step_grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(s->step_smem);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    QG_CUDA(cudaLaunchKernelEx(&cfg, step_kernel, P));
    return QG_OK;
}

}  // namespace qg
