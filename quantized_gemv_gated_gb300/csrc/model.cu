// C ABI: model and state lifecycle, teacher-forcing I/O, the per-layer
// building blocks and the whole-token step replayed as one CUDA graph
// (forward_qwen35_cuda.rs forward_single / forward_single_greedy; memra
// decode.rs GraphSession: device token and position slots, 4-byte readback).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>

#include "qg_internal.cuh"

using namespace qg;

namespace {


template <class T>
int dalloc(std::vector<void*>& list, T** p, size_t count, uint64_t* counter = nullptr) {
    void* v = nullptr;
    const size_t bytes = count * sizeof(T) > 0 ? count * sizeof(T) : 16;
    cudaError_t e = cudaMalloc(&v, bytes);
    if (e != cudaSuccess) return cuda_err(e, "cudaMalloc");
    list.push_back(v);
    if (counter) ++*counter;
    *p = static_cast<T*>(v);
    return QG_OK;
}

int upload(void* dst, const void* src, size_t bytes) {
    QG_CUDA(cudaMemcpy(dst, src, bytes, cudaMemcpyHostToDevice));
    return QG_OK;
}

size_t qbytes(const qg_qtensor& t) {
    const size_t nb = static_cast<size_t>(t.k) / 256;
    return static_cast<size_t>(t.n) * nb * (t.qtype == QG_QTYPE_Q4_K ? 144 : 210);
}

int check_q(const qg_qtensor& t, int qtype, int n, int k, const char* name) {
    if (!t.data) return set_err(QG_ERR_EMPTY, "%s: tensor data is NULL", name);
    if (t.qtype != qtype)
        return set_err(QG_ERR_QTYPE, "%s: GGML type %d has no kernel here (expected %d)", name, t.qtype, qtype);
    if (t.n != n || t.k != k) return set_err(QG_ERR_SHAPE, "%s: %d x %d, expected %d x %d", name, t.n, t.k, n, k);
    return QG_OK;
}

int upload_f32(qg_model* m, float** dst, const float* src, size_t n, const char* name) {
    if (!src) return set_err(QG_ERR_EMPTY, "%s: f32 vector is NULL", name);
    int rc = dalloc(m->allocs, dst, n);
    if (rc) return rc;
    return upload(*dst, src, n * sizeof(float));
}

// Concatenate Q4_K tensors with the same k row-wise and store them in the
// grouped layout of the GEMV engine (8-row groups, rows padded to 8).
int upload_fused(qg_model* m, uint8_t** dst, const qg_qtensor* const* parts, int count, int* rows) {
    size_t total = 0;
    int n = 0;
    const int k = parts[0]->k;
    for (int i = 0; i < count; ++i) {
        total += qbytes(*parts[i]);
        n += parts[i]->n;
    }
    const size_t grouped = static_cast<size_t>((n + 7) & ~7) * (k / 256) * 144;
    int rc = dalloc(m->allocs, dst, grouped);
    if (rc) return rc;
    uint8_t* tmp = nullptr;
    QG_CUDA(cudaMalloc(&tmp, total));
    size_t off = 0;
    for (int i = 0; i < count && !rc; ++i) {
        rc = upload(tmp + off, parts[i]->data, qbytes(*parts[i]));
        off += qbytes(*parts[i]);
    }
    if (!rc) rc = q4k_to_grouped(tmp, *dst, n, k, nullptr);
    cudaError_t e = cudaDeviceSynchronize();
    cudaFree(tmp);
    if (!rc && e != cudaSuccess) rc = cuda_err(e, "q4k repack");
    *rows = n;
    return rc;
}

int upload_q6k(qg_model* m, uint8_t** dst, const qg_qtensor& t) {
    const size_t pb = qg_q6k_planar_bytes(t.n, t.k);
    int rc = dalloc(m->allocs, dst, pb);
    if (rc) return rc;
    uint8_t* tmp = nullptr;
    QG_CUDA(cudaMalloc(&tmp, qbytes(t)));
    rc = upload(tmp, t.data, qbytes(t));
    if (!rc) rc = qg_q6k_to_planar(tmp, *dst, t.n, t.k, nullptr);
    cudaError_t e = cudaDeviceSynchronize();
    cudaFree(tmp);
    if (!rc && e != cudaSuccess) rc = cuda_err(e, "q6k repack");
    return rc;
}

int check_config(const qg_config* c) {
    if (!c->layer_kinds) return set_err(QG_ERR_ARG, "config: layer_kinds is NULL");
    if (c->n_layers < 1 || c->hidden < 1 || c->ffn < 1 || c->vocab < 1)
        return set_err(QG_ERR_EMPTY, "config: empty model");
    if (c->hidden % 256 || c->ffn % 256) return set_err(QG_ERR_SHAPE, "config: hidden and ffn must be multiples of 256");
    if (c->hidden > 16384 || c->ffn > 16384 || c->n_heads * c->head_dim > 16384 ||
        c->n_v_heads * c->head_v_dim > 16384)
        return set_err(QG_ERR_SHAPE, "config: a GEMV input is longer than 16384 (the engine's limit)");
    bool has_dn = false, has_attn = false;
    for (int i = 0; i < c->n_layers; ++i) {
        if (c->layer_kinds[i] == QG_LAYER_DELTANET) has_dn = true;
        else if (c->layer_kinds[i] == QG_LAYER_ATTENTION) has_attn = true;
        else return set_err(QG_ERR_LAYER_KIND, "config: layer %d has kind %d", i, c->layer_kinds[i]);
    }
    if (has_dn) {
        if (c->n_k_heads < 1 || c->n_v_heads % c->n_k_heads)
            return set_err(QG_ERR_SHAPE,
                           "config: the delta rule maps value head h onto key head h %% n_k_heads, so n_v_heads "
                           "(%d) must be a positive multiple of n_k_heads (%d)",
                           c->n_v_heads, c->n_k_heads);
        if (c->head_k_dim != 128) return set_err(QG_ERR_SHAPE, "config: head_k_dim %d (served: 128)", c->head_k_dim);
        if ((c->n_v_heads * c->head_v_dim) % 256)
            return set_err(QG_ERR_SHAPE, "config: n_v_heads*head_v_dim must be a multiple of 256");
        if (c->conv_kernel < 2 || c->conv_kernel > 8)
            return set_err(QG_ERR_SHAPE, "config: conv_kernel %d (served: 2..8)", c->conv_kernel);
        // the delta kernel takes 32 value rows per item; the ssm_out prologue
        // needs whole heads inside each 256-element super-block
        if (c->head_v_dim != 32 && c->head_v_dim != 64 && c->head_v_dim != 128)
            return set_err(QG_ERR_SHAPE, "config: head_v_dim %d (served: 32, 64, 128)", c->head_v_dim);
        if (c->n_v_heads > 64) return set_err(QG_ERR_SHAPE, "config: %d value heads (served: up to 64)", c->n_v_heads);
    }
    if (has_attn) {
        if (c->head_dim != 256) return set_err(QG_ERR_SHAPE, "config: head_dim %d (served: 256)", c->head_dim);
        if (c->n_kv_heads < 1 || c->n_heads % c->n_kv_heads)
            return set_err(QG_ERR_SHAPE, "config: n_heads %d is not a multiple of n_kv_heads %d", c->n_heads,
                           c->n_kv_heads);
        const int gs = c->n_heads / c->n_kv_heads;
        if (gs != 1 && gs != 2 && gs != 4 && gs != 8)
            return set_err(QG_ERR_SHAPE, "config: %d query heads per kv head (served: 1, 2, 4, 8)", gs);
        if (c->n_rot < 2 || c->n_rot % 2 || c->n_rot > c->head_dim)
            return set_err(QG_ERR_SHAPE, "config: n_rot %d", c->n_rot);
    }
    return QG_OK;
}

void free_all(std::vector<void*>& v) {
    for (void* p : v) cudaFree(p);
    v.clear();
}

// Whole token on stream st: layers, tail.  mode 0: graph step (slots filled
// by a host copy), 1: greedy (token and position already on the device).
int enqueue_token(qg_model* m, qg_state* s, cudaStream_t st, bool advance) {
    for (int il = 0; il < m->cfg.n_layers; ++il) {
        const bool first = il == 0;
        const ResidualIO io{s->hres, s->h, !first, first};
        int rc = m->kinds[il] == QG_LAYER_DELTANET ? run_deltanet_layer(m, s, il, io, st, !first)
                                                     : run_attention_layer(m, s, il, io, st, !first);
        if (rc) return rc;
    }
    return run_lmhead(m, s, s->hres, s->h, st, advance);
}

int count_kernel_nodes(cudaGraph_t g, uint64_t* out) {
    size_t n = 0;
    QG_CUDA(cudaGraphGetNodes(g, nullptr, &n));
    std::vector<cudaGraphNode_t> nodes(n);
    QG_CUDA(cudaGraphGetNodes(g, nodes.data(), &n));
    uint64_t k = 0;
    for (size_t i = 0; i < n; ++i) {
        cudaGraphNodeType t;
        QG_CUDA(cudaGraphNodeGetType(nodes[i], &t));
        if (t == cudaGraphNodeTypeKernel) ++k;
    }
    *out = k;
    return QG_OK;
}

// Capture the step graph (greedy == false: H2D of (token, pos), token, D2H
// of the output word) or the greedy graph (no host copies).
int capture(qg_model* m, qg_state* s, bool greedy, cudaGraphExec_t* exec) {
    cudaStream_t st = s->stream;
    cudaGraph_t g = nullptr;
    QG_CUDA(cudaStreamBeginCapture(st, cudaStreamCaptureModeRelaxed));
    int rc = QG_OK;
    if (!greedy) {
        cudaError_t e = cudaMemcpyAsync(s->slots, s->pinned, 2 * sizeof(int), cudaMemcpyHostToDevice, st);
        if (e != cudaSuccess) rc = cuda_err(e, "capture H2D");
    }
    if (!rc) rc = enqueue_token(m, s, st, greedy);
    if (!rc && !greedy) {
        cudaError_t e = cudaMemcpyAsync(s->pinned + 2, s->slots + 2, sizeof(int), cudaMemcpyDeviceToHost, st);
        if (e != cudaSuccess) rc = cuda_err(e, "capture D2H");
    }
    cudaError_t ee = cudaStreamEndCapture(st, &g);
    if (rc) {
        if (g) cudaGraphDestroy(g);
        return rc;
    }
    if (ee != cudaSuccess) return cuda_err(ee, "cudaStreamEndCapture");
    uint64_t nodes = 0;
    rc = count_kernel_nodes(g, &nodes);
    if (!rc) {
        cudaError_t e = cudaGraphInstantiate(exec, g, 0);
        if (e != cudaSuccess) rc = cuda_err(e, "cudaGraphInstantiate");
    }
    cudaGraphDestroy(g);
    if (!rc) {
        s->stats.graph_captures++;
        if (!greedy) s->stats.graph_kernel_nodes = nodes;
    }
    return rc;
}

int finish_step(qg_state* s, int pos, uint32_t* next_token) {
    const unsigned out = static_cast<unsigned>(s->pinned[2]);
    if (out & 0x80000000u) {
        unsigned e = 0;
        cudaMemcpy(&e, s->err, sizeof e, cudaMemcpyDeviceToHost);
        return set_err(QG_ERR_TIMEOUT, "a kernel of the step gave up on a bounded wait (flags 0x%x)", e);
    }
    *next_token = out;
    if (s->kv_len < pos + 1) s->kv_len = pos + 1;
    s->stats.steps++;
    return QG_OK;
}

int check_step(const qg_model* m, const qg_state* s, uint32_t token, int pos, const void* out) {
    if (!m || !s || !out) return set_err(QG_ERR_ARG, "decode: NULL argument");
    if (s->m != m) return set_err(QG_ERR_ARG, "decode: state belongs to another model");
    if (token >= static_cast<uint32_t>(m->cfg.vocab))
        return set_err(QG_ERR_TOKEN, "token %u is outside the %d-row embedding table", token, m->cfg.vocab);
    if (pos < 0 || pos >= s->max_seq)
        return set_err(QG_ERR_POS, "position %d is past the KV cache (%d rows)", pos, s->max_seq);
    return QG_OK;
}

}  // namespace

extern "C" {

int qg_model_create(const qg_config* cfg, const qg_host_weights* w, int device, qg_model** out) {
    if (!cfg || !w || !out) return set_err(QG_ERR_ARG, "model_create: NULL argument");
    *out = nullptr;
    int rc = check_config(cfg);
    if (rc) return rc;
    if (!w->layers || !w->token_embd || !w->output_norm)
        return set_err(QG_ERR_EMPTY, "model_create: missing embedding, output norm or layers");
    DeviceGuard dg(device);
    qg_model* m = new (std::nothrow) qg_model();
    if (!m) return set_err(QG_ERR_OOM, "model_create: host allocation");
    m->cfg = *cfg;
    m->kinds.assign(cfg->layer_kinds, cfg->layer_kinds + cfg->n_layers);
    m->cfg.layer_kinds = m->kinds.data();
    m->device = device;
    const qg_config& c = m->cfg;
    m->k_dim = c.n_k_heads * c.head_k_dim;
    m->v_dim = c.n_v_heads * c.head_v_dim;
    m->conv_dim = 2 * m->k_dim + m->v_dim;
    m->q_dim = c.n_heads * c.head_dim;
    m->kv_dim = c.n_kv_heads * c.head_dim;
    // theta_scale on the host in f32, as forward_qwen35_cuda.rs dims_of does
    m->theta_scale = powf(c.rope_theta, -2.0f / static_cast<float>(c.n_rot > 0 ? c.n_rot : 2));
    m->layers.resize(c.n_layers);
    const int H = c.hidden, F = c.ffn;
    for (int il = 0; il < c.n_layers && !rc; ++il) {
        const qg_layer_weights& L = w->layers[il];
        qg_layer_dev& D = m->layers[il];
        std::memset(&D, 0, sizeof D);
        D.kind = m->kinds[il];
        if (L.kind != D.kind) {
            rc = set_err(QG_ERR_LAYER_KIND, "layer %d: weights of kind %d, config says %d", il, L.kind, D.kind);
            break;
        }
        if ((rc = check_q(L.ffn_gate, QG_QTYPE_Q4_K, F, H, "ffn_gate")) || (rc = check_q(L.ffn_up, QG_QTYPE_Q4_K, F, H, "ffn_up")) ||
            (rc = check_q(L.ffn_down, QG_QTYPE_Q6_K, H, F, "ffn_down")))
            break;
        if ((rc = upload_f32(m, &D.attn_norm, L.attn_norm, H, "attn_norm")) ||
            (rc = upload_f32(m, &D.post_norm, L.post_attention_norm, H, "post_attention_norm")))
            break;
        int nr = 0;
        const qg_qtensor* g1[1] = {&L.ffn_gate};
        const qg_qtensor* u1[1] = {&L.ffn_up};
        if ((rc = upload_fused(m, &D.w_gate, g1, 1, &nr)) || (rc = upload_fused(m, &D.w_up, u1, 1, &nr)) ||
            (rc = upload_q6k(m, &D.w_down, L.ffn_down)))
            break;
        if (D.kind == QG_LAYER_DELTANET) {
            const int nv = c.n_v_heads;
            if ((rc = check_q(L.attn_qkv, QG_QTYPE_Q4_K, m->conv_dim, H, "attn_qkv")) ||
                (rc = check_q(L.ssm_alpha, QG_QTYPE_Q4_K, nv, H, "ssm_alpha")) ||
                (rc = check_q(L.ssm_beta, QG_QTYPE_Q4_K, nv, H, "ssm_beta")) ||
                (rc = check_q(L.attn_gate, QG_QTYPE_Q4_K, m->v_dim, H, "attn_gate")) ||
                (rc = check_q(L.ssm_out, QG_QTYPE_Q4_K, H, m->v_dim, "ssm_out")))
                break;
            const qg_qtensor* in[4] = {&L.attn_qkv, &L.ssm_alpha, &L.ssm_beta, &L.attn_gate};
            const qg_qtensor* o1[1] = {&L.ssm_out};
            if ((rc = upload_fused(m, &D.w_in, in, 4, &D.n_in)) || (rc = upload_fused(m, &D.w_out, o1, 1, &nr)) ||
                (rc = upload_f32(m, &D.conv_w, L.ssm_conv1d, static_cast<size_t>(m->conv_dim) * c.conv_kernel,
                                 "ssm_conv1d")) ||
                (rc = upload_f32(m, &D.dt_bias, L.ssm_dt_bias, nv, "ssm_dt_bias")) ||
                (rc = upload_f32(m, &D.ssm_norm, L.ssm_norm, c.head_v_dim, "ssm_norm")))
                break;
            float* alog = nullptr;
            if ((rc = upload_f32(m, &alog, L.ssm_a_log, nv, "ssm_a_log")) || (rc = dalloc(m->allocs, &D.a, nv)) ||
                (rc = run_neg_exp(alog, D.a, nv, nullptr)))
                break;
        } else {
            if ((rc = check_q(L.attn_q, QG_QTYPE_Q4_K, 2 * m->q_dim, H, "attn_q")) ||
                (rc = check_q(L.attn_k, QG_QTYPE_Q4_K, m->kv_dim, H, "attn_k")) ||
                (rc = check_q(L.attn_v, QG_QTYPE_Q4_K, m->kv_dim, H, "attn_v")) ||
                (rc = check_q(L.attn_output, QG_QTYPE_Q4_K, H, m->q_dim, "attn_output")))
                break;
            const qg_qtensor* in[3] = {&L.attn_q, &L.attn_k, &L.attn_v};
            const qg_qtensor* o1[1] = {&L.attn_output};
            if ((rc = upload_fused(m, &D.w_in, in, 3, &D.n_in)) || (rc = upload_fused(m, &D.w_out, o1, 1, &nr)) ||
                (rc = upload_f32(m, &D.q_norm, L.attn_q_norm, c.head_dim, "attn_q_norm")) ||
                (rc = upload_f32(m, &D.k_norm, L.attn_k_norm, c.head_dim, "attn_k_norm")))
                break;
        }
    }
    if (!rc) {
        if ((rc = check_q(w->lm_head, QG_QTYPE_Q6_K, c.vocab, H, "lm_head")) == QG_OK) {
            if (!(rc = upload_f32(m, &m->embd, w->token_embd, static_cast<size_t>(c.vocab) * H, "token_embd")) &&
                !(rc = upload_f32(m, &m->out_norm, w->output_norm, H, "output_norm")))
                rc = upload_q6k(m, &m->lm_head, w->lm_head);
        }
    }
    if (!rc) {
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess) rc = cuda_err(e, "model_create");
    }
    if (rc) {
        free_all(m->allocs);
        delete m;
        return rc;
    }
    *out = m;
    return QG_OK;
}

int qg_model_destroy(qg_model* m) {
    if (!m) return QG_OK;
    DeviceGuard dg(m->device);
    cudaDeviceSynchronize();
    free_all(m->allocs);
    delete m;
    return QG_OK;
}

int qg_state_create(const qg_model* m, int max_seq_len, qg_state** out) {
    return qg_state_create_kv(m, max_seq_len, QG_KV_F32, out);
}

int qg_state_create_kv(const qg_model* m, int max_seq_len, int kv_format, qg_state** out) {
    if (kv_format != QG_KV_F32 && kv_format != QG_KV_Q8_0_Q5_1)
        return set_err(QG_ERR_ARG, "state_create: unknown KV cache format %d", kv_format);
    if (!m || !out) return set_err(QG_ERR_ARG, "state_create: NULL argument");
    *out = nullptr;
    if (max_seq_len < 1) return set_err(QG_ERR_SHAPE, "state_create: max_seq_len must be at least 1");
    DeviceGuard dg(m->device);
    qg_state* s = new (std::nothrow) qg_state();
    if (!s) return set_err(QG_ERR_OOM, "state_create: host allocation");
    s->m = m;
    s->max_seq = max_seq_len;
    s->kv_format = kv_format;
    s->kv_len = 0;
    s->exec_step = nullptr;
    s->exec_greedy = nullptr;
    s->pf = nullptr;
    std::memset(&s->stats, 0, sizeof s->stats);
    const qg_config& c = m->cfg;
    uint64_t* cnt = &s->stats.device_allocs;
    int rc = QG_OK;
    s->conv.assign(c.n_layers, nullptr);
    s->ssm.assign(c.n_layers, nullptr);
    s->kc.assign(c.n_layers, nullptr);
    s->vc.assign(c.n_layers, nullptr);
    // keys per split: at most 32 splits (the combine reads every split), at
    // least 32 keys, a multiple of 8; fixed per state, so the key partition
    // of a step depends on its position only
    int T = (max_seq_len + 31) / 32;
    T = ((T + 7) / 8) * 8;
    if (T < 32) T = 32;
    s->keys_per_split = T;
    s->max_splits = (max_seq_len + T - 1) / T;
    const int gs = c.n_kv_heads > 0 ? c.n_heads / c.n_kv_heads : 1;
    for (int il = 0; il < c.n_layers && !rc; ++il) {
        if (m->kinds[il] == QG_LAYER_DELTANET) {
            if ((rc = dalloc(s->allocs, &s->conv[il], static_cast<size_t>(m->conv_dim) * (c.conv_kernel - 1), cnt)))
                break;
            rc = dalloc(s->allocs, &s->ssm[il], static_cast<size_t>(c.n_v_heads) * c.head_v_dim * c.head_k_dim, cnt);
        } else {
            // f32 rows, or (quantized cache) records of bytes, allocated as whole floats
            if ((rc = dalloc(s->allocs, &s->kc[il], kv_cache_bytes(s, 0) / sizeof(float), cnt))) break;
            rc = dalloc(s->allocs, &s->vc[il], kv_cache_bytes(s, 1) / sizeof(float), cnt);
        }
    }
    if (!rc) {
        const size_t H = c.hidden;
        (void)((rc = dalloc(s->allocs, &s->h, H, cnt)) || (rc = dalloc(s->allocs, &s->hres, H, cnt)) ||
               (rc = dalloc(s->allocs, &s->y, H, cnt)) || (rc = dalloc(s->allocs, &s->conv_out, m->conv_dim, cnt)) ||
               (rc = dalloc(s->allocs, &s->dt, c.n_v_heads + 1, cnt)) ||
               (rc = dalloc(s->allocs, &s->beta, c.n_v_heads + 1, cnt)) ||
               (rc = dalloc(s->allocs, &s->z, m->v_dim + 1, cnt)) || (rc = dalloc(s->allocs, &s->o, m->v_dim + 1, cnt)) ||
               (rc = dalloc(s->allocs, &s->act, c.ffn, cnt)) || (rc = dalloc(s->allocs, &s->qf, 2 * m->q_dim + 1, cnt)) ||
               (rc = dalloc(s->allocs, &s->kraw, m->kv_dim + 1, cnt)) ||
               (rc = dalloc(s->allocs, &s->vraw, m->kv_dim + 1, cnt)) ||
               (rc = dalloc(s->allocs, &s->attn, m->q_dim + 1, cnt)) ||
               (rc = dalloc(s->allocs, &s->part_acc,
                            static_cast<size_t>(c.n_kv_heads) * s->max_splits * gs * 256 + 1, cnt)) ||
               (rc = dalloc(s->allocs, &s->part_ml, static_cast<size_t>(c.n_kv_heads) * s->max_splits * gs * 2 + 1,
                            cnt)) ||
               (rc = dalloc(s->allocs, &s->attn_count, c.n_kv_heads + 1, cnt)) ||
               (rc = dalloc(s->allocs, &s->am_ws, 2, cnt)) || (rc = dalloc(s->allocs, &s->slots, 4, cnt)) ||
               (rc = dalloc(s->allocs, &s->hist, max_seq_len, cnt)) || (rc = dalloc(s->allocs, &s->err, 1, cnt)) ||
               (rc = dalloc(s->allocs, &s->allow, (static_cast<size_t>(c.vocab) + 31) / 32, cnt)) ||
               (rc = dalloc(s->allocs, &s->kpart,
                            static_cast<size_t>(std::max({gemv_slices(c.ffn), gemv_slices(m->v_dim > 0 ? m->v_dim : 256),
                                                          gemv_slices(m->q_dim > 0 ? m->q_dim : 256)})) *
                                ((H + 7) & ~size_t(7)),
                            cnt)) ||
               (rc = (s->ycur = s->y, s->ycur_parts = 1, s->ycur_stride = 0, QG_OK)));
    }
    if (!rc) rc = encode_kv_maps(s);
    if (!rc) {
        void* p = nullptr;
        cudaError_t e = cudaHostAlloc(&p, 4 * sizeof(int), cudaHostAllocDefault);
        if (e != cudaSuccess) rc = cuda_err(e, "cudaHostAlloc");
        else {
            s->pinned = static_cast<int*>(p);
            std::memset(s->pinned, 0, 4 * sizeof(int));
            ++*cnt;
        }
    }
    if (!rc) {
        cudaError_t e = cudaStreamCreateWithFlags(&s->stream, cudaStreamNonBlocking);
        if (e != cudaSuccess) rc = cuda_err(e, "cudaStreamCreate");
    }
    if (!rc) {
        s->kv_len = 0;
        rc = qg_state_reset(s);
    }
    if (rc) {
        if (s->pinned) cudaFreeHost(s->pinned);
        free_all(s->allocs);
        delete s;
        return rc;
    }
    *out = s;
    return QG_OK;
}

int qg_state_destroy(qg_state* s) {
    if (!s) return QG_OK;
    DeviceGuard dg(s->m->device);
    if (s->stream) cudaStreamSynchronize(s->stream);
    if (s->exec_step) cudaGraphExecDestroy(s->exec_step);
    if (s->exec_greedy) cudaGraphExecDestroy(s->exec_greedy);
    if (s->stream) cudaStreamDestroy(s->stream);
    if (s->pinned) cudaFreeHost(s->pinned);
    prefill_release(s);
    free_all(s->allocs);
    delete s;
    return QG_OK;
}

int qg_state_reset(qg_state* s) {
    if (!s) return set_err(QG_ERR_ARG, "state_reset: NULL state");
    DeviceGuard dg(s->m->device);
    QG_CUDA(cudaStreamSynchronize(s->stream));
    // every buffer starts at zero (windows, states, caches, counters, slots)
    const qg_model* m = s->m;
    const qg_config& c = m->cfg;
    for (int il = 0; il < c.n_layers; ++il) {
        if (s->conv[il]) QG_CUDA(cudaMemset(s->conv[il], 0, sizeof(float) * m->conv_dim * (c.conv_kernel - 1)));
        if (s->ssm[il])
            QG_CUDA(cudaMemset(s->ssm[il], 0, sizeof(float) * static_cast<size_t>(c.n_v_heads) * c.head_v_dim * c.head_k_dim));
        if (s->kc[il]) QG_CUDA(cudaMemset(s->kc[il], 0, kv_cache_bytes(s, 0)));
        if (s->vc[il]) QG_CUDA(cudaMemset(s->vc[il], 0, kv_cache_bytes(s, 1)));
    }
    QG_CUDA(cudaMemset(s->h, 0, sizeof(float) * c.hidden));
    QG_CUDA(cudaMemset(s->hres, 0, sizeof(float) * c.hidden));
    QG_CUDA(cudaMemset(s->y, 0, sizeof(float) * c.hidden));
    QG_CUDA(cudaMemset(s->attn_count, 0, sizeof(unsigned) * (c.n_kv_heads + 1)));
    QG_CUDA(cudaMemset(s->am_ws, 0, 2 * sizeof(unsigned long long)));
    QG_CUDA(cudaMemset(s->slots, 0, 4 * sizeof(int)));
    QG_CUDA(cudaMemset(s->err, 0, sizeof(unsigned)));
    QG_CUDA(cudaMemset(s->allow, 0xff, sizeof(uint32_t) * ((static_cast<size_t>(c.vocab) + 31) / 32)));  // no mask
    QG_CUDA(cudaDeviceSynchronize());
    s->kv_len = 0;
    return QG_OK;
}

int qg_state_upload_layer(qg_state* s, int il, const float* conv, const float* ssm) {
    if (!s || !conv || !ssm) return set_err(QG_ERR_ARG, "upload_layer: NULL argument");
    const qg_model* m = s->m;
    if (il < 0 || il >= m->cfg.n_layers) return set_err(QG_ERR_LAYER_KIND, "upload_layer: layer %d is out of range", il);
    if (m->kinds[il] != QG_LAYER_DELTANET)
        return set_err(QG_ERR_LAYER_KIND, "upload_layer: layer %d is a full-attention layer, not a Gated DeltaNet one", il);
    DeviceGuard dg(m->device);
    const qg_config& c = m->cfg;
    QG_CUDA(cudaStreamSynchronize(s->stream));
    QG_CUDA(cudaMemcpy(s->conv[il], conv, sizeof(float) * m->conv_dim * (c.conv_kernel - 1), cudaMemcpyHostToDevice));
    QG_CUDA(cudaMemcpy(s->ssm[il], ssm, sizeof(float) * static_cast<size_t>(c.n_v_heads) * c.head_v_dim * c.head_k_dim,
                       cudaMemcpyHostToDevice));
    return QG_OK;
}

int qg_state_upload_kv(qg_state* s, int il, const float* k, const float* v, int rows) {
    if (!s) return set_err(QG_ERR_ARG, "upload_kv: NULL state");
    const qg_model* m = s->m;
    if (il < 0 || il >= m->cfg.n_layers) return set_err(QG_ERR_LAYER_KIND, "upload_kv: layer %d is out of range", il);
    if (m->kinds[il] != QG_LAYER_ATTENTION)
        return set_err(QG_ERR_LAYER_KIND, "upload_kv: layer %d is a Gated DeltaNet layer, not a full-attention one", il);
    if (rows < 0 || rows > s->max_seq)
        return set_err(QG_ERR_SHAPE, "upload_kv: %d rows, the cache holds at most %d", rows, s->max_seq);
    if (rows > 0 && (!k || !v)) return set_err(QG_ERR_ARG, "upload_kv: NULL rows");
    DeviceGuard dg(m->device);
    QG_CUDA(cudaStreamSynchronize(s->stream));
    const size_t bytes = sizeof(float) * static_cast<size_t>(rows) * m->kv_dim;
    if (rows > 0 && s->kv_format == QG_KV_Q8_0_Q5_1) {
        // quantized cache: the f32 rows go through the append's quantizer on the device
        float* tmp = nullptr;
        QG_CUDA(cudaMalloc(&tmp, 2 * bytes));
        int rc = QG_OK;
        cudaError_t e = cudaMemcpy(tmp, k, bytes, cudaMemcpyHostToDevice);
        if (e == cudaSuccess) e = cudaMemcpy(tmp + bytes / sizeof(float), v, bytes, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) rc = cuda_err(e, "upload_kv: cudaMemcpy");
        if (!rc)
            rc = kv_quantize_rows(tmp, tmp + bytes / sizeof(float), rows, m->cfg.n_kv_heads, s->max_seq,
                                  reinterpret_cast<uint8_t*>(s->kc[il]), reinterpret_cast<uint8_t*>(s->vc[il]),
                                  s->stream);
        if (!rc && (e = cudaStreamSynchronize(s->stream)) != cudaSuccess) rc = cuda_err(e, "upload_kv: quantize");
        cudaFree(tmp);
        if (rc) return rc;
    } else if (rows > 0) {
        QG_CUDA(cudaMemcpy(s->kc[il], k, bytes, cudaMemcpyHostToDevice));
        QG_CUDA(cudaMemcpy(s->vc[il], v, bytes, cudaMemcpyHostToDevice));
    }
    s->kv_len = rows;
    return QG_OK;
}

int qg_state_download_kv_records(qg_state* s, int il, void* k, void* v, size_t* k_bytes, size_t* v_bytes) {
    if (!s || !k_bytes || !v_bytes) return set_err(QG_ERR_ARG, "download_kv_records: NULL argument");
    const qg_model* m = s->m;
    if (il < 0 || il >= m->cfg.n_layers || m->kinds[il] != QG_LAYER_ATTENTION)
        return set_err(QG_ERR_LAYER_KIND, "download_kv_records: layer %d is not a full-attention layer", il);
    if (s->kv_format != QG_KV_Q8_0_Q5_1)
        return set_err(QG_ERR_ARG, "download_kv_records: the state's KV cache is f32 (use qg_state_download_layer)");
    DeviceGuard dg(m->device);
    QG_CUDA(cudaStreamSynchronize(s->stream));
    QG_CUDA(cudaDeviceSynchronize());
    const int nkv = m->cfg.n_kv_heads;
    const size_t kr = kv_cache_bytes(s, 0) / (static_cast<size_t>(nkv) * s->max_seq);
    const size_t vr = kv_cache_bytes(s, 1) / (static_cast<size_t>(nkv) * s->max_seq);
    *k_bytes = static_cast<size_t>(nkv) * s->kv_len * kr;
    *v_bytes = static_cast<size_t>(nkv) * s->kv_len * vr;
    if (s->kv_len == 0) return QG_OK;
    const uint8_t* kc = reinterpret_cast<const uint8_t*>(s->kc[il]);
    const uint8_t* vc = reinterpret_cast<const uint8_t*>(s->vc[il]);
    for (int g = 0; g < nkv; ++g) {  // head g's first kv_len records, packed
        const size_t at = static_cast<size_t>(g) * s->max_seq, to = static_cast<size_t>(g) * s->kv_len;
        if (k) QG_CUDA(cudaMemcpy(static_cast<uint8_t*>(k) + to * kr, kc + at * kr, s->kv_len * kr, cudaMemcpyDeviceToHost));
        if (v) QG_CUDA(cudaMemcpy(static_cast<uint8_t*>(v) + to * vr, vc + at * vr, s->kv_len * vr, cudaMemcpyDeviceToHost));
    }
    return QG_OK;
}

int qg_state_kv_format(const qg_state* s, int* kv_format) {
    if (!s || !kv_format) return set_err(QG_ERR_ARG, "state_kv_format: NULL argument");
    *kv_format = s->kv_format;
    return QG_OK;
}

int qg_state_download_layer(qg_state* s, int il, float* a, float* b, size_t* n) {
    if (!s || !n) return set_err(QG_ERR_ARG, "download_layer: NULL argument");
    const qg_model* m = s->m;
    if (il < 0 || il >= m->cfg.n_layers) return set_err(QG_ERR_LAYER_KIND, "download_layer: layer %d is out of range", il);
    DeviceGuard dg(m->device);
    const qg_config& c = m->cfg;
    QG_CUDA(cudaStreamSynchronize(s->stream));
    QG_CUDA(cudaDeviceSynchronize());
    if (m->kinds[il] == QG_LAYER_DELTANET) {
        const size_t cl = static_cast<size_t>(m->conv_dim) * (c.conv_kernel - 1);
        const size_t sl = static_cast<size_t>(c.n_v_heads) * c.head_v_dim * c.head_k_dim;
        *n = sl > cl ? sl : cl;
        if (a) QG_CUDA(cudaMemcpy(a, s->conv[il], cl * sizeof(float), cudaMemcpyDeviceToHost));
        if (b) QG_CUDA(cudaMemcpy(b, s->ssm[il], sl * sizeof(float), cudaMemcpyDeviceToHost));
        return QG_OK;
    }
    if (s->kv_format != QG_KV_F32)
        return set_err(QG_ERR_ARG, "download_layer: layer %d holds a quantized cache (use qg_state_download_kv_records)", il);
    const size_t cnt = static_cast<size_t>(s->kv_len) * m->kv_dim;
    *n = cnt;
    if (cnt && a) QG_CUDA(cudaMemcpy(a, s->kc[il], cnt * sizeof(float), cudaMemcpyDeviceToHost));
    if (cnt && b) QG_CUDA(cudaMemcpy(b, s->vc[il], cnt * sizeof(float), cudaMemcpyDeviceToHost));
    return QG_OK;
}

int qg_state_download_hidden(qg_state* s, float* hidden_host) {
    if (!s || !hidden_host) return set_err(QG_ERR_ARG, "download_hidden: NULL argument");
    DeviceGuard dg(s->m->device);
    QG_CUDA(cudaStreamSynchronize(s->stream));
    QG_CUDA(cudaMemcpy(hidden_host, s->h, sizeof(float) * s->m->cfg.hidden, cudaMemcpyDeviceToHost));
    return QG_OK;
}

int qg_state_kv_len(const qg_state* s, int* kv_len) {
    if (!s || !kv_len) return set_err(QG_ERR_ARG, "kv_len: NULL argument");
    *kv_len = s->kv_len;
    return QG_OK;
}

int qg_state_set_token_mask(qg_state* s, const uint32_t* allow, int n_words) {
    if (!s) return set_err(QG_ERR_ARG, "set_token_mask: NULL state");
    const int words = (s->m->cfg.vocab + 31) / 32;
    if (n_words != 0 && n_words != words)
        return set_err(QG_ERR_SHAPE, "set_token_mask: %d words (the vocabulary needs %d, or 0 to clear)", n_words,
                       words);
    if (n_words && !allow) return set_err(QG_ERR_ARG, "set_token_mask: NULL mask");
    DeviceGuard dg(s->m->device);
    // in stream order with the steps, and done before returning: the caller may free `allow`
    if (n_words)
        QG_CUDA(cudaMemcpyAsync(s->allow, allow, sizeof(uint32_t) * words, cudaMemcpyHostToDevice, s->stream));
    else
        QG_CUDA(cudaMemsetAsync(s->allow, 0xff, sizeof(uint32_t) * words, s->stream));
    QG_CUDA(cudaStreamSynchronize(s->stream));
    return QG_OK;
}

int qg_state_stream(const qg_state* s, qg_stream* out) {
    if (!s || !out) return set_err(QG_ERR_ARG, "state_stream: NULL argument");
    *out = reinterpret_cast<qg_stream>(s->stream);
    return QG_OK;
}

int qg_state_stats(const qg_state* s, qg_stats* out) {
    if (!s || !out) return set_err(QG_ERR_ARG, "stats: NULL argument");
    *out = s->stats;
    return QG_OK;
}

int qg_deltanet_step(const qg_model* m, qg_state* s, int il, float* hidden_dev, qg_stream stream) {
    if (!m || !s || !hidden_dev) return set_err(QG_ERR_ARG, "deltanet_step: NULL argument");
    if (il < 0 || il >= m->cfg.n_layers) return set_err(QG_ERR_LAYER_KIND, "deltanet_step: layer %d is out of range", il);
    if (m->kinds[il] != QG_LAYER_DELTANET)
        return set_err(QG_ERR_LAYER_KIND, "deltanet_step: layer %d is a full-attention layer", il);
    if (reinterpret_cast<uintptr_t>(hidden_dev) & 15u) return set_err(QG_ERR_ARG, "deltanet_step: hidden not 16-byte aligned");
    DeviceGuard dg(m->device);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const ResidualIO io{hidden_dev, s->h, false, false};
    int rc = run_deltanet_layer(m, s, il, io, st, true);
    if (rc) return rc;
    return run_residual(s, hidden_dev, m->cfg.hidden, st);
}

int qg_attn_decode_step(const qg_model* m, qg_state* s, int il, float* hidden_dev, int pos, qg_stream stream) {
    if (!m || !s || !hidden_dev) return set_err(QG_ERR_ARG, "attn_decode_step: NULL argument");
    if (il < 0 || il >= m->cfg.n_layers) return set_err(QG_ERR_LAYER_KIND, "attn_decode_step: layer %d is out of range", il);
    if (m->kinds[il] != QG_LAYER_ATTENTION)
        return set_err(QG_ERR_LAYER_KIND, "attn_decode_step: layer %d is a Gated DeltaNet layer", il);
    if (pos < 0 || pos >= s->max_seq)
        return set_err(QG_ERR_POS, "position %d is past the KV cache (%d rows)", pos, s->max_seq);
    if (reinterpret_cast<uintptr_t>(hidden_dev) & 15u) return set_err(QG_ERR_ARG, "attn_decode_step: hidden not 16-byte aligned");
    DeviceGuard dg(m->device);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int p = pos;  // pageable source: the copy is staged before the call returns
    QG_CUDA(cudaMemcpyAsync(s->slots + 1, &p, sizeof(int), cudaMemcpyHostToDevice, st));
    const ResidualIO io{hidden_dev, s->h, false, false};
    int rc = run_attention_layer(m, s, il, io, st, false);
    if (!rc) rc = run_residual(s, hidden_dev, m->cfg.hidden, st);
    if (rc) return rc;
    if (s->kv_len < pos + 1) s->kv_len = pos + 1;
    return QG_OK;
}

int qg_bench_kernel(const qg_model* m, qg_state* s, int kind, int launches, qg_stream stream) {
    if (!m || !s) return set_err(QG_ERR_ARG, "bench_kernel: NULL argument");
    if (s->m != m) return set_err(QG_ERR_ARG, "bench_kernel: the state belongs to another model");
    if (launches < 1) return set_err(QG_ERR_ARG, "bench_kernel: %d launches", launches);
    DeviceGuard dg(m->device);
    return run_kernel_kind(m, s, kind, launches, reinterpret_cast<cudaStream_t>(stream));
}

int qg_decode_token(qg_model* m, qg_state* s, uint32_t token, int pos, uint32_t* next_token) {
    int rc = check_step(m, s, token, pos, next_token);
    if (rc) return rc;
    DeviceGuard dg(m->device);
    if (!s->exec_step && (rc = capture(m, s, false, &s->exec_step))) return rc;
    s->pinned[0] = static_cast<int>(token);
    s->pinned[1] = pos;
    QG_CUDA(cudaGraphLaunch(s->exec_step, s->stream));
    QG_CUDA(cudaStreamSynchronize(s->stream));
    s->stats.graph_launches++;
    s->stats.h2d_bytes += 2 * sizeof(int);
    s->stats.d2h_bytes += sizeof(int);
    return finish_step(s, pos, next_token);
}

int qg_decode_token_eager(qg_model* m, qg_state* s, uint32_t token, int pos, uint32_t* next_token) {
    int rc = check_step(m, s, token, pos, next_token);
    if (rc) return rc;
    DeviceGuard dg(m->device);
    s->pinned[0] = static_cast<int>(token);
    s->pinned[1] = pos;
    QG_CUDA(cudaMemcpyAsync(s->slots, s->pinned, 2 * sizeof(int), cudaMemcpyHostToDevice, s->stream));
    if ((rc = enqueue_token(m, s, s->stream, false))) return rc;
    QG_CUDA(cudaMemcpyAsync(s->pinned + 2, s->slots + 2, sizeof(int), cudaMemcpyDeviceToHost, s->stream));
    QG_CUDA(cudaStreamSynchronize(s->stream));
    s->stats.h2d_bytes += 2 * sizeof(int);
    s->stats.d2h_bytes += sizeof(int);
    return finish_step(s, pos, next_token);
}

int qg_decode_greedy(qg_model* m, qg_state* s, int pos0, int n_steps, uint32_t* tokens_host) {
    if (!m || !s || !tokens_host) return set_err(QG_ERR_ARG, "decode_greedy: NULL argument");
    if (n_steps < 0) return set_err(QG_ERR_ARG, "decode_greedy: n_steps %d", n_steps);
    if (pos0 < 0 || pos0 + n_steps > s->max_seq)
        return set_err(QG_ERR_POS, "positions %d..%d are past the KV cache (%d rows)", pos0, pos0 + n_steps - 1,
                       s->max_seq);
    if (n_steps == 0) return QG_OK;
    DeviceGuard dg(m->device);
    int rc;
    if (!s->exec_greedy && (rc = capture(m, s, true, &s->exec_greedy))) return rc;
    s->pinned[1] = pos0;
    QG_CUDA(cudaMemcpyAsync(s->slots + 1, s->pinned + 1, sizeof(int), cudaMemcpyHostToDevice, s->stream));
    for (int i = 0; i < n_steps; ++i) QG_CUDA(cudaGraphLaunch(s->exec_greedy, s->stream));
    QG_CUDA(cudaMemcpyAsync(tokens_host, s->hist + pos0, sizeof(uint32_t) * n_steps, cudaMemcpyDeviceToHost, s->stream));
    QG_CUDA(cudaStreamSynchronize(s->stream));
    unsigned e = 0;
    QG_CUDA(cudaMemcpy(&e, s->err, sizeof e, cudaMemcpyDeviceToHost));
    if (e) return set_err(QG_ERR_TIMEOUT, "a kernel gave up on a bounded wait (flags 0x%x)", e);
    s->stats.graph_launches += n_steps;
    s->stats.h2d_bytes += sizeof(int);
    s->stats.d2h_bytes += sizeof(uint32_t) * n_steps;
    s->stats.steps += n_steps;
    if (s->kv_len < pos0 + n_steps) s->kv_len = pos0 + n_steps;
    return QG_OK;
}

}  // extern "C"
