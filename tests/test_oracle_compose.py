"""Pins of the oracle's layer compositions.

or_deltanet_layer, or_attention_layer and or_forward_token wire the pinned
primitives (norms, GEMV, conv, gates, delta rule, rope, attention, argmax)
together in the op order of forward_qwen35_cuda.rs (deltanet_layer_inner,
attention_layer_inner, forward_single).  Here each composition is restated in
numpy from those primitives, with non-zero output projections and distinct
norm weights, and must agree with the oracle bit for bit (the primitives run
the same code, in the same accumulation order).  Each restatement is also run
with one plausible wiring mistake planted -- a wrong norm weight, a wrong
input vector, swapped operands, a residual added in the wrong place -- and
must then disagree: the pins are sensitive to every one of them.
"""
import ctypes
import ctypes.util

import numpy as np
import pytest

import oracle
import synth

_libm = ctypes.CDLL(ctypes.util.find_library("m") or "libm.so.6")
_libm.expf.restype = ctypes.c_float
_libm.expf.argtypes = [ctypes.c_float]

# two layers (one of each kind), value heads over fewer key heads, a
# vocabulary that is not a multiple of any tile
CFG = synth.ModelConfig(name="compose", n_layers=2, hidden=512, ffn=768, vocab=1000, n_k_heads=2,
                        n_v_heads=4, n_heads=4, n_kv_heads=2, max_seq_len=16,
                        layer_kinds=(synth.DELTANET, synth.ATTENTION))


def neg_exp(a_log):
    """a = -exp(A_log) with the C library's expf (the arithmetic the oracle
    uses for this step; the wiring, not expf, is under test here)."""
    return np.array([-_libm.expf(float(v)) for v in a_log], np.float32)


def deltanet(cfg, L, conv, ssm, h, bug=None):
    """One Gated DeltaNet layer from the primitives: returns (h, conv, ssm)."""
    kd, nk, nv, dk, dv = cfg.k_dim, cfg.n_k_heads, cfg.n_v_heads, cfg.head_k_dim, cfg.head_v_dim
    xn = oracle.rmsnorm(h, L.attn_norm)
    qkv = oracle.gemv(L.attn_qkv, xn)
    c, conv = oracle.conv1d_silu(qkv, conv, L.ssm_conv1d)
    q = oracle.l2norm_heads(c[:kd], dk)
    k = oracle.l2norm_heads(c[kd:2 * kd], dk)
    v = c[2 * kd:]
    if bug == "swap_qk":
        q, k = k, q
    al = oracle.gemv(L.ssm_alpha, xn)
    br = oracle.gemv(L.ssm_beta, xn)
    dt, be = oracle.gates(al, L.ssm_dt_bias, neg_exp(L.ssm_a_log), br)
    z = oracle.gemv(L.attn_gate, h if bug == "gate_unnormed" else xn)
    o, ssm = oracle.delta_rule(q, k, v, be, dt, ssm, nk, dk, nv, dv)
    u = oracle.gated_rmsnorm(z, o, L.ssm_norm, dv) if bug == "swap_oz" else oracle.gated_rmsnorm(o, z, L.ssm_norm, dv)
    y = oracle.gemv(L.ssm_out, o if bug == "ssm_out_of_o" else u)
    h1 = h + y
    h2 = ffn(L, h1, bug)
    return h2, conv, ssm


def ffn(L, h1, bug=None):
    """Post-attention norm, SwiGLU FFN and its residual."""
    xn2 = oracle.rmsnorm(h1, L.attn_norm if bug == "ffn_attn_norm" else L.post_attention_norm)
    act = oracle.swiglu(oracle.gemv(L.ffn_gate, xn2), oracle.gemv(L.ffn_up, xn2))
    if bug == "swap_gate_up":
        act = oracle.swiglu(oracle.gemv(L.ffn_up, xn2), oracle.gemv(L.ffn_gate, xn2))
    y = oracle.gemv(L.ffn_down, act)
    return (xn2 if bug == "residual_after_norm" else h1) + y


def attention(cfg, L, kc, vc, h, pos, bug=None):
    """One full-attention layer from the primitives: returns (h, kc, vc)."""
    hd, nh, nkv = cfg.head_dim, cfg.n_heads, cfg.n_kv_heads
    ts = oracle.theta_scale(cfg.rope_theta, cfg.n_rot)
    kc, vc = kc.copy(), vc.copy()
    xn = oracle.rmsnorm(h, L.attn_norm)
    qf = oracle.gemv(L.attn_q, xn)
    kraw = oracle.gemv(L.attn_k, xn)
    vc[pos] = oracle.gemv(L.attn_v, xn)
    q, gate = oracle.split_q_gate(qf, nh, hd)
    if bug == "swap_q_gate":
        q, gate = gate, q
    qn = oracle.rmsnorm_heads(q, L.attn_q_norm, hd)
    krow = oracle.rmsnorm_heads(kraw, L.attn_q_norm if bug == "k_with_q_norm" else L.attn_k_norm, hd)
    qn = oracle.rope_neox(qn, hd, cfg.n_rot, pos, ts)
    kc[pos] = krow if bug == "k_no_rope" else oracle.rope_neox(krow, hd, cfg.n_rot, pos, ts)
    att = oracle.attention(qn, kc, vc, nh, nkv, hd, pos if bug == "skip_new_row" else pos + 1)
    att = oracle.sigmoid_gate(att, gate)
    y = oracle.gemv(L.attn_output, att)
    h1 = h + y
    return ffn(L, h1, bug), kc, vc


def _weights(dmax):
    return synth.make_model_weights(CFG, dmax=dmax)


def _state(m, w, seed):
    st = oracle.State(m)
    conv0, ssm0 = synth.initial_deltanet_state(CFG, 0)
    st.conv[0][:] = conv0
    st.ssm[0][:] = ssm0
    # earlier cache rows of the attention layer
    r = np.random.default_rng(seed)
    rows = 5
    st.set_kv_rows(1, r.standard_normal((rows, CFG.kv_dim)).astype(np.float32),
                   r.standard_normal((rows, CFG.kv_dim)).astype(np.float32))
    st.kv_len = rows
    return st


DN_BUGS = ["ffn_attn_norm", "gate_unnormed", "ssm_out_of_o", "swap_oz", "residual_after_norm", "swap_qk",
           "swap_gate_up"]
ATT_BUGS = ["ffn_attn_norm", "residual_after_norm", "swap_q_gate", "k_with_q_norm", "k_no_rope", "skip_new_row",
            "swap_gate_up"]


@pytest.mark.parametrize("dmax", [5e-5, 2e-3])
def test_deltanet_layer_is_its_composition(dmax):
    w = _weights(dmax)
    L = w.layers[0]
    assert not np.array_equal(L.attn_norm, L.post_attention_norm)
    m = oracle.Model(w)
    st = _state(m, w, 1)
    h = np.random.default_rng(2).standard_normal(CFG.hidden).astype(np.float32)
    conv0, ssm0 = st.conv[0].copy(), st.ssm[0].copy()
    want_h, want_conv, want_ssm = deltanet(CFG, L, conv0, ssm0, h)
    got = oracle.deltanet_layer(m, st, 0, h)
    assert np.array_equal(got, want_h)
    assert np.array_equal(st.conv[0], want_conv)
    assert np.array_equal(st.ssm[0], want_ssm)
    assert not np.array_equal(got, h)  # the layer is not a pass-through
    for bug in DN_BUGS:
        bad_h, _, bad_ssm = deltanet(CFG, L, conv0, ssm0, h, bug)
        assert not (np.array_equal(bad_h, got) and np.array_equal(bad_ssm, want_ssm)), bug


@pytest.mark.parametrize("dmax", [5e-5, 2e-3])
def test_attention_layer_is_its_composition(dmax):
    w = _weights(dmax)
    L = w.layers[1]
    m = oracle.Model(w)
    st = _state(m, w, 3)
    pos = 5
    h = np.random.default_rng(4).standard_normal(CFG.hidden).astype(np.float32)
    kc0, vc0 = st.kc[1].copy(), st.vc[1].copy()
    want_h, want_kc, want_vc = attention(CFG, L, kc0, vc0, h, pos)
    got = oracle.attention_layer(m, st, 1, h, pos)
    assert np.array_equal(got, want_h)
    assert np.array_equal(st.kc[1], want_kc)
    assert np.array_equal(st.vc[1], want_vc)
    assert st.kv_len == pos + 1
    for bug in ATT_BUGS:
        bad_h, bad_kc, _ = attention(CFG, L, kc0, vc0, h, pos, bug)
        assert not (np.array_equal(bad_h, got) and np.array_equal(bad_kc, want_kc)), bug


def test_forward_token_is_its_composition():
    w = _weights(5e-5)
    m = oracle.Model(w)
    st = _state(m, w, 5)
    conv0, ssm0, kc0, vc0 = st.conv[0].copy(), st.ssm[0].copy(), st.kc[1].copy(), st.vc[1].copy()
    token, pos = 617, 5
    tok, hidden, logits = oracle.forward_token(m, st, token, pos, want_logits=True)
    h = w.token_embd[token].copy()
    h, _, _ = deltanet(CFG, w.layers[0], conv0, ssm0, h)
    h, _, _ = attention(CFG, w.layers[1], kc0, vc0, h, pos)
    assert np.array_equal(hidden, h)
    want_logits = oracle.gemv(w.lm_head, oracle.rmsnorm(h, w.output_norm))
    assert np.array_equal(logits, want_logits)
    assert tok == oracle.argmax(want_logits)
    # the output norm's weight, not a layer's, scales the lm_head input
    wrong = oracle.gemv(w.lm_head, oracle.rmsnorm(h, w.layers[1].post_attention_norm))
    assert not np.array_equal(logits, wrong)
    # layers run in index order
    h2 = w.token_embd[token].copy()
    h2, _, _ = attention(CFG, w.layers[1], kc0, vc0, h2, pos)
    h2, _, _ = deltanet(CFG, w.layers[0], conv0, ssm0, h2)
    assert not np.array_equal(hidden, h2)


def test_two_steps_carry_the_state():
    """The second token's layer reads the conv window, recurrent state and
    cache rows the first token left."""
    w = _weights(5e-5)
    m = oracle.Model(w)
    st = _state(m, w, 6)
    conv, ssm, kc, vc = st.conv[0].copy(), st.ssm[0].copy(), st.kc[1].copy(), st.vc[1].copy()
    for token, pos in ((11, 5), (909, 6)):
        _, hidden, _ = oracle.forward_token(m, st, token, pos, want_logits=False)
        h = w.token_embd[token].copy()
        h, conv, ssm = deltanet(CFG, w.layers[0], conv, ssm, h)
        h, kc, vc = attention(CFG, w.layers[1], kc, vc, h, pos)
        assert np.array_equal(hidden, h)
    assert np.array_equal(st.ssm[0], ssm) and np.array_equal(st.kc[1], kc)
