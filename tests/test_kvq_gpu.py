"""Quantized KV cache (q8_0 K / q5_1 V, quantize-on-append in the attention
kernel) on the GPU through the C ABI, against the oracle's quantized cache on
the same seeded inputs.

Bars:
- the quantizer, on identical f32 rows (qg_state_upload_kv), gives the
  oracle's blocks byte for byte, rearranged into the cache's records;
- after a decode step, every older record is untouched; in the new row each
  code equals the oracle's wherever the rounding decision is clear by more
  than the two sides' pre-quantization rows can differ (1e-5 of the row's
  max |value|, the bar of the f32 K/V rows), and is one of the two
  neighbouring codes elsewhere; scales are exact;
- the hidden state is within 1e-3 normwise plus, for each near-tie code
  taken the other way, a bound on what one code step of the new row can move
  it (computed from the weights and the oracle's values, see flip_bound);
- whole tokens, teacher-forced: after every step the oracle's cache rows are
  set to the GPU's records (tests/kvq_sync.py), so near-tie codes taken the
  other way do not accumulate; every code then differs by at most one step
  with identical scales, the hidden state stays within 1e-3 at every step,
  the tokens are the oracle's, and the graph and eager steps agree bitwise.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from kvq_sync import records, sync_rows

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
qg = pytest.importorskip("quantized_gemv_gated_gb300")

TOL = 1e-3
ROW_TOL = 1e-5  # the f32 K/V row bar of the attention layer tests


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def k_codes(K):  # [nkv][t][272] -> [t][nkv*256] int codes, [t][nkv*8] f16 bits
    nkv, t = K.shape[:2]
    q = K[..., 16:].view(np.int8).astype(np.int32).transpose(1, 0, 2).reshape(t, -1)
    d = K[..., :16].copy().view(np.uint16).transpose(1, 0, 2).reshape(t, -1)
    return q, d


def v_codes(V):  # [nkv][t][192] -> [t][nkv*256] codes 0..31, [t][nkv*16] f16 bits (d, m)
    nkv, t = V.shape[:2]
    dm = V[..., :32].copy().view(np.uint16).transpose(1, 0, 2).reshape(t, -1)
    qh = V[..., 32:64].copy().view(np.uint32)  # [nkv][t][8]
    qs = V[..., 64:].reshape(nkv, t, 8, 16).astype(np.int32)
    j = np.arange(32)
    nib = np.where(j < 16, qs[..., j % 16] & 15, qs[..., j % 16] >> 4)  # [nkv][t][8][32]
    hi = (qh[..., None] >> j.astype(np.uint32)) & 1
    q = (nib | (hi.astype(np.int32) << 4)).reshape(nkv, t, 256).transpose(1, 0, 2).reshape(t, -1)
    return q, dm


def _attn_cfg(base, max_seq):
    return dataclasses.replace(base, name=base.name + "-attn1", n_layers=1, vocab=512,
                               layer_kinds=(synth.ATTENTION,), max_seq_len=max_seq)


# ------------------------------------------------------------ the quantizer
@pytest.mark.parametrize("base,max_seq,rows", [(synth.CFG_TINY, 96, 96), (synth.CFG_4B, 512, 300)])
def test_upload_quantizer_matches_oracle_bytes(base, max_seq, rows):
    cfg = _attn_cfg(base, max_seq)
    w = synth.make_model_weights(cfg)
    m = qg.Model(w)
    k, v = synth.long_context_kv(cfg, 0, rows)
    k, v = k.copy(), v.copy()
    kvd = cfg.kv_dim
    # special rows: zeros, a constant, exact ties, a d below FLT_MIN, large values
    k[0], v[0] = 0.0, 0.0
    k[1], v[1] = 3.0, -2.0
    ties8 = np.tile(np.r_[127.0, np.arange(31) - 15 + 0.5], kvd // 32)  # max|x| = 127: d = 1, x.5 ties
    ties5 = np.tile(np.r_[0.0, 31.0, np.arange(30) + 0.5], kvd // 32)  # min 0, max 31: d = 1, x.5 ties
    k[2], v[2] = ties8, ties5
    k[3], v[3] = k[10] * 1e-37, v[10] * 1e-37
    k[4], v[4] = k[11] * 1e4, v[11] * 1e4
    st = qg.State(m, max_seq, qg.KV_Q8_0_Q5_1)
    st.upload_kv(0, k, v)
    K, V = st.download_kv_records(0)
    wantK, wantV = records(oracle.quantize_q8_0(k.reshape(-1)).reshape(rows, -1),
                           oracle.quantize_q5_1(v.reshape(-1)).reshape(rows, -1), cfg.n_kv_heads)
    assert K.shape == wantK.shape and V.shape == wantV.shape
    bk, bv = np.argwhere(K != wantK), np.argwhere(V != wantV)
    assert bk.size == 0, f"K records differ at {bk[:5].tolist()}"
    assert bv.size == 0, f"V records differ at {bv[:5].tolist()}"
    st.close()


# ------------------------------------------------------- decode-step parity
def flip_bound(w, cfg, qn, gate, vmax, e, is_v, d):
    """What one code step d of element e of the new K or V row can move the
    layer's output (before the FFN, whose input is that output normalised):
    V: each query head h of the group adds p_h * d * sigmoid(gate) along
    column (h, j) of W_o, p_h <= 1; K: head h's score moves by
    |q_h[j]| * d / sqrt(hd), which moves its softmax weights by at most that
    much in sum, hence its output by at most that times max |V| per dim."""
    hd = cfg.head_dim
    gs = cfg.n_heads // cfg.n_kv_heads
    g, j = divmod(int(e), hd)
    Wo = oracle.dequant(w.layers[0].attn_output).astype(np.float64)  # [hidden][q_dim]
    b = np.zeros(cfg.hidden)
    for h in range(g * gs, (g + 1) * gs):
        if is_v:
            b += np.abs(Wo[:, h * hd + j]) * d
        else:
            ds = abs(qn[h * hd + j]) * d / np.sqrt(hd)
            b += np.abs(Wo[:, h * hd:(h + 1) * hd]).sum(axis=1) * ds * vmax
    return float(b.max())


@pytest.mark.parametrize("base,max_seq,positions", [
    (synth.CFG_TINY, 96, [0, 1, 31, 32, 33, 63, 64, 95]),
    (synth.CFG_0P8B, 1024, [0, 849, 1023]),
    (synth.CFG_4B, 8192, [8000, 8191]),
])
def test_attention_layer_quantized_cache_positions(base, max_seq, positions):
    cfg = _attn_cfg(base, max_seq)
    w = synth.make_model_weights(cfg)
    m, om = qg.Model(w), oracle.Model(w)
    L = w.layers[0]
    nh, hd, nkv = cfg.n_heads, cfg.head_dim, cfg.n_kv_heads
    for pos in positions:
        st = qg.State(m, max_seq, qg.KV_Q8_0_Q5_1)
        sq, sf = oracle.State(om, oracle.KV_Q8_0_Q5_1), oracle.State(om)
        k = v = None
        if pos > 0:
            k, v = synth.long_context_kv(cfg, 0, pos)
            st.upload_kv(0, k, v)
            sq.set_kv_rows(0, k, v)
        x = synth.normal(synth.subseed(synth.MASTER_SEED, f"attn.x.{pos}"), cfg.hidden)
        h = dev(x)
        qg.qg_attn_decode_step(m, st, 0, h, pos)
        ref = oracle.attention_layer(om, sq, 0, x, pos)
        oracle.attention_layer(om, sf, 0, x, pos)  # its row pos: the K/V values before quantization
        K, V = st.download_kv_records(0)
        assert K.shape[1] == pos + 1 and st.kv_len == pos + 1
        wantK, wantV = records(sq.kq[0][:pos + 1], sq.vq[0][:pos + 1], nkv)
        if pos > 0:  # older records untouched
            assert np.array_equal(K[:, :pos], wantK[:, :pos]) and np.array_equal(V[:, :pos], wantV[:, :pos])
        qk, dk = k_codes(K[:, pos:pos + 1])
        wk, wdk = k_codes(wantK[:, pos:pos + 1])
        qv, dmv = v_codes(V[:, pos:pos + 1])
        wv, wdmv = v_codes(wantV[:, pos:pos + 1])
        assert np.array_equal(dk, wdk) and np.array_equal(dmv, wdmv), f"pos {pos}: block scales differ"
        krow, vrow = sf.kc[0][pos].astype(np.float64), sf.vc[0][pos].astype(np.float64)
        # near-tie slots: the rounded value is within the rows' agreement of a half-integer boundary
        flips = []
        for which, row, got, want, nbytes in ((0, krow, qk[0], wk[0], 34), (1, vrow, qv[0], wv[0], 24)):
            pre = oracle.kv_prescaled(row.astype(np.float32), which).astype(np.float64)
            blocks = (sq.kq if which == 0 else sq.vq)[0][pos].reshape(-1, nbytes)
            d = blocks[:, :2].copy().view(np.float16).astype(np.float64).reshape(-1)
            # |x - x'| <= dx moves x/d by dx/d and d itself (max|x|/127, range/31) by at most
            # dx/127 or 2dx/31: a decision moves by at most 2dx/d (q8_0) or 4dx/d (q5_1)
            dx = ROW_TOL * np.max(np.abs(row))
            slack = np.repeat(np.where(d > 0, (2 + 2 * which) * dx / np.maximum(d, 1e-300), np.inf), 32)
            tie = np.abs(pre - np.floor(pre) - 0.5) <= slack
            bad = (got != want) & ~tie
            assert not bad.any(), f"pos {pos}: {'KV'[which]} codes differ at decisive slots {np.flatnonzero(bad)[:8]}"
            assert np.all(np.abs(got - want) <= 1), f"pos {pos}: {'KV'[which]} codes differ by more than one step"
            for e in np.flatnonzero(got != want):
                flips.append((which, e, d[e // 32]))
        allow = TOL
        if flips:
            xn = oracle.rmsnorm(x, L.attn_norm, cfg.eps)
            q, gate = oracle.split_q_gate(oracle.gemv(L.attn_q, xn), nh, hd)
            qn = oracle.rope_neox(oracle.rmsnorm_heads(q, L.attn_q_norm, hd, cfg.eps), hd, cfg.n_rot, pos,
                                  oracle.theta_scale(cfg.rope_theta, cfg.n_rot))
            vmax = float(np.max(np.abs(sq.vc[0][:pos + 1])))
            extra = sum(flip_bound(w, cfg, qn, gate, vmax, e, which == 1, dd) for which, e, dd in flips)
            allow = TOL + extra / np.max(np.abs(ref))
        e = rel(h.cpu().numpy(), ref)
        assert e <= allow, f"pos {pos}: hidden {e:.3g} > {allow:.3g} ({len(flips)} near-tie codes taken the other way)"
        st.close()
    qg.qg_device_status()


# --------------------------------------------------------- whole-token path
def _prefill_both(cfg, states, ostates, rows):
    """Cache rows 0..rows-1 of every attention layer from the same f32 rows on
    both sides (the GPU's quantizer gives the oracle's bytes on identical
    rows), and the same DeltaNet windows and states."""
    for il, kind in enumerate(cfg.kinds()):
        if kind == synth.DELTANET:
            c, s = synth.initial_deltanet_state(cfg, il)
            for st in states:
                st.upload_layer(il, c, s)
            for ost in ostates:
                ost.conv[il][:] = c
                ost.ssm[il][:] = s
        else:
            k, v = synth.long_context_kv(cfg, il, rows)
            for st in states:
                st.upload_kv(il, k, v)
            for ost in ostates:
                ost.set_kv_rows(il, k, v)
    for ost in ostates:
        ost.kv_len = rows


def test_quantized_cache_teacher_forced_steps_and_graph_eager_identity():
    cfg = synth.CFG_0P8B
    w = synth.make_model_weights(cfg, dmax=5e-5)  # near unit-scale stream: the argmax follows the token
    m, om = qg.Model(w), oracle.Model(w)
    sg = qg.State(m, cfg.max_seq_len, qg.KV_Q8_0_Q5_1)
    se = qg.State(m, cfg.max_seq_len, qg.KV_Q8_0_Q5_1)
    ost = oracle.State(om, oracle.KV_Q8_0_Q5_1)
    pos0 = 16  # the new row is one of 17+: one code step of it moves the output by ~1e-5 (flip_bound)
    _prefill_both(cfg, [sg, se], [ost], pos0)
    attn = [il for il, k in enumerate(cfg.kinds()) if k == synth.ATTENTION]
    toks = synth.prompt_tokens(cfg, 24)
    worst, flips = 0.0, 0
    for i, t in enumerate(toks):
        pos = pos0 + i
        a = qg.qg_decode_token(m, sg, int(t), pos)
        b = qg.qg_decode_token_eager(m, se, int(t), pos)
        assert a == b and np.array_equal(sg.download_hidden(), se.download_hidden())
        want, hid, logits = oracle.forward_token(om, ost, int(t), pos, want_logits=True)
        e = rel(sg.download_hidden(), hid)
        worst = max(worst, e)
        assert e <= TOL, f"pos {pos}: hidden {e:.3g}"
        if a != want:
            v1, v2 = oracle.top2(logits)
            assert logits[a] >= v1 - 1e-3 * abs(v1), f"pos {pos}: token {a} != oracle {want} (margin {v1 - v2:.3g})"
        for il in attn:  # teacher forcing of the new row
            diff, step, scales = sync_rows(sg, ost, il, pos, pos + 1, cfg.n_kv_heads)
            assert scales <= 1 and step <= 1, f"pos {pos} layer {il}: a value moved {scales:.3g} steps or a code {step}"
            flips += diff
    print(f"24 teacher-forced steps: worst hidden rel err {worst:.3g}, {flips} near-tie codes synced")
    # the device-resident greedy loop: its own choices, the oracle's tokens
    n = 8
    got = qg.qg_decode_greedy(m, sg, pos0 + len(toks), n).tolist()
    tok, want = want, []
    for i in range(n):
        tok, _, _ = oracle.forward_token(om, ost, tok, pos0 + len(toks) + i)
        want.append(tok)
    assert got == want
    assert sg.kv_len == pos0 + len(toks) + n


def test_quantized_cache_arguments():
    cfg = synth.CFG_TINY
    w = synth.make_model_weights(cfg)
    m = qg.Model(w)
    with pytest.raises(qg.QgError) as e:
        qg.State(m, cfg.max_seq_len, 7)
    assert e.value.code == qg.QG_ERR_ARG
    st = qg.State(m, cfg.max_seq_len, qg.KV_Q8_0_Q5_1)
    fmt = qg.ctypes.c_int()
    qg._check(qg.lib().qg_state_kv_format(st.handle, qg.ctypes.byref(fmt)))
    assert fmt.value == qg.KV_Q8_0_Q5_1
    il = cfg.kinds().index(synth.ATTENTION)
    with pytest.raises(qg.QgError) as e:
        st.download_layer(il)
    assert e.value.code == qg.QG_ERR_ARG
    toks = synth.prompt_tokens(cfg, 4)
    for p, t in enumerate(toks):
        qg.qg_decode_token(m, st, int(t), p)
    K, V = st.download_kv_records(il)
    assert K.shape == (cfg.n_kv_heads, 4, 272) and V.shape == (cfg.n_kv_heads, 4, 192)
    st.reset()
    K, V = st.download_kv_records(il)
    assert K.size == 0 and V.size == 0
    f32 = qg.State(m, cfg.max_seq_len)
    with pytest.raises(qg.QgError) as e:
        f32.download_kv_records(il)
    assert e.value.code == qg.QG_ERR_ARG
