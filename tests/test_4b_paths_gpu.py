"""The batched prefill and the batched decode at the 4B shapes that bench.py
times, through the C ABI, against the oracle decoding token by token.

These shapes reach paths the smaller models do not: the input-projection and
gate/up GEMMs over K = 2560 (a 32-chunk and an 8-chunk slice), ffn_down over
K = 9216 (four 32-chunk slices and a 16-chunk one), the tensor-core prefill
GEMM with K splits on few row tiles (a 40-token prompt: one 128-token tile,
ffn_down and ssm_out split seven ways; 136 tokens: the 256-wide instructions
over a partly filled second tile; 8 tokens take the small-batch GEMV),
and the batched lm_head whose row sums add up over two K slices before the
per-sequence argmax.

Bars as in the prefill and batch tests: the token equals the oracle's (exact
where its top-2 margin is decisive), the residual stream within 1e-3
normwise, the recurrent states within 1e-3, the conv windows and K/V rows
within 1e-4 at layer 0 and within the hidden-state bar deeper in (they are
projections of the residual stream at their layer).  The weights take
dmax = 5e-5 (the varied workload) so that the tokens move and the margins are
of order 0.03-1 logit.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
qg = pytest.importorskip("quantized_gemv_gated_gb300")

TOL = 1e-3
CFG = synth.CFG_4B


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))


def _token_ok(got, want, logits):
    top = np.sort(logits.astype(np.float64))[::-1]
    tol = 1e-3 * max(1.0, float(np.max(np.abs(logits))))
    if top[0] - top[1] > tol:
        return got == want
    return logits[got] >= top[0] - tol


@pytest.fixture(scope="module")
def models():
    w = synth.make_model_weights(CFG, dmax=5e-5)
    return qg.Model(w), oracle.Model(w)


@pytest.mark.parametrize("n_prompt", [8, 40, 136])  # the small-batch GEMV; the tensor-core GEMM (N 128, N 256)
def test_prefill_4b_shapes(models, n_prompt):
    m, om = models
    toks = synth.prompt_tokens(CFG, n_prompt)
    st, ost = qg.State(m, CFG.max_seq_len), oracle.State(om)
    got = qg.qg_prefill(m, st, toks)
    want = hid = logits = None
    for p, t in enumerate(toks):
        want, hid, logits = oracle.forward_token(om, ost, int(t), p, want_logits=True)
    assert _token_ok(got, want, logits), f"token {got} vs oracle {want}"
    assert rel(st.download_hidden(), hid) <= TOL
    for il, kind in enumerate(CFG.kinds()):
        bar = 1e-4 if il == 0 else TOL  # as row_bar in the prefill tests
        if kind == synth.DELTANET:
            conv, ssm = st.download_layer(il)
            assert rel(conv, ost.conv[il]) <= bar, f"layer {il}: conv window"
            assert rel(ssm, ost.ssm[il]) <= 1e-3, f"layer {il}: recurrent state"
        else:
            k, v = st.download_layer(il)
            assert rel(k, ost.kc[il][: len(toks)]) <= bar and rel(v, ost.vc[il][: len(toks)]) <= bar, f"layer {il}"
    qg.qg_device_status()


def test_batch_4b_shapes(models):
    m, om = models
    n = 4
    states = [qg.State(m, CFG.max_seq_len) for _ in range(n)]
    ostates = [oracle.State(om) for _ in range(n)]
    toks, pos = [], []
    for i in range(n):  # one- or two-token prompts of their own
        prompt = synth.tokens(synth.subseed(synth.MASTER_SEED, f"batch4b.prompt.{i}"), CFG.vocab, 1 + (i & 1))
        qg.qg_prefill(m, states[i], prompt)
        t = None
        for p, tk in enumerate(prompt):
            t, _, _ = oracle.forward_token(om, ostates[i], int(tk), p)
        toks.append(int(t))
        pos.append(len(prompt))
    for step in range(2):
        got = qg.qg_decode_batch(m, states, toks, pos)
        for i in range(n):
            want, hid, lg = oracle.forward_token(om, ostates[i], toks[i], pos[i], want_logits=True)
            assert _token_ok(got[i], want, lg), f"step {step} seq {i}: {got[i]} vs oracle {want}"
            assert rel(states[i].download_hidden(), hid) <= TOL, f"step {step} seq {i}"
            toks[i], pos[i] = want, pos[i] + 1
    qg.qg_device_status()
