"""Token mask on the GPU (the decode session's grammar mask: banned logits
become -FLT_MAX before the fused first-index argmax), through the C ABI,
against the oracle's masked argmax of its own logits on the same seeded
model and inputs.

Bars: token ids exact wherever the masked top-2 margin of the oracle's logits
is decisive; graph and eager replays identical; setting,
changing and clearing the mask between steps needs no recapture.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
qg = pytest.importorskip("quantized_gemv_gated_gb300")


@pytest.fixture(scope="module")
def tiny():
    cfg = synth.CFG_TINY
    w = synth.make_model_weights(cfg)
    return cfg, w, qg.Model(w), oracle.Model(w)


def _allow(n, ids):
    w = np.zeros((n + 31) // 32, np.uint32)
    for i in ids:
        w[i >> 5] |= np.uint32(1) << np.uint32(i & 31)
    return w


def _masked(logits, words):
    x = logits.astype(np.float64).copy()
    i = np.arange(x.size)
    ok = (words[i >> 5] >> (i & 31).astype(np.uint32)) & np.uint32(1)
    x[ok == 0] = -np.finfo(np.float32).max
    return x


def _check(got, logits, words, want):
    """Exact when the masked top-2 margin is decisive, else one of the tied ids."""
    x = logits.astype(np.float64) if words is None else _masked(logits, words)
    top = np.sort(x)[::-1]
    tol = 1e-3 * max(1.0, float(np.max(np.abs(logits))))
    if top[0] - top[1] > tol:
        assert got == want
        return True
    assert x[got] >= top[0] - tol
    return False


def test_masked_tokens_match_oracle_graph_and_eager(tiny):
    cfg, w, m, om = tiny
    V = cfg.vocab
    sg, se = qg.State(m, cfg.max_seq_len), qg.State(m, cfg.max_seq_len)
    ost = oracle.State(om)
    rng = np.random.default_rng(synth.subseed(synth.MASTER_SEED, "token-mask"))
    toks = synth.prompt_tokens(cfg, 32)
    exact = 0
    for pos, t in enumerate(toks):
        ref, _, logits = oracle.forward_token(om, ost, int(t), pos, want_logits=True)
        kind = pos % 4
        if kind == 0:
            words = None  # no mask (cleared)
        elif kind == 1:
            words = _allow(V, np.flatnonzero(rng.random(V) < 0.3))
        elif kind == 2:
            words = _allow(V, [i for i in range(V) if i != ref])  # the unmasked choice banned
        else:
            words = _allow(V, [int(rng.integers(V))])  # one id allowed
        want = ref if words is None else oracle.argmax_masked(logits, words)
        for s in (sg, se):
            s.set_token_mask(words)
        a = qg.qg_decode_token(m, sg, int(t), pos)
        b = qg.qg_decode_token_eager(m, se, int(t), pos)
        assert a == b, f"pos {pos}: graph {a} != eager {b}"
        if words is not None:
            assert (words[a >> 5] >> np.uint32(a & 31)) & 1, f"pos {pos}: banned id {a} chosen"
        exact += _check(a, logits, words, want)
        assert np.array_equal(sg.download_hidden(), se.download_hidden())
    assert exact >= len(toks) - 2
    st = sg.stats()
    assert st["graph_captures"] == 1 and st["graph_launches"] == len(toks)


def test_masked_greedy_device_loop(tiny):
    """qg_decode_greedy under a fixed mask set after an unmasked prompt: the
    loop starts from the prompt's last (unmasked) choice and then feeds back
    its own masked choices; the oracle does the same with argmax_masked."""
    cfg, w, m, om = tiny
    V = cfg.vocab
    st = qg.State(m, cfg.max_seq_len)
    ost = oracle.State(om)
    toks = synth.prompt_tokens(cfg, 8)
    last = None
    for pos, t in enumerate(toks):
        got_last = qg.qg_decode_token(m, st, int(t), pos)
        last, _, _ = oracle.forward_token(om, ost, int(t), pos)
        assert got_last == last
    rng = np.random.default_rng(synth.subseed(synth.MASTER_SEED, "token-mask-greedy"))
    words = _allow(V, np.flatnonzero(rng.random(V) < 0.1))
    st.set_token_mask(words)
    n = 16
    got = qg.qg_decode_greedy(m, st, len(toks), n).tolist()
    expect = []
    for i in range(n):
        _, _, lg = oracle.forward_token(om, ost, last, len(toks) + i, want_logits=True)
        last = oracle.argmax_masked(lg, words)
        expect.append(last)
    assert got == expect
    assert all((words[g >> 5] >> np.uint32(g & 31)) & 1 for g in got)


def test_mask_arguments_and_reset(tiny):
    cfg, w, m, om = tiny
    V, nw = cfg.vocab, (cfg.vocab + 31) // 32
    st = qg.State(m, cfg.max_seq_len)
    with pytest.raises(qg.QgError) as e:
        st.set_token_mask(np.zeros(nw - 1, np.uint32))
    assert e.value.code == qg.QG_ERR_SHAPE
    with pytest.raises(qg.QgError) as e:
        qg._check(qg.lib().qg_state_set_token_mask(st.handle, None, nw))
    assert e.value.code == qg.QG_ERR_ARG
    toks = synth.prompt_tokens(cfg, 4)
    free = [qg.qg_decode_token(m, st, int(t), p) for p, t in enumerate(toks)]
    st.reset()
    st.set_token_mask(_allow(V, [V - 1]))
    assert qg.qg_decode_token(m, st, int(toks[0]), 0) == V - 1
    st.reset()  # reset clears the mask
    assert [qg.qg_decode_token(m, st, int(t), p) for p, t in enumerate(toks)] == free
    st.set_token_mask(_allow(V, []))  # every id banned: all -FLT_MAX, the first index
    assert qg.qg_decode_token(m, st, int(toks[0]), 4) == 0
    st.set_token_mask(None)
