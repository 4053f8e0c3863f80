"""Batched lockstep decode (qg_decode_batch) on the GPU through the C ABI:
n sequences, each with its own state, prompt and position, against the oracle
decoding each sequence on its own.

Bars: every sequence's token equals its oracle token (exact where the top-2
margin is decisive); every sequence's residual stream within 1e-3 normwise;
the batched step of one sequence agrees with the single-sequence step.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from kvq_sync import sync_rows

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
qg = pytest.importorskip("quantized_gemv_gated_gb300")

TOL = 1e-3


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))


def _token_ok(got, want, logits):
    top = np.sort(logits.astype(np.float64))[::-1]
    tol = 1e-3 * max(1.0, float(np.max(np.abs(logits))))
    if top[0] - top[1] > tol:
        return got == want
    return logits[got] >= top[0] - tol


def _run(cfg, n, steps, kv_format=qg.KV_F32, dmax=0.02):
    w = synth.make_model_weights(cfg, dmax=dmax)
    m, om = qg.Model(w), oracle.Model(w)
    ofmt = oracle.KV_Q8_0_Q5_1 if kv_format == qg.KV_Q8_0_Q5_1 else oracle.KV_F32
    states = [qg.State(m, cfg.max_seq_len, kv_format) for _ in range(n)]
    ostates = [oracle.State(om, ofmt) for _ in range(n)]
    rng = np.random.default_rng(synth.subseed(synth.MASTER_SEED, f"batch.{cfg.name}.{n}"))
    toks, pos = [], []
    for i in range(n):  # prompts of different lengths, prefilled one sequence at a time
        plen = int(rng.integers(1, 12))
        prompt = synth.tokens(synth.subseed(synth.MASTER_SEED, f"batch.prompt.{i}"), cfg.vocab, plen)
        qg.qg_prefill(m, states[i], prompt)
        t = None
        for p, tk in enumerate(prompt):
            t, _, _ = oracle.forward_token(om, ostates[i], int(tk), p)
        toks.append(int(t))
        pos.append(plen)
    for step in range(steps):
        got = qg.qg_decode_batch(m, states, toks, pos)
        for i in range(n):
            want, hid, lg = oracle.forward_token(om, ostates[i], toks[i], pos[i], want_logits=True)
            assert _token_ok(got[i], want, lg), f"step {step} seq {i}: {got[i]} vs oracle {want}"
            e = rel(states[i].download_hidden(), hid)
            assert e <= TOL, f"step {step} seq {i}: hidden {e:.3g}"
            toks[i], pos[i] = want, pos[i] + 1
    for i in range(n):
        assert states[i].kv_len == pos[i]
    qg.qg_device_status()


@pytest.mark.parametrize("n", [1, 3, 4, 5, 6, 8, 9])
def test_batch_tiny(n):
    _run(dataclasses.replace(synth.CFG_TINY, max_seq_len=64), n, steps=5)


def test_batch_0p8b_shapes():
    _run(synth.CFG_0P8B, 4, steps=3, dmax=5e-5)


def test_batch_quantized_cache():
    """Two sequences in lockstep over quantized caches, teacher-forced per
    step: each new cache row on the oracle's side is set to the GPU's record
    (each side quantizes its own f32 row; near-tie codes may come out one
    step apart), so every step is held to the decode's 1e-3 bar."""
    cfg = dataclasses.replace(synth.CFG_TINY, max_seq_len=64)
    w = synth.make_model_weights(cfg)
    m, om = qg.Model(w), oracle.Model(w)
    states = [qg.State(m, cfg.max_seq_len, qg.KV_Q8_0_Q5_1) for _ in range(2)]
    ostates = [oracle.State(om, oracle.KV_Q8_0_Q5_1) for _ in range(2)]
    attn = [il for il, k in enumerate(cfg.kinds()) if k == synth.ATTENTION]
    toks, pos = [3, 7], [0, 0]
    for step in range(6):
        got = qg.qg_decode_batch(m, states, toks, pos)
        for i in range(2):
            want, hid, lg = oracle.forward_token(om, ostates[i], toks[i], pos[i], want_logits=True)
            assert _token_ok(got[i], want, lg)
            assert rel(states[i].download_hidden(), hid) <= TOL, f"step {step} seq {i}"
            for il in attn:
                _, dstep, scales = sync_rows(states[i], ostates[i], il, pos[i], pos[i] + 1, cfg.n_kv_heads)
                assert scales <= 1 and dstep <= 1  # one step of the block's scale at most
            toks[i], pos[i] = want, pos[i] + 1


def test_batch_of_one_matches_single_step():
    cfg = dataclasses.replace(synth.CFG_TINY, max_seq_len=64)
    w = synth.make_model_weights(cfg)
    m = qg.Model(w)
    a, b = qg.State(m, cfg.max_seq_len), qg.State(m, cfg.max_seq_len)
    ta = tb = 5
    for p in range(8):
        ta = qg.qg_decode_token(m, a, ta, p)
        tb = qg.qg_decode_batch(m, [b], [tb], [p])[0]
        assert ta == tb
        assert rel(b.download_hidden(), a.download_hidden()) <= TOL


def test_batch_arguments():
    cfg = synth.CFG_TINY
    w = synth.make_model_weights(cfg)
    m = qg.Model(w)
    s1, s2 = qg.State(m, cfg.max_seq_len), qg.State(m, cfg.max_seq_len)
    q = qg.State(m, cfg.max_seq_len, qg.KV_Q8_0_Q5_1)
    with pytest.raises(qg.QgError) as e:
        qg.qg_decode_batch(m, [s1, s1], [1, 2], [0, 0])
    assert e.value.code == qg.QG_ERR_ARG
    with pytest.raises(qg.QgError) as e:
        qg.qg_decode_batch(m, [s1, q], [1, 2], [0, 0])
    assert e.value.code == qg.QG_ERR_ARG
    with pytest.raises(qg.QgError) as e:
        qg.qg_decode_batch(m, [s1, s2], [1, cfg.vocab], [0, 0])
    assert e.value.code == qg.QG_ERR_TOKEN
    with pytest.raises(qg.QgError) as e:
        qg.qg_decode_batch(m, [s1, s2], [1, 2], [0, cfg.max_seq_len])
    assert e.value.code == qg.QG_ERR_POS
    many = [qg.State(m, 8) for _ in range(17)]
    with pytest.raises(qg.QgError) as e:
        qg.qg_decode_batch(m, many, [1] * 17, [0] * 17)
    assert e.value.code == qg.QG_ERR_SHAPE


def test_batch_token_masks_per_sequence():
    """The batched lm_head keeps each sequence's own token mask: sequence 0
    unmasked, sequence 1 under a random allow set, sequence 2 allowed one id."""
    cfg = dataclasses.replace(synth.CFG_TINY, max_seq_len=64)
    w = synth.make_model_weights(cfg)
    m, om = qg.Model(w), oracle.Model(w)
    V = cfg.vocab
    rng = np.random.default_rng(synth.subseed(synth.MASTER_SEED, "batch.masks"))

    def allow(ids):
        words = np.zeros((V + 31) // 32, np.uint32)
        for i in ids:
            words[i >> 5] |= np.uint32(1) << np.uint32(i & 31)
        return words

    masks = [None, allow(np.flatnonzero(rng.random(V) < 0.2)), allow([int(rng.integers(V))])]
    states = [qg.State(m, cfg.max_seq_len) for _ in range(3)]
    ostates = [oracle.State(om) for _ in range(3)]
    for st, mk in zip(states, masks):
        st.set_token_mask(mk)
    toks, pos = [11, 12, 13], [0, 0, 0]
    for step in range(5):
        got = qg.qg_decode_batch(m, states, toks, pos)
        for i in range(3):
            ref, _, lg = oracle.forward_token(om, ostates[i], toks[i], pos[i], want_logits=True)
            want = ref if masks[i] is None else oracle.argmax_masked(lg, masks[i])
            if masks[i] is not None:
                assert (masks[i][got[i] >> 5] >> np.uint32(got[i] & 31)) & 1, f"seq {i}: banned id {got[i]}"
                x = lg.astype(np.float64).copy()
                ids = np.arange(V)
                x[((masks[i][ids >> 5] >> (ids & 31).astype(np.uint32)) & 1) == 0] = -np.finfo(np.float32).max
                assert _token_ok(got[i], want, x.astype(np.float32))
            else:
                assert _token_ok(got[i], want, lg)
            toks[i], pos[i] = want, pos[i] + 1


@pytest.mark.parametrize("kv_format", [qg.KV_F32, qg.KV_Q8_0_Q5_1])
def test_batch_graph_matches_eager_bitwise(kv_format):
    """qg_batch_step (one captured graph, positions read on the device) against
    qg_decode_batch on twin states: the same kernels in the same order, so the
    same tokens and bitwise the same residual streams, step after step."""
    cfg = dataclasses.replace(synth.CFG_TINY, max_seq_len=64)
    w = synth.make_model_weights(cfg)
    m = qg.Model(w)
    n = 3
    ea = [qg.State(m, cfg.max_seq_len, kv_format) for _ in range(n)]
    gr = [qg.State(m, cfg.max_seq_len, kv_format) for _ in range(n)]
    toks, pos = [], []
    for i in range(n):
        prompt = synth.tokens(synth.subseed(synth.MASTER_SEED, f"batch.graph.{i}"), cfg.vocab, 3 + 2 * i)
        a = qg.qg_prefill(m, ea[i], prompt)
        b = qg.qg_prefill(m, gr[i], prompt)
        assert a == b
        toks.append(a)
        pos.append(len(prompt))
    bt = qg.Batch(m, gr)
    for step in range(6):
        te = qg.qg_decode_batch(m, ea, toks, pos)
        tg = bt.step(toks, pos)
        assert te == tg, f"step {step}: eager {te} graph {tg}"
        for i in range(n):
            assert np.array_equal(ea[i].download_hidden(), gr[i].download_hidden())
        toks, pos = te, [p + 1 for p in pos]
    for i in range(n):
        assert gr[i].kv_len == pos[i]
    bt.close()
    qg.qg_device_status()


def test_batch_graph_arguments():
    cfg = synth.CFG_TINY
    w = synth.make_model_weights(cfg)
    m = qg.Model(w)
    s1, s2 = qg.State(m, cfg.max_seq_len), qg.State(m, cfg.max_seq_len)
    with pytest.raises(qg.QgError) as e:
        qg.Batch(m, [s1, s1])
    assert e.value.code == qg.QG_ERR_ARG
    with pytest.raises(qg.QgError) as e:
        qg.Batch(m, [s1, qg.State(m, cfg.max_seq_len, qg.KV_Q8_0_Q5_1)])
    assert e.value.code == qg.QG_ERR_ARG
    bt = qg.Batch(m, [s1, s2])
    with pytest.raises(qg.QgError) as e:
        bt.step([1, cfg.vocab], [0, 0])
    assert e.value.code == qg.QG_ERR_TOKEN
    with pytest.raises(qg.QgError) as e:
        bt.step([1, 2], [0, cfg.max_seq_len])
    assert e.value.code == qg.QG_ERR_POS
    # refused inputs change nothing: the first real step still matches the eager call
    t3, t4 = qg.State(m, cfg.max_seq_len), qg.State(m, cfg.max_seq_len)
    assert bt.step([1, 2], [0, 0]) == qg.qg_decode_batch(m, [t3, t4], [1, 2], [0, 0])
    bt.close()
