"""Pins of the oracle's quantized KV cache (q8_0 K / q5_1 V blocks, f32 ->
f16 rounding, quantize-on-append in the attention layer) against things other
than itself: hand-worked block bytes, numpy's IEEE binary16 conversion, exact
round trips of representable values, the rounding rule at exact ties, the
error bound of a rounding quantizer, and the f32 cache path of the same layer.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import synth


# ------------------------------------------------------------ f32 -> f16
def test_f32_to_f16_matches_numpy_ieee_binary16():
    rng = np.random.default_rng(7)
    xs = [rng.standard_normal(20000).astype(np.float32) * np.float32(s) for s in (1e-7, 1e-5, 1e-2, 1, 1e3, 3e4)]
    # every half value and every midpoint between neighbours (exact ties), both signs
    h = np.arange(0, 0x7c00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = ((h[:-1] + h[1:]) / 2).astype(np.float32)
    assert np.all(mids.astype(np.float64) == (h[:-1] + h[1:]) / 2)  # the ties are exact in f32
    special = np.array([0.0, -0.0, 65504, 65519.996, 65520, 65536, 1e6, -1e6, 2.0 ** -24, 2.0 ** -25,
                        1.5 * 2.0 ** -25, 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 1e-40, np.inf, -np.inf],
                       np.float32)
    x = np.concatenate(xs + [h.astype(np.float32), mids, -mids, special])
    got = oracle.f32_to_f16_bits(x)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, f"{bad.size} mismatches, first x={x[bad[0]]!r}: {got[bad[0]]:#x} vs {want[bad[0]]:#x}"
    assert (oracle.f32_to_f16_bits(np.float32(np.nan))[0] & 0x7fff) > 0x7c00


# ---------------------------------------------------------------- q8_0
def test_q8_0_hand_block_exact_round_trip():
    """Codes -127..121 step 8 times 1/8: max|x| = 127/8, so d = 1/8 exactly
    (half 0x3000), every code is x*8, and the round trip is exact."""
    q = np.arange(-127, 129, 8)
    x = (q / 8).astype(np.float32)
    b = oracle.quantize_q8_0(x)
    assert b.size == 34
    assert b[0] == 0x00 and b[1] == 0x30
    assert np.array_equal(b[2:].view(np.int8), q.astype(np.int8))
    assert np.array_equal(oracle.dequantize_q8_0(b), x)


def test_q8_0_ties_round_half_away_and_zero_block():
    # max|x| = 127 -> d = 1, id = 1: x * id is x itself
    x = np.zeros(32, np.float32)
    x[:8] = [127, 2.5, -2.5, 0.5, -0.5, 1.5, -126.5, 3.4999998]
    b = oracle.quantize_q8_0(x)
    assert (b[0], b[1]) == (0x00, 0x3c)
    assert list(b[2:10].view(np.int8)) == [127, 3, -3, 1, -1, 2, -127, 3]
    z = oracle.quantize_q8_0(np.zeros(64, np.float32))
    assert not z.any() and not oracle.dequantize_q8_0(z).any()


def test_q8_0_error_bound_random():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(32 * 400) * np.repeat(10.0 ** rng.uniform(-3, 2, 400), 32)).astype(np.float32)
    b = oracle.quantize_q8_0(x)
    xr = oracle.dequantize_q8_0(b)
    for blk in range(400):
        xb, rb = x[32 * blk:32 * blk + 32].astype(np.float64), xr[32 * blk:32 * blk + 32].astype(np.float64)
        d = np.abs(xb).max() / 127
        d16 = float(b[34 * blk:34 * blk + 2].view(np.float16)[0])
        assert abs(d16 - d) <= max(d * 2.0 ** -11, 2.0 ** -25) * 1.0001  # relative, or half a subnormal step
        # a rounding quantizer: half a step, plus the f16 rounding of d times the code
        assert np.all(np.abs(xb - rb) <= d / 2 * 1.0001 + 127 * abs(d16 - d) + 1e-30)


# ---------------------------------------------------------------- q5_1
def test_q5_1_hand_blocks():
    """x_j = j: min 0, max 31 -> d = 1, m = 0, q_j = j; qh has bits 16..31;
    qs[i] packs q_i (low) and q_{i+16} (high nibble i) -> 0x11 * i."""
    b = oracle.quantize_q5_1(np.arange(32, dtype=np.float32))
    assert b.size == 24
    assert b[:8].tobytes() == bytes([0x00, 0x3c, 0x00, 0x00, 0x00, 0x00, 0xff, 0xff])
    assert b[8:].tobytes() == bytes(0x11 * i for i in range(16))
    assert np.array_equal(oracle.dequantize_q5_1(b), np.arange(32, dtype=np.float32))
    # x_j = 2j - 10: d = 2 (0x4000), m = -10 (0xc900), the same codes
    b2 = oracle.quantize_q5_1((2 * np.arange(32) - 10).astype(np.float32))
    assert b2[:4].tobytes() == bytes([0x00, 0x40, 0x00, 0xc9])
    assert b2[4:].tobytes() == b[4:].tobytes()
    assert np.array_equal(oracle.dequantize_q5_1(b2), (2 * np.arange(32) - 10).astype(np.float32))


def test_q5_1_ties_and_constant_block():
    x = np.zeros(32, np.float32)
    x[1] = 31.0  # min 0, max 31 -> d = 1
    x[2:6] = [2.5, 0.5, 30.5, 15.5]
    b = oracle.quantize_q5_1(x)
    r = oracle.dequantize_q5_1(b)
    assert list(r[:6]) == [0, 31, 3, 1, 31, 16]
    c = oracle.quantize_q5_1(np.full(32, 3.0, np.float32))  # max == min: d = 0, every code 0, x = m
    assert c[:2].tobytes() == b"\x00\x00" and c[2:4].tobytes() == bytes([0x00, 0x42])
    assert not c[4:].any()
    assert np.array_equal(oracle.dequantize_q5_1(c), np.full(32, 3.0, np.float32))


def test_q5_1_error_bound_random():
    rng = np.random.default_rng(12)
    x = (rng.standard_normal(32 * 400) * np.repeat(10.0 ** rng.uniform(-3, 2, 400), 32)
         + np.repeat(rng.standard_normal(400), 32)).astype(np.float32)
    b = oracle.quantize_q5_1(x)
    xr = oracle.dequantize_q5_1(b)
    for blk in range(400):
        xb, rb = x[32 * blk:32 * blk + 32].astype(np.float64), xr[32 * blk:32 * blk + 32].astype(np.float64)
        d, m = (xb.max() - xb.min()) / 31, xb.min()
        d16, m16 = (float(v) for v in b[24 * blk:24 * blk + 4].view(np.float16))
        bound = d / 2 * 1.0001 + 31 * abs(d16 - d) + abs(m16 - m) + 4 * np.spacing(np.float32(np.abs(xb).max()))
        assert np.all(np.abs(xb - rb) <= bound)


def test_prescaled_values_decide_the_codes():
    rng = np.random.default_rng(13)
    x = rng.standard_normal(32 * 50).astype(np.float32)
    q8 = oracle.quantize_q8_0(x).reshape(50, 34)[:, 2:].view(np.int8).reshape(-1)
    pre8 = oracle.kv_prescaled(x, 0).astype(np.float64)
    half_away = np.sign(pre8) * np.floor(np.abs(pre8) + 0.5)
    assert np.array_equal(q8, half_away.astype(np.int8))
    pre5 = oracle.kv_prescaled(x, 1).astype(np.float64)
    r5 = oracle.dequantize_q5_1(oracle.quantize_q5_1(x)).reshape(50, 32)
    b5 = oracle.quantize_q5_1(x).reshape(50, 24)
    d16 = b5[:, 0:2].copy().view(np.float16).astype(np.float64)
    m16 = b5[:, 2:4].copy().view(np.float16).astype(np.float64)
    codes = np.rint((r5 - m16) / d16).reshape(-1)
    assert np.array_equal(codes, np.clip(np.floor(pre5 + 0.5), 0, 31))


# ------------------------------------------- quantize-on-append in the layer
def _attn_cfg():
    return dataclasses.replace(synth.CFG_TINY, name="tiny-attn1", n_layers=1, vocab=512,
                               layer_kinds=(synth.ATTENTION,), max_seq_len=64)


def test_attention_layer_quantized_cache_appends_the_f32_rows_quantized():
    """Side by side, an f32-cache state and a quantized-cache state with the
    same history (the quantized one holding its q8_0/q5_1 blocks): the new
    row's blocks are the quantization of the f32 path's new K/V rows at pos,
    the rows the attention read are their dequantized values, older rows are
    untouched, and the two outputs differ by no more than quantization
    noise."""
    cfg = _attn_cfg()
    w = synth.make_model_weights(cfg)
    om = oracle.Model(w)
    pos = 20
    k, v = synth.long_context_kv(cfg, 0, pos)
    sf, sq = oracle.State(om), oracle.State(om, oracle.KV_Q8_0_Q5_1)
    sf.set_kv_rows(0, k, v)
    sq.set_kv_rows(0, k, v)
    kq0, vq0 = sq.kq[0].copy(), sq.vq[0].copy()
    x = synth.normal(synth.subseed(synth.MASTER_SEED, "kvq.layer"), cfg.hidden)
    hf = oracle.attention_layer(om, sf, 0, x, pos)
    hq = oracle.attention_layer(om, sq, 0, x, pos)
    assert np.array_equal(sq.kq[0][pos], oracle.quantize_q8_0(sf.kc[0][pos]))
    assert np.array_equal(sq.vq[0][pos], oracle.quantize_q5_1(sf.vc[0][pos]))
    assert np.array_equal(sq.kc[0][pos], oracle.dequantize_q8_0(sq.kq[0][pos]))
    assert np.array_equal(sq.vc[0][pos], oracle.dequantize_q5_1(sq.vq[0][pos]))
    assert np.array_equal(sq.kq[0][:pos], kq0[:pos]) and np.array_equal(sq.vq[0][:pos], vq0[:pos])
    assert not sq.kq[0][pos + 1:].any()
    e = np.max(np.abs(hq - hf)) / np.max(np.abs(hf))
    assert 0 < e < 5e-2, e


def test_attention_layer_quantized_equals_f32_on_representable_cache():
    """When every K/V value the attention reads is exactly representable in
    its block format, the quantized cache changes nothing: history rows made
    of q8_0 / q5_1 codes times power-of-two scales, and the new row's K/V
    forced representable by zero projection weights (its K row is then zero,
    its V row zero: both exact)."""
    cfg = _attn_cfg()
    w = synth.make_model_weights(cfg)
    L = w.layers[0]
    for name in ("attn_k", "attn_v"):
        t = getattr(L, name)
        z = dataclasses.replace(t, data=np.zeros_like(t.data))
        setattr(L, name, z)
    om = oracle.Model(w)
    pos, kvd = 12, cfg.kv_dim
    rng = np.random.default_rng(5)
    kcodes = rng.integers(-127, 128, (pos, kvd))
    kcodes[:, ::32] = 127  # max |code| 127 in every block: d = 2^-5 exactly
    k = (kcodes * 2.0 ** -5).astype(np.float32)
    vcodes = rng.integers(0, 32, (pos, kvd))
    vcodes[:, ::32], vcodes[:, 1::32] = 0, 31  # min code 0, max 31: d = 2^-4, m = -1
    v = (vcodes * 2.0 ** -4 - 1).astype(np.float32)
    sf, sq = oracle.State(om), oracle.State(om, oracle.KV_Q8_0_Q5_1)
    sf.set_kv_rows(0, k, v)
    sq.set_kv_rows(0, k, v)
    assert np.array_equal(sq.kc[0][:pos], k) and np.array_equal(sq.vc[0][:pos], v)
    x = synth.normal(synth.subseed(synth.MASTER_SEED, "kvq.exact"), cfg.hidden)
    hf = oracle.attention_layer(om, sf, 0, x, pos)
    hq = oracle.attention_layer(om, sq, 0, x, pos)
    assert np.array_equal(hf, hq)
