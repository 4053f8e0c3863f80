"""The record <-> GGUF block conversion of the quantized-cache teacher forcing
(tests/kvq_sync.py), on random bytes and on the oracle's own blocks."""
import numpy as np

import oracle
from kvq_sync import codes, gguf_blocks, records


def test_records_and_blocks_are_inverse():
    rng = np.random.default_rng(5)
    for nkv, t in ((1, 3), (2, 5), (4, 7)):
        kb = rng.integers(0, 256, (t, nkv * 8 * 34), dtype=np.uint8)
        vb = rng.integers(0, 256, (t, nkv * 8 * 24), dtype=np.uint8)
        K, V = records(kb, vb, nkv)
        assert K.shape == (nkv, t, 272) and V.shape == (nkv, t, 192)
        kb2, vb2 = gguf_blocks(K, V)
        assert np.array_equal(kb2, kb) and np.array_equal(vb2, vb)


def test_codes_of_the_oracle_quantizer():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((3, 512)).astype(np.float32)
    kb = oracle.quantize_q8_0(x.reshape(-1)).reshape(3, -1)
    vb = oracle.quantize_q5_1(x.reshape(-1)).reshape(3, -1)
    kq, vq, ks, vs = codes(kb, vb)
    kd = ks.view(np.float16).astype(np.float32).reshape(3, -1)          # per 32-value block
    vd = vs.view(np.float16).astype(np.float32).reshape(3, -1, 2)
    assert np.array_equal(np.repeat(kd, 32, axis=1) * kq, oracle.dequantize_q8_0(kb.reshape(-1)).reshape(3, -1))
    want_v = np.repeat(vd[..., 0], 32, axis=1) * vq + np.repeat(vd[..., 1], 32, axis=1)
    assert np.array_equal(want_v.astype(np.float32), oracle.dequantize_q5_1(vb.reshape(-1)).reshape(3, -1))
    assert kq.min() >= -127 and kq.max() <= 127 and vq.min() >= 0 and vq.max() <= 31


def test_f16_step_distance():
    from kvq_sync import _f16_steps
    a = np.array([1.0, -2.0, 0.5], np.float16).view(np.uint8)
    b = np.array([np.nextafter(np.float16(1.0), np.float16(2.0)), -2.0, 0.5], np.float16).view(np.uint8)
    assert _f16_steps(a, a) == 0 and _f16_steps(a, b) == 1
    c = np.array([1.0, np.nextafter(np.float16(-2.0), np.float16(-3.0)), 0.5], np.float16).view(np.uint8)
    assert _f16_steps(a, c) == 1


def test_sync_distance_of_requantized_rows():
    """Rows that differ by 1e-6 of their magnitude quantize to records whose
    reconstructions sync_rows finds within one step of each other."""
    import types
    from kvq_sync import sync_rows, records
    rng = np.random.default_rng(8)
    nkv, t = 2, 6
    x = rng.standard_normal((t, nkv * 256)).astype(np.float32)
    y = (x * (1 + 1e-6 * rng.standard_normal(x.shape))).astype(np.float32)
    kx, vx = oracle.quantize_q8_0(x.reshape(-1)).reshape(t, -1), oracle.quantize_q5_1(x.reshape(-1)).reshape(t, -1)
    ky, vy = oracle.quantize_q8_0(y.reshape(-1)).reshape(t, -1), oracle.quantize_q5_1(y.reshape(-1)).reshape(t, -1)
    K, V = records(ky, vy, nkv)
    gpu = types.SimpleNamespace(download_kv_records=lambda il: (K, V))
    ost = types.SimpleNamespace(kq=[kx.copy()], vq=[vx.copy()], kc=[np.zeros((t, nkv * 256), np.float32)],
                                vc=[np.zeros((t, nkv * 256), np.float32)])
    diff, step, dist = sync_rows(gpu, ost, 0, 0, t, nkv)
    assert step <= 1 and dist <= 1.0
    assert np.array_equal(ost.kq[0], ky) and np.array_equal(ost.vq[0], vy)
    assert np.array_equal(ost.vc[0], oracle.dequantize_q5_1(vy.reshape(-1)).reshape(t, -1))
