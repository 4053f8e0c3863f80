"""The quantized KV cache's records and the oracle's GGUF blocks, both ways,
and teacher forcing of the oracle's cache to the GPU's.

The GPU keeps, per (kv head, position), a 272-byte K record (the eight
q8_0 scales f16, then the 256 int8 codes) and a 192-byte V record (eight q5_1
(d, m) f16 pairs, eight qh words, eight 16-byte qs runs); the oracle keeps
each row as GGUF q8_0 (34-byte) / q5_1 (24-byte) blocks in kv-dimension
order.  Each side quantizes a new row from its own f32 row, and the two f32
rows agree to ~1e-6 of their magnitude, so a code within that distance of a
rounding boundary may come out one step apart.  sync_rows puts the GPU's
records into the oracle's cache (bytes and dequantized rows), so that such a
difference does not carry into later steps: every step is then compared at
the decode's own bar.
"""
import numpy as np

import oracle


def records(kb, vb, nkv):
    """GGUF-order q8_0 / q5_1 blocks of rows [t][kvd/32 blocks] -> the cache's
    records: K [nkv][t][d x8 | q x256], V [nkv][t][(d, m) x8 | qh x8 | qs x8]."""
    t = kb.shape[0]
    kb = kb.reshape(t, nkv, 8, 34)
    K = np.concatenate([kb[..., :2].reshape(t, nkv, 16), kb[..., 2:].reshape(t, nkv, 256)], axis=2)
    vb = vb.reshape(t, nkv, 8, 24)
    V = np.concatenate([vb[..., :4].reshape(t, nkv, 32), vb[..., 4:8].reshape(t, nkv, 32),
                        vb[..., 8:].reshape(t, nkv, 128)], axis=2)
    return np.ascontiguousarray(K.transpose(1, 0, 2)), np.ascontiguousarray(V.transpose(1, 0, 2))


def gguf_blocks(K, V):
    """The inverse of records: K [nkv][t][272], V [nkv][t][192] -> the rows'
    GGUF q8_0 blocks [t][nkv*8*34] and q5_1 blocks [t][nkv*8*24]."""
    nkv, t = K.shape[:2]
    Kt = K.transpose(1, 0, 2)  # [t][nkv][272]
    kb = np.concatenate([Kt[..., :16].reshape(t, nkv, 8, 2), Kt[..., 16:].reshape(t, nkv, 8, 32)], axis=3)
    Vt = V.transpose(1, 0, 2)  # [t][nkv][192]
    vb = np.concatenate([Vt[..., :32].reshape(t, nkv, 8, 4), Vt[..., 32:64].reshape(t, nkv, 8, 4),
                         Vt[..., 64:].reshape(t, nkv, 8, 16)], axis=3)
    return np.ascontiguousarray(kb.reshape(t, -1)), np.ascontiguousarray(vb.reshape(t, -1))


def codes(kb, vb):
    """int codes of GGUF rows: q8_0 [t][kvd] in -128..127, q5_1 [t][kvd] in 0..31,
    and the scale bytes of both."""
    t = kb.shape[0]
    k = kb.reshape(t, -1, 34)
    kq = k[..., 2:].view(np.int8).astype(np.int32).reshape(t, -1)
    v = vb.reshape(t, -1, 24)
    qh = v[..., 4:8].copy().view(np.uint32)  # [t][blocks][1]
    qs = v[..., 8:].astype(np.int32)         # [t][blocks][16]
    j = np.arange(32)
    nib = np.where(j < 16, qs[..., j % 16] & 15, qs[..., j % 16] >> 4)
    hi = ((qh >> j.astype(np.uint32)) & 1).astype(np.int32)
    vq = (nib | (hi << 4)).reshape(t, -1)
    return kq, vq, k[..., :2].copy(), v[..., :4].copy()


def _f16_steps(a, b):
    """How many binary16 values apart two arrays of f16 bytes are (ordered
    integer keys of the bit patterns)."""
    def key(x):
        u = x.copy().view(np.uint16).astype(np.int32)
        return np.where(u & 0x8000, -(u & 0x7fff), u)
    return int(np.max(np.abs(key(a) - key(b)))) if a.size else 0


def sync_rows(gpu_state, ost, il, r0, r1, nkv, row_tol=1e-5):
    """Rows r0..r1-1 of attention layer il: compare the GPU's records with the
    oracle's, then give the oracle the GPU's records (bytes and dequantized
    rows).  Returns (codes that differ, largest code difference, largest
    distance of a reconstructed value from the oracle's in units of its
    block's step plus the rows' agreement).  The two sides' f32 rows agree to
    row_tol of the row's largest magnitude (the bar of the f32 K/V rows); each
    side's reconstruction is within half a step of its own row, so the two
    are within one step plus that agreement: the returned distance is <= 1
    unless a record is wrong.  A scale may round to another f16 value and a
    code be one step apart without breaking it."""
    K, V = gpu_state.download_kv_records(il)
    kb, vb = gguf_blocks(K[:, r0:r1], V[:, r0:r1])
    gk, gv, _, _ = codes(kb, vb)
    ok_, ov_, oks, ovs = codes(ost.kq[il][r0:r1], ost.vq[il][r0:r1])
    diff = int(np.count_nonzero(gk != ok_) + np.count_nonzero(gv != ov_))
    step = int(max(np.max(np.abs(gk - ok_)), np.max(np.abs(gv - ov_))))
    t = r1 - r0
    dist = 0.0
    for gb, ob, deq, sc in ((kb, ost.kq[il][r0:r1], oracle.dequantize_q8_0, oks),
                            (vb, ost.vq[il][r0:r1], oracle.dequantize_q5_1, ovs)):
        xg = deq(gb.reshape(-1)).reshape(t, -1).astype(np.float64)
        xo = deq(np.ascontiguousarray(ob).reshape(-1)).reshape(t, -1).astype(np.float64)
        d = np.abs(sc.reshape(t, -1, sc.shape[-1] // 2 * 2)[..., :2].copy().view(np.float16).astype(np.float64))
        unit = np.repeat(d.reshape(t, -1), 32, axis=1) + row_tol * np.max(np.abs(xo), axis=1, keepdims=True) + 1e-30
        dist = max(dist, float(np.max(np.abs(xg - xo) / unit)))
    scales = dist
    ost.kq[il][r0:r1] = kb
    ost.vq[il][r0:r1] = vb
    ost.kc[il][r0:r1] = oracle.dequantize_q8_0(kb.reshape(-1)).reshape(r1 - r0, -1)
    ost.vc[il][r0:r1] = oracle.dequantize_q5_1(vb.reshape(-1)).reshape(r1 - r0, -1)
    return diff, step, scales
