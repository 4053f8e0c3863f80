"""GEMV (Q4_K from raw rows; Q6_K from raw rows and from the planar repack),
the Q6_K planar repack, fused lm_head + argmax and argmax on the GPU, through
the C ABI, against the CPU oracle on the same seeded inputs.

Bar (pages' float-GEMV parity, forward_qwen35_cuda.rs pin_reference_gemv):
the GPU result must sit inside the error bound of the exact (f64) product
that its arithmetic guarantees and within 1e-5 normwise of the f32 oracle.
On the GEMV engine x is held to 2^-23 of each 256-element block's largest
magnitude M_b, sub-block sums are exact integers, accumulation is f32:
|y - y_exact| <= 2^-23 * sum_k |w_k| M_b(k) + 8 * 2^-24 * sum_k |w_k x_k|.
The raw-row Q6_K kernel is plain f32 with at most k/256 + 13 roundings per
product: |y - y_exact| <= (k/256 + 16) * 2^-24 * sum_k |w_k x_k|.  Argmax
indices are compared bit-exactly.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

qg = pytest.importorskip("quantized_gemv_gated_gb300")

F32_EPS = 2.0 ** -24


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def planar(t):
    """Device planar copy of a synth Q6_K tensor (through the library's repack)."""
    src = dev(t.data)
    dst = torch.empty(qg.qg_q6k_planar_bytes(t.n, t.k), dtype=torch.uint8, device="cuda")
    qg.qg_q6k_to_planar(src, dst, t.n, t.k)
    return dst


def run_gemv(t, x, layout="engine"):
    """y = W x on the GPU.  layout "engine": Q4_K from raw rows and Q6_K from
    the planar repack, both on the GEMV engine; "rows": Q6_K straight from raw
    GGUF rows (qg_gemv_q6k, plain f32 arithmetic)."""
    y = torch.empty(t.n, dtype=torch.float32, device="cuda")
    xd = dev(x)
    if t.qtype == synth.QTYPE_Q4_K:
        assert layout == "engine"
        qg.qg_gemv_q4k(dev(t.data), xd, y, t.n, t.k)
    elif layout == "rows":
        qg.qg_gemv_q6k(dev(t.data), xd, y, t.n, t.k)
    else:
        qg.qg_gemv_q6k_planar(planar(t), xd, y, t.n, t.k)
    torch.cuda.synchronize()
    qg.qg_device_status()
    return y.cpu().numpy()


def check_against_oracle(t, x, y, tight=True, layout="engine"):
    exact = oracle.gemv_f64(t, x)
    W = np.abs(oracle.dequant(t).astype(np.float64))
    ax = np.abs(x.astype(np.float64))
    if layout == "rows":
        # plain f32: each product passes through at most k/256 + 13 roundings
        bound = (t.k // 256 + 16) * F32_EPS * (W @ ax) + 1e-30
        tight = True
    else:
        blockmax = np.repeat(ax.reshape(-1, 256).max(axis=1), 256)
        bound = 2 * F32_EPS * (W @ blockmax) + 8 * F32_EPS * (W @ ax) + 1e-30
    err = np.abs(y.astype(np.float64) - exact)
    assert np.all(err <= bound), f"max err/bound {float(np.max(err / bound)):.3g}"
    ref = oracle.gemv(t, x)
    rel = np.max(np.abs(y - ref)) / max(np.max(np.abs(ref)), 1e-30)
    assert rel <= (1e-5 if tight else 1e-4), rel


SMALL = [(1, 256), (13, 256), (37, 768), (300, 2560), (1000, 1024), (129, 3584), (64, 4096)]


# (quant type, layout) of every GEMV entry point: qg_gemv_q4k, qg_gemv_q6k_planar, qg_gemv_q6k
PATHS = [(synth.QTYPE_Q4_K, "engine"), (synth.QTYPE_Q6_K, "engine"), (synth.QTYPE_Q6_K, "rows")]


@pytest.mark.parametrize("n,k", SMALL)
@pytest.mark.parametrize("qtype,layout", PATHS)
def test_gemv_small_shapes(qtype, layout, n, k):
    gen = synth.q4k_tensor if qtype == synth.QTYPE_Q4_K else synth.q6k_tensor
    t = gen(1000 + n + k, n, k)
    x = synth.normal(77 + n, k)
    check_against_oracle(t, x, run_gemv(t, x, layout), layout=layout)


@pytest.mark.parametrize("qtype,layout", PATHS)
def test_gemv_special_inputs(qtype, layout):
    gen = synth.q4k_tensor if qtype == synth.QTYPE_Q4_K else synth.q6k_tensor
    t = gen(5, 40, 512)
    cases = [(np.zeros(512, np.float32), True),
             (np.full(512, 3.0, np.float32), True),
             ((synth.normal(6, 512) * np.float32(1e-30)).astype(np.float32), True),  # tiny blocks
             ((synth.normal(7, 512) * np.float32(1e20)).astype(np.float32), True),   # huge values
             # one large element per 256-block: the small ones keep only 2^-23 of the block's
             # largest magnitude, so only the representation bound is promised
             (np.where(np.arange(512) % 256 == 5, 100.0, 1e-3).astype(np.float32), False)]
    for x, tight in cases:
        y = run_gemv(t, x, layout)
        if not np.any(x):
            assert np.all(y == 0)
        else:
            check_against_oracle(t, x, y, tight, layout)


# the standalone-kernel sweep shapes, all rows against the oracle
SWEEP = [(1024, 1024), (6144, 1024), (9216, 2560), (2560, 9216)]


@pytest.mark.parametrize("n,k", SWEEP)
@pytest.mark.parametrize("qtype,layout", PATHS)
def test_gemv_sweep_shapes(qtype, layout, n, k):
    gen = synth.q4k_tensor if qtype == synth.QTYPE_Q4_K else synth.q6k_tensor
    t = gen(synth.subseed(synth.MASTER_SEED, f"sweep.{qtype}.{n}x{k}"), n, k)
    x = synth.normal(synth.subseed(synth.MASTER_SEED, f"sweep.x.{k}"), k)
    y = run_gemv(t, x, layout)
    ref = oracle.gemv(t, x)
    rel = np.max(np.abs(y - ref)) / np.max(np.abs(ref))
    assert rel <= 1e-5, rel
    rows = np.arange(0, n, max(1, n // 97))
    sub = synth.QTensor(t.data.reshape(n, -1)[rows].ravel().copy(), t.qtype, len(rows), k)
    check_against_oracle(sub, x, y[rows], layout=layout)


@pytest.mark.parametrize("off", [2, 6, 14])
def test_gemv_q6k_rows_odd_offset_and_long_k(off):
    """Raw Q6_K rows start wherever the file puts them: 210-byte blocks leave
    a row (and a tensor inside a mapped file) only 2-byte aligned, and the
    row kernel has no K limit.  W at an offset of `off` bytes from a 16-byte
    boundary, k = 16640 (past the engine's 16384; 65 blocks, so every row
    takes four full 16-block chunks and a one-block chunk, each with its own
    ragged head and tail)."""
    n, k = 45, 16640
    t = synth.q6k_tensor(synth.subseed(synth.MASTER_SEED, "rows.odd"), n, k)
    x = synth.normal(synth.subseed(synth.MASTER_SEED, "rows.odd.x"), k)
    buf = torch.zeros(t.data.size + 16, dtype=torch.uint8, device="cuda")
    buf[off:off + t.data.size] = dev(t.data)
    y = torch.empty(n, dtype=torch.float32, device="cuda")
    qg.qg_gemv_q6k(buf[off:], dev(x), y, n, k)
    torch.cuda.synchronize()
    qg.qg_device_status()
    check_against_oracle(t, x, y.cpu().numpy(), layout="rows")
    with pytest.raises(qg.QgError) as e:  # odd byte address: refused before any launch
        qg.qg_gemv_q6k(buf[1:], dev(x), y, n, k)
    assert e.value.code == qg.QG_ERR_ARG


def _planar_slice(nb, b):
    """(first block, width) of the K slice holding super-block b: slices of 8
    blocks, then 4, 2 and 1 for the remainder (qg.h, planar Q6_K)."""
    full = nb // 8
    if b < 8 * full:
        return b - b % 8, 8
    c = 8 * full
    for w in (4, 2, 1):
        if (nb - 8 * full) & w:
            if b < c + w:
                return c, w
            c += w
    raise AssertionError(b)


@pytest.mark.parametrize("n,k", [(13, 512), (13, 2560), (21, 3584)])
def test_q6k_planar_roundtrip_bytes(n, k):
    """The planar (8-row grouped, slice-major) Q6_K layout of qg.h, byte by
    byte: in each 1680-byte group-block, per row rr and quarter cq (u = 4 rr
    + cq) a 48-byte record [ql A | ql B | qh] at 48u, the quarter's four
    scales at 1536 + 4u, d at 1664 + 2 rr; padding rows are zero."""
    nb = k // 256
    t = synth.q6k_tensor(3 + k, n, k)
    p = planar(t).cpu().numpy()
    n8 = (n + 7) // 8 * 8
    assert p.size == n8 * nb * 210
    blocks = t.data.reshape(n, nb, 210)
    seen = set()
    for g in range(n8 // 8):
        for b in range(nb):
            b0, kb = _planar_slice(nb, b)
            off = ((n8 // 8) * b0 + g * kb + (b - b0)) * 1680
            seen.add(off)
            gb = p[off:off + 1680]
            for rr in range(8):
                r = 8 * g + rr
                recs = [gb[48 * (4 * rr + cq):48 * (4 * rr + cq + 1)] for cq in range(4)]
                scs = [gb[1536 + 4 * (4 * rr + cq):1536 + 4 * (4 * rr + cq + 1)] for cq in range(4)]
                dd = gb[1664 + 2 * rr:1666 + 2 * rr]
                if r >= n:
                    assert not any(np.any(x) for x in recs + scs) and not np.any(dd)
                    continue
                blk = blocks[r, b]
                ql, qh, sc = blk[:128], blk[128:192], blk[192:208]
                for cq in range(4):
                    half, part = cq >> 1, cq & 1
                    rec = recs[cq]
                    assert np.array_equal(rec[:16], ql[64 * half + 16 * part:64 * half + 16 * part + 16])
                    assert np.array_equal(rec[16:32], ql[64 * half + 32 + 16 * part:64 * half + 48 + 16 * part])
                    assert np.array_equal(rec[32:48], qh[16 * cq:16 * cq + 16])
                    assert np.array_equal(scs[cq], sc[[8 * half + part + 2 * s for s in range(4)]])
                assert np.array_equal(dd, blk[208:210])
    assert len(seen) == (n8 // 8) * nb  # every group-block has its own place


# ------------------------------------------------------------------ argmax

def lmhead(t, x):
    w = planar(t)
    ws = torch.zeros(qg.qg_lmhead_argmax_workspace_bytes() // 8, dtype=torch.int64, device="cuda")
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    qg.qg_lmhead_argmax(w, dev(x), t.n, t.k, ws, tok)
    torch.cuda.synchronize()
    assert int(ws.abs().sum()) == 0  # the workspace is left zeroed
    return int(tok.item())


def test_lmhead_argmax_full_vocab():
    V, H = 248320, 1024
    t = synth.q6k_tensor(synth.subseed(synth.MASTER_SEED, "lmhead.test"), V, H)
    x = synth.normal(synth.subseed(synth.MASTER_SEED, "lmhead.x"), H)
    logits = oracle.gemv(t, x)
    a, b = oracle.top2(logits)
    assert a - b > 1e-3 * abs(a)  # a clear winner for this seed
    assert lmhead(t, x) == oracle.argmax(logits)


def test_lmhead_argmax_planted_ties_pick_first_index():
    V, H = 50000, 1024
    t = synth.q6k_tensor(11, V, H)
    x = synth.normal(12, H)
    rows = t.data.reshape(V, -1)
    best = oracle.argmax(oracle.gemv(t, x))
    rng = np.random.default_rng(3)
    for trial in range(3):
        copies = rng.choice(V, size=rng.integers(2, 8), replace=False)
        data = rows.copy()
        data[copies] = rows[best]  # identical bytes -> identical logits
        tt = synth.QTensor(data.ravel(), t.qtype, V, H)
        expect = int(min(list(copies) + [best]))
        assert oracle.argmax(oracle.gemv(tt, x)) == expect
        assert lmhead(tt, x) == expect


def test_lmhead_ragged_vocab():
    t = synth.q6k_tensor(21, 3001, 512)
    x = synth.normal(22, 512)
    assert lmhead(t, x) == oracle.argmax(oracle.gemv(t, x))


def test_argmax_f32_planted_ties_inf_nan():
    rng = np.random.default_rng(9)
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    for trial in range(10):
        n = int(rng.integers(1, 300000))
        x = rng.standard_normal(n).astype(np.float32)
        idx = np.sort(rng.choice(n, size=min(n, int(rng.integers(1, 9))), replace=False))
        x[idx] = np.float32(x.max() + 1)
        qg.qg_argmax_f32(dev(x), n, out)
        torch.cuda.synchronize()
        assert int(out.item()) == oracle.argmax(x) == idx[0]
    x = np.zeros(1000, np.float32)
    x[10], x[500], x[3] = np.nan, np.inf, np.nan
    qg.qg_argmax_f32(dev(x), 1000, out)
    torch.cuda.synchronize()
    assert int(out.item()) == 500 == oracle.argmax(x)
    x = np.full(7, np.nan, np.float32)
    qg.qg_argmax_f32(dev(x), 7, out)
    torch.cuda.synchronize()
    assert int(out.item()) == 0 == oracle.argmax(x)
    x = np.array([-1.0, -0.0, 0.0], np.float32)
    qg.qg_argmax_f32(dev(x), 3, out)
    torch.cuda.synchronize()
    assert int(out.item()) == 1 == oracle.argmax(x)


def test_gemv_argument_errors():
    w = torch.zeros(144 * 4, dtype=torch.uint8, device="cuda")
    x = torch.zeros(1024, dtype=torch.float32, device="cuda")
    y = torch.zeros(4, dtype=torch.float32, device="cuda")
    with pytest.raises(qg.QgError) as e:
        qg.qg_gemv_q4k(w, x, y, 4, 300)
    assert e.value.code == qg.QG_ERR_SHAPE
    with pytest.raises(qg.QgError) as e:
        qg.qg_gemv_q4k(w, x, y, 0, 256)
    assert e.value.code == qg.QG_ERR_EMPTY
    with pytest.raises(qg.QgError) as e:
        qg.qg_gemv_q4k(w.data_ptr() + 4, x, y, 1, 256)
    assert e.value.code == qg.QG_ERR_ARG


def planar4(t):
    """Device planar copy of a synth Q4_K tensor (through the library's repack)."""
    src = dev(t.data)
    dst = torch.empty(qg.qg_q4k_planar_bytes(t.n, t.k), dtype=torch.uint8, device="cuda")
    qg.qg_q4k_to_planar(src, dst, t.n, t.k)
    return dst


@pytest.mark.parametrize("n,k", [(13, 512), (13, 2560), (21, 3584)])
def test_q4k_planar_roundtrip_bytes(n, k):
    """The planar Q4_K layout of qg.h byte by byte: 1152-byte group-blocks of
    the 8 rows' GGUF blocks in row order, slice-major; padding rows zero."""
    nb = k // 256
    t = synth.q4k_tensor(5 + k, n, k)
    p = planar4(t).cpu().numpy()
    n8 = (n + 7) // 8 * 8
    assert p.size == n8 * nb * 144 == qg.qg_q4k_planar_bytes(n, k)
    blocks = t.data.reshape(n, nb, 144)
    seen = set()
    for g in range(n8 // 8):
        for b in range(nb):
            b0, kb = _planar_slice(nb, b)
            off = ((n8 // 8) * b0 + g * kb + (b - b0)) * 1152
            seen.add(off)
            for rr in range(8):
                r = 8 * g + rr
                got = p[off + 144 * rr:off + 144 * (rr + 1)]
                if r >= n:
                    assert not np.any(got)
                else:
                    assert np.array_equal(got, blocks[r, b])
    assert len(seen) == (n8 // 8) * nb


@pytest.mark.parametrize("n,k", SMALL + [(6144, 1024), (9216, 2560)])
def test_gemv_q4k_planar_matches_raw_and_oracle(n, k):
    """The model's Q4_K GEMV path (planar layout) inside the oracle's error
    bound, and bitwise equal to the raw-layout building block (the same
    arithmetic in the same order, only the bytes' placement differs)."""
    t = synth.q4k_tensor(synth.subseed(synth.MASTER_SEED, f"q4p.{n}.{k}"), n, k)
    x = synth.normal(synth.subseed(synth.MASTER_SEED, f"q4p.x.{k}"), k)
    y = torch.empty(n, dtype=torch.float32, device="cuda")
    qg.qg_gemv_q4k_planar(planar4(t), dev(x), y, n, k)
    torch.cuda.synchronize()
    qg.qg_device_status()
    yp = y.cpu().numpy()
    assert np.array_equal(yp, run_gemv(t, x))
    if n * k <= 4_000_000:
        check_against_oracle(t, x, yp)
