"""qg_lmhead_argmax_noalloc (workspace in the library's static device memory)
against qg_lmhead_argmax (caller's workspace) and the CPU oracle, through the
C ABI.

The two entry points share the GEMV + argmax kernel, so their token ids must
be identical; both must give the oracle's first-index argmax of W x.  Two
calls in a row on each input check that the static scratch is left zeroed (a
stale best key or arrival count would change the second answer or never
publish it); a call on x followed by one on -x, whose best logit is lower,
checks it deterministically.  The file sorts last so that it also runs after
every other GPU test in one session; it needs no fixture of theirs and passes
alone.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
qg = pytest.importorskip("quantized_gemv_gated_gb300")


def _planar(t):
    src = torch.from_numpy(t.data).cuda()
    dst = torch.empty(qg.qg_q6k_planar_bytes(t.n, t.k), dtype=torch.uint8, device="cuda")
    qg.qg_q6k_to_planar(src, dst, t.n, t.k)
    return dst


@pytest.mark.parametrize("n_vocab,k", [(248320, 1024), (50001, 2560)])
def test_noalloc_matches_workspace_entry_point_twice(n_vocab, k):
    t = synth.q6k_tensor(synth.subseed(synth.MASTER_SEED, f"noalloc.{n_vocab}"), n_vocab, k)
    w = _planar(t)
    ws = torch.zeros(qg.qg_lmhead_argmax_workspace_bytes() // 8, dtype=torch.int64, device="cuda")
    for trial in range(2):
        x = torch.from_numpy(synth.normal(synth.subseed(synth.MASTER_SEED, f"noalloc.x{trial}"), k)).cuda()
        ref = torch.zeros(1, dtype=torch.int32, device="cuda")
        qg.qg_lmhead_argmax(w, x, n_vocab, k, ws, ref)
        got = []
        for _ in range(2):  # two calls in a row on the same input
            tok = torch.full((1,), -1, dtype=torch.int32, device="cuda")
            qg.qg_lmhead_argmax_noalloc(w, x, n_vocab, k, tok)
            torch.cuda.synchronize()
            got.append(int(tok.item()))
        assert got == [int(ref.item())] * 2, f"trial {trial}: {got} vs {int(ref.item())}"
        logits = oracle.gemv(t, x.cpu().numpy())
        a, b = oracle.top2(logits)
        if a - b > 1e-4 * abs(a):  # a clear winner: the GPU's f32 sums cannot reorder it
            assert got[0] == oracle.argmax(logits)
        else:  # near tie: the GPU's pick is within the GEMV's rounding of the maximum
            assert logits[got[0]] >= a - 1e-4 * abs(a)
    qg.qg_device_status()


def test_noalloc_after_a_larger_maximum():
    """x and -x, the one with the larger best logit first: the second call's
    best logit is below the first's, so a best key left over in the static
    scratch would win and give the first call's token; the answer must be the
    oracle's argmax of the second input."""
    n_vocab, k = 30000, 1024
    t = synth.q6k_tensor(synth.subseed(synth.MASTER_SEED, "noalloc.neg"), n_vocab, k)
    w = _planar(t)
    xh = synth.normal(synth.subseed(synth.MASTER_SEED, "noalloc.neg.x"), k)
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    runs = []
    for xs in (xh, -xh):
        logits = oracle.gemv(t, xs)
        a, b = oracle.top2(logits)
        assert a - b > 1e-4 * abs(a)  # a clear winner for this seed
        runs.append((a, oracle.argmax(logits), xs))
    runs.sort(key=lambda r: -r[0])  # larger maximum first
    assert runs[1][0] < runs[0][0] and runs[0][1] != runs[1][1]
    for _, expect, xs in runs:
        qg.qg_lmhead_argmax_noalloc(w, torch.from_numpy(xs).cuda(), n_vocab, k, tok)
        torch.cuda.synchronize()
        assert int(tok.item()) == expect
    qg.qg_device_status()


def test_noalloc_planted_tie_and_errors():
    k = 1024
    t = synth.q6k_tensor(synth.subseed(synth.MASTER_SEED, "noalloc.tie"), 4096, k)
    data = t.data.reshape(4096, k // 256, 210).copy()
    data[17, :, 208:210] = np.frombuffer(np.float16(1.0).tobytes(), np.uint8)  # d = 1: row 17 dominates
    data[3000] = data[17]  # row 3000 repeats row 17: an exact tie, the first index must win
    t.data = data.reshape(-1)
    w = _planar(t)
    x = torch.from_numpy(synth.normal(synth.subseed(synth.MASTER_SEED, "noalloc.tie.x"), k)).cuda()
    ws = torch.zeros(2, dtype=torch.int64, device="cuda")
    ref = torch.zeros(1, dtype=torch.int32, device="cuda")
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    seen = []
    for sign in (1.0, -1.0):  # the tied rows lead for one sign of x
        xs = x * sign
        qg.qg_lmhead_argmax(w, xs, 4096, k, ws, ref)
        qg.qg_lmhead_argmax_noalloc(w, xs, 4096, k, tok)
        torch.cuda.synchronize()
        assert int(tok.item()) == int(ref.item())
        seen.append(int(tok.item()))
    assert 17 in seen and 3000 not in seen
    for sign, got in zip((1.0, -1.0), seen):  # the oracle's first-index argmax, where the winner is clear
        logits = oracle.gemv(t, sign * x.cpu().numpy())
        a, b = oracle.top2(logits)
        if got == 17 or a - b > 1e-4 * abs(a):
            assert got == oracle.argmax(logits)
    with pytest.raises(qg.QgError):
        qg.qg_lmhead_argmax_noalloc(w, x, 4096, 1000, tok)  # k not a multiple of 256
    with pytest.raises(qg.QgError):
        qg.qg_lmhead_argmax_noalloc(w, x, 0, k, tok)
    # a token slot that is not 4-byte aligned is refused on the host (no launch)
    slot = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(qg.QgError):
        qg.qg_lmhead_argmax_noalloc(w, x, 4096, k, slot.data_ptr() + 2)
    with pytest.raises(qg.QgError):
        qg.qg_lmhead_argmax(w, x, 4096, k, ws, slot.data_ptr() + 1)
