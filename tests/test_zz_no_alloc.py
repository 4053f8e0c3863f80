"""qg_lmhead_argmax_noalloc (workspace in the library's static device memory)
against qg_lmhead_argmax (caller's workspace) through the C ABI.

The two share the GEMV + argmax kernel, so the token ids must be identical.
Two calls in a row on each input check that the static scratch is left zeroed
(a stale best key or arrival count would change the second answer or never
publish it).  The file sorts last so that it also runs after every other GPU
test in one session; it needs no fixture of theirs and passes alone.
"""
import numpy as np
import pytest

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
    with pytest.raises(qg.QgError):
        qg.qg_lmhead_argmax_noalloc(w, x, 4096, 1000, tok)  # k not a multiple of 256
    with pytest.raises(qg.QgError):
        qg.qg_lmhead_argmax_noalloc(w, x, 0, k, tok)
