"""Host allocations of the steady-state decode step, counted below the C ABI.

aprender PR #4332 (counters table) counts host allocations per token with a
counting allocator: 1713 before the change, 0 after.  Here a child process runs
with tests/alloc_count.c preloaded, which counts every malloc-family call on
the calling thread (the library, the C++ runtime and the CUDA runtime and
driver below it), and brackets the step calls of the C ABI with the count:

  - qg_decode_token (one graph replay, 8 bytes in, 4 bytes out) x 20,
  - qg_decode_greedy (20 device-resident steps in one call),

each after a warm-up call (the first call on a state captures the graph).  The
same bracket around 20 calls of qg_state_kv_len (a C-ABI call that touches no
device) gives the Python side's own allocations per call, which are
subtracted.  Both step paths must add no host allocation at all.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

CHILD = r"""
import ctypes, json, sys
sys.path.insert(0, sys.argv[1])
import numpy as np
import synth
import quantized_gemv_gated_gb300 as qg

count = ctypes.CDLL(None).qg_test_thread_allocs
count.restype = ctypes.c_ulonglong
cfg = synth.CFG_TINY
w = synth.make_model_weights(cfg)
m = qg.Model(w)
st = qg.State(m, cfg.max_seq_len)
L = qg.lib()
toks = [int(t) for t in synth.prompt_tokens(cfg, 8)]
out = ctypes.c_uint32()
outp = ctypes.byref(out)
kvl = ctypes.c_int()
kvlp = ctypes.byref(kvl)
mh, sh = m.handle, st.handle
args = [(mh, sh, t, p, outp) for p, t in enumerate(toks)]
n = 20
assert L.qg_decode_token(*args[0]) == 0  # warm-up: captures the graph
# Python-side baseline: the same bracket around a C-ABI call with no device work
c0 = count()
for i in range(n):
    L.qg_state_kv_len(sh, kvlp)
base = count() - c0
# one decode_token per step (positions 1.. of the prompt, then its own tokens)
tok = out.value
c0 = count()
for p in range(1, n + 1):
    L.qg_decode_token(mh, sh, tok, p, outp)
    tok = out.value
per_token = count() - c0
greedy = np.empty(n, np.uint32)
gp = greedy.ctypes.data_as(ctypes.c_void_p)
assert L.qg_decode_greedy(mh, sh, n + 1, 1, gp) == 0  # warm-up of the greedy loop
c0 = count()
rc = L.qg_decode_greedy(mh, sh, n + 2, n, gp)
greedy_allocs = count() - c0
c0 = count()
L.qg_state_kv_len(sh, kvlp)
base1 = count() - c0
print(json.dumps({"baseline_20": base, "decode_token_20": per_token, "greedy_rc": rc,
                  "decode_greedy_20": greedy_allocs, "baseline_1": base1}))
"""


def test_steady_state_step_makes_no_host_allocation(tmp_path):
    so = str(tmp_path / "libqg_alloc_count.so")
    subprocess.run(["gcc", "-O2", "-shared", "-fPIC", os.path.join(HERE, "alloc_count.c"), "-o", so], check=True)
    env = dict(os.environ, LD_PRELOAD=so)
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    print(res)
    assert res["greedy_rc"] == 0
    assert res["decode_token_20"] - res["baseline_20"] <= 0, res
    assert res["decode_greedy_20"] - res["baseline_1"] <= 0, res
