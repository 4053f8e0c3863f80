"""Write the oracle's expected token streams for the model workloads.

TEST INFRASTRUCTURE: calls only the CPU oracle (and the seeded input
generator).  For each workload it records, per step, the oracle's argmax token
(first index on ties), the top-1 logit and the top-1 minus top-2 margin, and
the final residual stream at a few sampled steps (base64 f32), into
tests/golden/stream_<workload>.json.

  0.8b / 4b : 850 seeded prompt tokens fed at positions 0..849, then 128
              greedy tokens (each step's input = the previous step's argmax).
  0.8b-varied: the 0.8b workload with every quantized matrix's d / dmin
              drawn below 5e-5 instead of 0.02: the residual stream stays
              near unit scale, so the argmax follows the token (at 0.02 one
              token wins every step by a margin of ~50 logits).
  4b-varied : the same for the 4b workload.
  4b-long   : every attention layer's K/V rows 0..7999 ~ N(0,1), DeltaNet
              windows and states ~ N(0,0.1), a seeded first token at
              position 8000, then 63 greedy tokens (64 steps in all).

  python oracle/make_golden.py 0.8b [0.8b-varied 4b 4b-varied 4b-long] [--threads N]
"""
import argparse
import base64
import json
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

GOLDEN = os.path.join(ROOT, "tests", "golden")
CFGS = {"0.8b": synth.CFG_0P8B, "0.8b-varied": synth.CFG_0P8B, "4b": synth.CFG_4B, "4b-varied": synth.CFG_4B,
        "4b-long": synth.CFG_4B_LONG}
DMAX = {"0.8b-varied": 5e-5, "4b-varied": 5e-5}  # quantized-scale bound per workload (default 0.02)


def b64(a):
    return base64.b64encode(np.ascontiguousarray(a, np.float32).tobytes()).decode()


def run(name, log=print):
    cfg = CFGS[name]
    w = synth.make_model_weights(cfg, dmax=DMAX.get(name, 0.02))
    om = oracle.Model(w)
    st = oracle.State(om)
    steps = []  # (pos, input token)
    if name == "4b-long":
        for il, kind in enumerate(cfg.kinds()):
            if kind == synth.DELTANET:
                c, s = synth.initial_deltanet_state(cfg, il)
                st.conv[il][:] = c
                st.ssm[il][:] = s
            else:
                k, v = synth.long_context_kv(cfg, il, synth.LONG_PREFILL)
                st.kc[il][:synth.LONG_PREFILL] = k
                st.vc[il][:synth.LONG_PREFILL] = v
        st.kv_len = synth.LONG_PREFILL
        first = int(synth.tokens(synth.subseed(synth.MASTER_SEED, "long.first"), cfg.vocab, 1)[0])
        start, n_prompt, n_greedy = synth.LONG_PREFILL, 1, synth.LONG_DECODE - 1
        prompt = [first]
        sample = {start, start + 1, start + 31, start + n_greedy}
    else:
        prompt = [int(t) for t in synth.prompt_tokens(cfg)]
        start, n_prompt, n_greedy = 0, len(prompt), synth.DECODE_LEN
        sample = {0, 1, n_prompt - 1, n_prompt, n_prompt + n_greedy - 1}
    out_tok, top1, margin, hidden = [], [], [], {}
    t0 = time.time()
    tok = None
    for i in range(n_prompt + n_greedy):
        pos = start + i
        inp = prompt[i] if i < n_prompt else tok
        tok, h, logits = oracle.forward_token(om, st, inp, pos, want_logits=True)
        a, b = oracle.top2(logits)
        out_tok.append(int(tok))
        top1.append(float(a))
        margin.append(float(a - b))
        if pos in sample:
            hidden[str(pos)] = b64(h)
        if i % 50 == 0:
            log(f"{name}: step {i}/{n_prompt + n_greedy} ({time.time() - t0:.0f} s)")
    doc = {
        "source": "written by oracle/make_golden.py from the CPU oracle (f32, natural-order accumulation) on the "
                  "seeded synthetic workload; master seed 0x5147",
        "workload": name, "config": cfg.as_dict(), "dmax": DMAX.get(name, 0.02), "start_pos": start, "n_prompt": n_prompt,
        "n_greedy": n_greedy, "prompt": prompt, "tokens": out_tok, "top1": top1, "margin": margin,
        "hidden": hidden, "oracle_threads": oracle.max_threads(), "seconds": round(time.time() - t0, 1),
    }
    path = os.path.join(GOLDEN, f"stream_{name}.json")
    with open(path, "w") as f:
        json.dump(doc, f)
    log(f"{name}: wrote {path} in {time.time() - t0:.0f} s")
    return path


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("workloads", nargs="+", choices=sorted(CFGS))
    ap.add_argument("--threads", type=int, default=0)
    args = ap.parse_args()
    if args.threads:
        oracle.set_threads(args.threads)
    for name in args.workloads:
        run(name, log=lambda m: print(m, flush=True))
