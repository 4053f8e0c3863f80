#!/usr/bin/env python
"""Batch-1 decode benchmark of the hybrid Gated-DeltaNet / attention model on GB300.

One step = one whole token (every layer, output norm, lm_head + argmax) of
the chosen workload.  Default workload: the 4B-shaped hybrid (32 layers,
850 prompt tokens fed one per step, then greedy tokens), the largest
single-GPU configuration.  Prints ONE JSON line.

  value      tokens/s of the device-resident greedy loop (qg_decode_greedy: one
             CUDA-graph replay per token, token and position stay on the GPU),
             timed with CUDA events on the state's stream, max over ranks.
  e2e        tokens/s through qg_decode_token: per token an 8-byte H2D of
             (token, position) from pinned memory and a 4-byte D2H of the id.
  kernels    every kernel kind of the step timed live with CUDA events: a CUDA
             graph of PDL-chained launches of that exact kernel over the
             model's layers (qg_bench_kernel), per-launch time, algorithmic
             bytes, HBM rate and share of the step (launches per token x time).
  roofline   the kernel with the largest share: algorithmic bytes per launch /
             its CUDA-event duration vs the measured HBM peak.
  cpu_baseline  the CPU oracle on a bounded sample of the same workload, at the
             same positions (the state before them synthetic), all host cores
             and one core.

  python bench.py [--workload 4b|0.8b|4b-long] [--steps K] [--warmup W]
  python bench.py --impl reference ...   (the CPU oracle as the reference arm)
  python bench.py --layer                (one DeltaNet layer step, us per step)
  python bench.py --kernels              (GEMV building blocks, one line per shape)
Multi-GPU: torchrun --nproc-per-node N bench.py --gpus N: N independent
replicas (weak scaling, no collective on the data path).
"""
import argparse
import hashlib
import json
import os
import platform
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "batch-1 decode tok/s and achieved HBM GB/s vs 8 TB/s roofline, 1×GB300"
WORKLOADS = {
    "0.8b": (synth.CFG_0P8B, "random-init 0.8B-shaped hybrid: 24 layers (18 Gated DeltaNet + 6 full attention), "
                             "hidden 1024, FFN 3584, vocab 248320, Q4_K + Q6_K (ffn_down, lm_head); "
                             "850 seeded prompt tokens then greedy decode"),
    "4b": (synth.CFG_4B, "random-init 4B-shaped hybrid: 32 layers (24 Gated DeltaNet + 8 full attention), "
                         "hidden 2560, FFN 9216, vocab 248320, 32 v-heads over 16 k-heads; "
                         "850 seeded prompt tokens then greedy decode"),
    "4b-long": (synth.CFG_4B_LONG, "4B-shaped hybrid, KV cache of 8192 positions prefilled with N(0,1) rows "
                                   "0..7999, greedy decode from position 8000"),
}


KV_FORMATS = {"f32": 0, "q8_0-q5_1": 1}  # qg_state_create_kv formats
KV_DESC = {"f32": "f32 K/V cache", "q8_0-q5_1": "q8_0 K / q5_1 V cache (272 + 192 bytes per position and kv head)"}


def algorithmic_bytes(cfg, t_rows, kv="f32"):
    """HBM bytes one token must move at KV length t_rows (rows read, incl. the
    new one): every weight as stored (Q4_K 144 B / Q6_K 210 B per 256), the f32
    vectors the kernels read, DeltaNet state and conv window read + write, the
    KV rows read plus the K/V row written (f32 rows, or the quantized records
    plus the f32 V row the quantizer reads), the embedding row."""
    H, F = cfg.hidden, cfg.ffn
    q4 = lambda n, k: n * k // 256 * 144  # noqa: E731
    q6 = lambda n, k: n * k // 256 * 210  # noqa: E731
    total = 0
    for kind in cfg.kinds():
        total += 2 * q4(F, H) + q6(H, F) + 2 * H * 4
        if kind == synth.DELTANET:
            total += q4(cfg.conv_dim + 2 * cfg.n_v_heads + cfg.v_dim, H) + q4(H, cfg.v_dim)
            total += cfg.conv_dim * cfg.conv_kernel * 4 + 2 * cfg.n_v_heads * 4 + cfg.head_v_dim * 4
            total += 2 * cfg.n_v_heads * cfg.head_v_dim * cfg.head_k_dim * 4  # state r + w
            total += 2 * cfg.conv_dim * (cfg.conv_kernel - 1) * 4              # window r + w
        else:
            total += q4(2 * cfg.q_dim + 2 * cfg.kv_dim, H) + q4(H, cfg.q_dim) + 2 * cfg.head_dim * 4
            if kv == "f32":
                total += 2 * t_rows * cfg.kv_dim * 4 + 2 * cfg.kv_dim * 4        # KV read + row write
            else:
                rec = cfg.n_kv_heads * (272 + 192)
                total += t_rows * rec + rec + 2 * cfg.kv_dim * 4                 # records r/w, V row w + r
    total += q6(cfg.vocab, H) + H * 4 + H * 4                                   # lm_head, out norm, embed row
    return total


def lmhead_bytes(cfg):
    return cfg.vocab * cfg.hidden // 256 * 210 + cfg.hidden * 4


DTYPE = ("f32 (GEMV: each activation a 24-bit block-fixed-point integer per 256-element block, exact integer "
         "sub-block sums with dp4a, f32 accumulation; norms, recurrences and attention in f32)")

# kernel kinds of the step (qg_bench_kernel): name, launches per token
KERNEL_KINDS = [("dn_in", 0), ("delta", 1), ("ssm_out", 2), ("attn_in", 3), ("attn", 4), ("attn_out", 5),
                ("ffn_up", 6), ("ffn_down", 7), ("lmhead", 8)]


def kernel_bytes(cfg, kind, t_rows, kv="f32"):
    """Algorithmic HBM bytes of one launch of a kernel kind: its weights as
    stored, the state it reads and writes (DeltaNet state and conv window, KV
    rows), the f32 vectors it reads or writes; the same accounting as
    algorithmic_bytes, split by kernel (the per-layer sums add up to it)."""
    H, F = cfg.hidden, cfg.ffn
    q4 = lambda n, k: n * k // 256 * 144  # noqa: E731
    q6 = lambda n, k: n * k // 256 * 210  # noqa: E731
    if kind == "dn_in":
        return (q4(cfg.conv_dim + 2 * cfg.n_v_heads + cfg.v_dim, H) + cfg.conv_dim * cfg.conv_kernel * 4
                + 2 * cfg.conv_dim * (cfg.conv_kernel - 1) * 4 + 2 * cfg.n_v_heads * 4 + H * 4)
    if kind == "delta":
        return 2 * cfg.n_v_heads * cfg.head_v_dim * cfg.head_k_dim * 4
    if kind == "ssm_out":
        return q4(H, cfg.v_dim) + cfg.head_v_dim * 4
    if kind == "attn_in":
        return q4(2 * cfg.q_dim + 2 * cfg.kv_dim, H) + H * 4
    if kind == "attn":
        if kv == "f32":
            return 2 * t_rows * cfg.kv_dim * 4 + 2 * cfg.kv_dim * 4 + 2 * cfg.head_dim * 4
        rec = cfg.n_kv_heads * (272 + 192)
        return t_rows * rec + rec + 2 * cfg.kv_dim * 4 + 2 * cfg.head_dim * 4
    if kind == "attn_out":
        return q4(H, cfg.q_dim)
    if kind == "ffn_up":
        return 2 * q4(F, H) + H * 4
    if kind == "ffn_down":
        return q6(H, F)
    return q6(cfg.vocab, H) + H * 4 + H * 4  # + the output norm and the embedding row


def kernel_launches(cfg, kind):
    """Launches of a kernel kind per token."""
    kinds = cfg.kinds()
    n_dn = sum(1 for k in kinds if k == synth.DELTANET)
    return {"dn_in": n_dn, "delta": n_dn, "ssm_out": n_dn, "attn_in": len(kinds) - n_dn, "attn": len(kinds) - n_dn,
            "attn_out": len(kinds) - n_dn, "ffn_up": len(kinds), "ffn_down": len(kinds), "lmhead": 1}[kind]


def time_kernels(qg, m, cfg, kvf, kv_name, pos, long_ctx, peak, reps=4):
    """Each kernel kind of the step timed with CUDA events: a CUDA graph of
    PDL-chained launches of that kernel over the model's layers (qg_bench_kernel,
    on a separate state brought to the timed position), replayed `reps` times;
    per-launch time = graph time / launches.  Weights rotate over the layers, so
    every launch streams from HBM as in the step (the lm_head's 208-521 MB
    exceed the L2 by themselves)."""
    import torch
    st = qg.State(m, cfg.max_seq_len, kvf)
    prefill_synthetic(qg, st, cfg, pos)
    # one step at `pos`: its position is in the state's device slot, where the
    # attention kernel reads it, so the timed attention covers pos + 1 rows
    qg.qg_decode_token(m, st, int(synth.tokens(synth.subseed(synth.MASTER_SEED, "bench.kernels"), cfg.vocab, 1)[0]),
                       pos)
    stream = torch.cuda.Stream()
    out, total = [], 0.0
    t_rows = pos + 1
    for name, kind in KERNEL_KINDS:
        n_per_tok = kernel_launches(cfg, name)
        if n_per_tok == 0:
            continue
        launches = 4 if name == "lmhead" else max(2 * n_per_tok, 16)
        with torch.cuda.stream(stream):
            qg.qg_bench_kernel(m, st, kind, launches, stream.cuda_stream)  # eager: grants shared memory
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            qg.qg_bench_kernel(m, st, kind, launches, stream.cuda_stream)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        e1.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (reps * launches)
        b = kernel_bytes(cfg, name, t_rows, kv_name)
        gbs = b / us / 1e3
        out.append({"kernel": name, "launches_per_token": n_per_tok, "us_per_launch": round(us, 3),
                    "bytes_per_launch": int(b), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4)})
        total += n_per_tok * us
        del g
    qg.qg_device_status()
    st.close()
    for k in out:
        k["share"] = round(k["launches_per_token"] * k["us_per_launch"] / total, 4)
    return out


def prefill_synthetic(qg, st, cfg, pos):
    """A state at position `pos` with synthetic contents: every attention
    layer's K/V rows 0..pos-1 N(0,1), every DeltaNet window and state
    N(0,0.1) (the same recipe as the long-context workload)."""
    for il, kind in enumerate(cfg.kinds()):
        if kind == synth.DELTANET:
            st.upload_layer(il, *synth.initial_deltanet_state(cfg, il))
        elif pos > 0:
            st.upload_kv(il, *synth.long_context_kv(cfg, il, pos))


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# profiles/traffic.json records ncu DRAM bytes per launch of the step's kernels,
# keyed by kernel kind, with a hash of the CUDA sources they were taken from:
# a record taken from other sources reads as unknown (null).  Translation
# units that compile no decode-step kernel are left out: the batched prefill
# and the standalone building-block entry points with their repacks.
STEP_FREE_SOURCES = ("prefill.cu", "gemv.cu", "gemv_rows.cu")


def kernel_sources_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_gemv_gated_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")) and name not in STEP_FREE_SOURCES:
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode())
                h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or
    None when the counters were taken on other shapes than the workload's or
    the kernel sources changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("sources") != kernel_sources_hash() or workload not in e.get("shapes", ()):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons every 200 ms during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                      stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.p.terminate()
        self.p.wait()
        self.f.seek(0)
        rows = [ln.split(",") for ln in self.f.read().strip().splitlines() if ln.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for nm, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def prefill(qg, m, st, cfg, long_ctx, n_prompt=synth.PROMPT_LEN):
    """Bring a state to the start of the timed decode; returns the next position
    and the token to feed there."""
    if long_ctx:
        for il, kind in enumerate(cfg.kinds()):
            if kind == synth.DELTANET:
                st.upload_layer(il, *synth.initial_deltanet_state(cfg, il))
            else:
                st.upload_kv(il, *synth.long_context_kv(cfg, il, synth.LONG_PREFILL))
        first = int(synth.tokens(synth.subseed(synth.MASTER_SEED, "long.first"), cfg.vocab, 1)[0])
        tok = qg.qg_decode_token(m, st, first, synth.LONG_PREFILL)
        return synth.LONG_PREFILL + 1, tok
    toks = synth.prompt_tokens(cfg, n_prompt)
    tok = 0
    for pos, t in enumerate(toks):
        tok = qg.qg_decode_token(m, st, int(t), pos)
    return len(toks), tok


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.processor() or platform.machine()


def oracle_at(cfg, pos0, kv="f32"):
    """The oracle's model and a state at position pos0 with synthetic contents
    (K/V rows 0..pos0-1 N(0,1), DeltaNet windows and states N(0,0.1)): a token
    at pos0.. then costs what it costs in the decode being timed."""
    import oracle
    w = synth.make_model_weights(cfg)
    om = oracle.Model(w)
    ost = oracle.State(om, KV_FORMATS[kv])
    for il, kind in enumerate(cfg.kinds()):
        if kind == synth.DELTANET:
            c, s_ = synth.initial_deltanet_state(cfg, il)
            ost.conv[il][:] = c
            ost.ssm[il][:] = s_
        elif pos0 > 0:
            ost.set_kv_rows(il, *synth.long_context_kv(cfg, il, pos0))
    ost.kv_len = pos0
    return om, ost


def time_oracle(om, ost, pos0, n_max, budget_s, threads):
    """Tokens per second of oracle.forward_token at positions pos0.. on
    `threads` host threads (0: all), at least one token, stopping when the
    budget is spent."""
    import oracle
    oracle.set_threads(threads if threads else os.cpu_count() or 1)
    tok = int(synth.tokens(synth.subseed(synth.MASTER_SEED, "bench.oracle"), om.cfg.vocab, 1)[0])
    n, t0 = 0, time.perf_counter()
    while n < n_max and (n < 1 or time.perf_counter() - t0 < budget_s):
        tok, _, _ = oracle.forward_token(om, ost, tok, pos0 + n)
        n += 1
    dt = time.perf_counter() - t0
    used = oracle.max_threads()
    oracle.set_threads(os.cpu_count() or 1)
    return n, dt, used


def time_oracle_layer(budget_s, threads):
    """Microseconds per step of the oracle's single DeltaNet layer (the
    one-layer workload: 8 steps, fresh N(0,1) hidden each step)."""
    import oracle
    cfg = synth.CFG_LAYER
    w = synth.make_model_weights(cfg)
    om = oracle.Model(w)
    ost = oracle.State(om)
    c, s_ = synth.initial_deltanet_state(cfg, 0)
    ost.conv[0][:] = c
    ost.ssm[0][:] = s_
    hs = synth.layer_inputs(cfg, 8)
    oracle.set_threads(threads if threads else os.cpu_count() or 1)
    n, t0 = 0, time.perf_counter()
    while n < 8 or time.perf_counter() - t0 < min(budget_s, 2.0):
        oracle.deltanet_layer(om, ost, 0, hs[n % 8])
        n += 1
        if n >= 400:
            break
    dt = time.perf_counter() - t0
    used = oracle.max_threads()
    oracle.set_threads(os.cpu_count() or 1)
    return round(1e6 * dt / n, 1), n, used


def cpu_baseline(cfg, pos0, n_max, kv="f32", budget_s=12.0):
    """The oracle as it stands, on the host cores, on a bounded sample of the
    timed workload: tokens at the GPU arm's positions pos0.. from a synthetic
    state at pos0, on all cores (the value) and on one core; plus the
    one-layer step in microseconds."""
    om, ost = oracle_at(cfg, pos0, kv)
    n, dt, used = time_oracle(om, ost, pos0, n_max, budget_s, 0)
    om1, ost1 = oracle_at(cfg, pos0, kv)
    n1, dt1, _ = time_oracle(om1, ost1, pos0, max(1, min(n_max, 2)), budget_s / 3, 1)
    layer_all, nl, _ = time_oracle_layer(budget_s, 0)
    layer_one, _, _ = time_oracle_layer(budget_s, 1)
    return {"value": round(n / dt, 4), "unit": "tok/s", "cores": used, "kind": "oracle",
            "cpu": cpu_model(), "host_cores": os.cpu_count(),
            "sample": f"{n} tokens at positions {pos0}..{pos0 + n - 1} (the GPU arm's timed positions) by the f32 C "
                      f"oracle with OpenMP over GEMV rows on {used} threads, from a synthetic state at position "
                      f"{pos0} (K/V rows N(0,1), DeltaNet windows and states N(0,0.1)), {dt:.1f} s",
            "single_core": {"value": round(n1 / dt1, 4), "unit": "tok/s", "cores": 1,
                            "sample": f"{n1} tokens at positions {pos0}.., {dt1:.1f} s"},
            "layer_step_us": {"all_cores": layer_all, "one_core": layer_one,
                              "workload": "one Gated DeltaNet layer (hidden 1024, FFN 3072, 16 heads x 128)"}}


def run_ours(args, rank, world, local):
    import torch
    import quantized_gemv_gated_gb300 as qg
    torch.cuda.set_device(local)
    cfg, desc = WORKLOADS[args.workload]
    long_ctx = args.workload == "4b-long"
    K, W = args.steps, args.warmup
    w = synth.make_model_weights(cfg)
    m = qg.Model(w, device=local)
    kvf = KV_FORMATS[args.kv_format]
    st = qg.State(m, cfg.max_seq_len, kvf)
    # warm up (graph capture, clocks), then restart the sequence for the timed run
    pos, _ = prefill(qg, m, st, cfg, long_ctx, args.prompt)
    qg.qg_decode_greedy(m, st, pos, W)
    st.reset()
    pos0, _ = prefill(qg, m, st, cfg, long_ctx, args.prompt)
    assert pos0 + K <= cfg.max_seq_len, "steps exceed the KV cache"
    ext = torch.cuda.ExternalStream(st.stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    clk = ClockSampler(local)
    e0.record(ext)
    toks = qg.qg_decode_greedy(m, st, pos0, K)
    e1.record(ext)
    e1.synchronize()
    torch.cuda.synchronize()
    clocks = clk.stop()
    barrier(world)
    dt = max_over_ranks(e0.elapsed_time(e1) / 1000.0, world)
    stats = st.stats()
    nodes = stats["graph_kernel_nodes"]

    # e2e: the host API, one decode_token per step on a second state
    dt2 = None
    if not args.no_e2e:
        st2 = qg.State(m, cfg.max_seq_len, kvf)
        p2, tok = prefill(qg, m, st2, cfg, long_ctx, args.prompt)
        ext2 = torch.cuda.ExternalStream(st2.stream)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        f0.record(ext2)
        for i in range(K):
            tok = qg.qg_decode_token(m, st2, tok, p2 + i)
        f1.record(ext2)
        f1.synchronize()
        dt2 = max_over_ranks(f0.elapsed_time(f1) / 1000.0, world)
        st2.close()

    peak, peak_kind = measured_peaks()
    tokps = world * K / dt
    mean_t = pos0 + (K + 1) / 2.0  # KV rows read, averaged over the timed steps
    bpt = algorithmic_bytes(cfg, mean_t, args.kv_format)
    step_gbs = bpt * K / dt / 1e9 * world
    # every kernel kind of the step, timed with CUDA events (PDL-chained graphs
    # of that kernel over the layers); the largest share is the roofline kernel
    kernels = time_kernels(qg, m, cfg, kvf, args.kv_format, pos0 + K // 2, long_ctx, peak)
    dom = max(kernels, key=lambda k: k["share"])
    lm = next(k for k in kernels if k["kernel"] == "lmhead")
    out = {
        "metric": METRIC, "value": round(tokps, 3), "unit": "tok/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(1000.0 * dt / K, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE, "data": "synthetic (seeded random-init weights and prompt)",
        "config": {"workload": f"{args.workload}: {desc}", "global_batch": world, "seq_len": cfg.max_seq_len,
                   "parallelism": f"replicas x{world}",
                   "kv_cache": KV_DESC[args.kv_format], "prompt_tokens": pos0, "timed_positions": [pos0, pos0 + K - 1],
                   "l2": f"no flush: {bpt / 1e6:.1f} MB of weights and state per token > 129 MB L2",
                   "greedy_tokens_head": [int(t) for t in toks[:4]]},
        "bytes_per_token": int(bpt),
        "step_roofline": {"achieved": round(step_gbs / world, 1), "peak": peak, "unit": "GB/s",
                          "frac": round(step_gbs / world / peak, 4), "peak_kind": peak_kind},
        "roofline": {"bound": "hbm", "kernel": dom["kernel"], "achieved": dom["GB/s"], "peak": peak, "unit": "GB/s",
                     "frac": dom["frac"], "traffic": ncu_traffic(dom["kernel"], args.workload),
                     "bytes_per_launch": dom["bytes_per_launch"], "launch_us": dom["us_per_launch"],
                     "share_of_step": dom["share"], "peak_kind": peak_kind,
                     "how": "CUDA events around a graph of PDL-chained launches of this kernel over the model's "
                            "layers (qg_bench_kernel), on the launching stream"},
        "roofline_lmhead": {"achieved": lm["GB/s"], "frac": lm["frac"], "launch_us": lm["us_per_launch"],
                            "bytes_per_launch": lm["bytes_per_launch"], "traffic": ncu_traffic("lmhead", args.workload)},
        "kernels": kernels,
        "clocks": clocks,
        "e2e": ({"value": round(world * K / dt2, 3), "unit": "tok/s", "h2d_bytes_per_step": 8,
                 "d2h_bytes_per_step": 4} if dt2 else None),
        "gpu_launches": int(nodes * K),
        "kernels_per_token": int(nodes),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(cfg, pos0, K, kv=args.kv_format)
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: the workload's decode timed at the
    positions the GPU arm times (pos0.. after the prompt, or 8000.. for the
    long context), from a synthetic state at pos0, on all host cores; K steps
    of a bounded sample after W warm-up tokens."""
    if rank != 0:
        return
    cfg, desc = WORKLOADS[args.workload]
    K, W = args.steps, args.warmup
    pos0 = synth.LONG_PREFILL + 1 if args.workload == "4b-long" else args.prompt
    om, ost = oracle_at(cfg, pos0 - W, args.kv_format)
    time_oracle(om, ost, pos0 - W, W, 1e9, 0)  # warm-up tokens at pos0 - W .. pos0 - 1
    n, dt, used = time_oracle(om, ost, pos0, K, 1e9, 0)
    v = round(n / dt, 4)
    sample = (f"{n} tokens at positions {pos0}..{pos0 + n - 1} (the GPU arm's timed positions) by the f32 C oracle "
              f"with OpenMP over GEMV rows on {used} threads, after {W} warm-up tokens, from a synthetic state "
              f"(K/V rows N(0,1), DeltaNet windows and states N(0,0.1))")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tok/s", "n_gpus": world, "steps": n,
        "warmup": W, "ms_per_step": round(1000.0 * dt / n, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded random-init weights and prompt)",
        "config": {"workload": f"{args.workload}: {desc}", "global_batch": 1, "seq_len": cfg.max_seq_len,
                   "kv_cache": KV_DESC[args.kv_format], "timed_positions": [pos0, pos0 + n - 1]},
        "cpu_baseline": {"value": v, "unit": "tok/s", "cores": used, "kind": "oracle", "cpu": cpu_model(),
                         "host_cores": os.cpu_count(), "sample": sample},
        "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_layer(args):
    """One JSON line: the one-layer workload (one Gated DeltaNet layer,
    hidden 1024, FFN 3072, 16 heads x 128, 8 steps from seeded state) through
    qg_deltanet_step, microseconds per step (CUDA events around a graph of the
    steps on one stream, each step on a fresh N(0,1) hidden), against the
    oracle's layer step on all host cores and on one."""
    import torch
    import quantized_gemv_gated_gb300 as qg
    cfg = synth.CFG_LAYER
    w = synth.make_model_weights(cfg)
    m = qg.Model(w)
    st = qg.State(m, cfg.max_seq_len)
    st.upload_layer(0, *synth.initial_deltanet_state(cfg, 0))
    hs = torch.from_numpy(synth.layer_inputs(cfg, 8)).cuda()
    hbuf = torch.empty(cfg.hidden, device="cuda")
    stream = torch.cuda.Stream()
    n_steps = 8
    with torch.cuda.stream(stream):
        for i in range(n_steps):
            hbuf.copy_(hs[i])
            qg.qg_deltanet_step(m, st, 0, hbuf, stream.cuda_stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n_steps):
            hbuf.copy_(hs[i])
            qg.qg_deltanet_step(m, st, 0, hbuf, stream.cuda_stream)
    reps = max(4, args.steps // 8)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    qg.qg_device_status()
    us = e0.elapsed_time(e1) * 1e3 / (reps * n_steps)
    q4 = lambda n, k: n * k // 256 * 144  # noqa: E731
    H, F = cfg.hidden, cfg.ffn
    b = (kernel_bytes(cfg, "dn_in", 0) + kernel_bytes(cfg, "delta", 0) + kernel_bytes(cfg, "ssm_out", 0)
         + kernel_bytes(cfg, "ffn_up", 0) + kernel_bytes(cfg, "ffn_down", 0))
    peak, peak_kind = measured_peaks()
    line = {"mode": "layer", "workload": "one Gated DeltaNet layer, hidden 1024, FFN 3072, 16 k-heads / 16 v-heads "
                                         "x 128, conv 4, 8 steps from seeded state",
            "us_per_step": round(us, 3), "bytes_per_step": int(b), "GB/s": round(b / us / 1e3, 1),
            "frac": round(b / us / 1e3 / peak, 4), "peak_kind": peak_kind,
            "how": "CUDA events around a graph of 8 qg_deltanet_step calls (5 layer kernels + the residual add each)"}
    if not args.no_cpu_baseline:
        a, n, used = time_oracle_layer(10.0, 0)
        one, _, _ = time_oracle_layer(10.0, 1)
        line["cpu_baseline"] = {"us_per_step": a, "cores": used, "one_core_us_per_step": one, "cpu": cpu_model(),
                                "kind": "oracle", "sample": f"{n} layer steps"}
    del q4, H, F
    print(json.dumps(line), flush=True)


def run_prefill(args):
    """One JSON line: the workload's seeded prompt prefilled in one qg_prefill
    call (timed with CUDA events on the state's stream, the state reset
    between runs outside the timed region) against the same prompt decoded
    token by token (one captured-graph step per token), and the FLOP rate of
    the prefill's projections (2 x the projection weights x tokens)."""
    import torch
    import quantized_gemv_gated_gb300 as qg
    cfg, desc = WORKLOADS[args.workload]
    w = synth.make_model_weights(cfg)
    m = qg.Model(w)
    kvf = KV_FORMATS[args.kv_format]
    st = qg.State(m, cfg.max_seq_len, kvf)
    toks = synth.prompt_tokens(cfg, args.prompt)
    n = len(toks)
    ext = torch.cuda.ExternalStream(st.stream)
    first = None
    for _ in range(max(1, args.warmup)):
        st.reset()
        first = qg.qg_prefill(m, st, toks)
    times = []
    for _ in range(max(1, args.steps // 16)):
        st.reset()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(ext)
        tok = qg.qg_prefill(m, st, toks)
        e1.record(ext)
        e1.synchronize()
        times.append(e0.elapsed_time(e1) / 1000.0)
        assert tok == first
    t_pf = sorted(times)[len(times) // 2]
    # token by token through the decode step
    st.reset()
    qg.qg_decode_token(m, st, int(toks[0]), 0)
    st.reset()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(ext)
    for pos, t in enumerate(toks):
        tok2 = qg.qg_decode_token(m, st, int(t), pos)
    f1.record(ext)
    f1.synchronize()
    t_tw = f0.elapsed_time(f1) / 1000.0
    qg.qg_device_status()
    H, F = cfg.hidden, cfg.ffn
    params = 0
    for kind in cfg.kinds():
        params += 3 * F * H
        if kind == synth.DELTANET:
            params += (cfg.conv_dim + 2 * cfg.n_v_heads + cfg.v_dim) * H + H * cfg.v_dim
        else:
            params += (2 * cfg.q_dim + 2 * cfg.kv_dim) * H + H * cfg.q_dim
    flops = 2.0 * params * n
    print(json.dumps({
        "mode": "prefill", "workload": f"{args.workload}: {desc}", "kv_cache": KV_DESC[args.kv_format],
        "prompt_tokens": n, "prefill_ms": round(t_pf * 1e3, 3), "prefill_tok_s": round(n / t_pf, 1),
        "tokenwise_ms": round(t_tw * 1e3, 3), "tokenwise_tok_s": round(n / t_tw, 1),
        "speedup": round(t_tw / t_pf, 2), "projection_tflops": round(flops / t_pf / 1e12, 2),
        "same_first_token": bool(tok == tok2), "runs": len(times),
        "arith": "tcgen05.mma on a three-way bf16 split (hi, mid, lo: 6 products per K step), f32 accumulators in tensor memory; Q4_K/Q6_K dequantized into shared-memory tiles",
    }), flush=True)


def run_batch(args):
    """One JSON line: --batch B sequences decoded in lockstep (qg_batch_step:
    the step as one captured graph),
    each prefilled with its own seeded prompt, for K steps (the synchronous
    calls timed by CUDA events on the first state's stream, host copies of the
    B tokens and positions included), against one sequence through the
    captured single-sequence step over the same K steps."""
    import torch
    import quantized_gemv_gated_gb300 as qg
    cfg, desc = WORKLOADS[args.workload]
    B, K = args.batch, args.steps
    w = synth.make_model_weights(cfg)
    m = qg.Model(w)
    kvf = KV_FORMATS[args.kv_format]
    states = [qg.State(m, cfg.max_seq_len, kvf) for _ in range(B)]

    def prefill_all():
        toks, pos = [], []
        for i, st in enumerate(states):
            st.reset()
            prompt = synth.tokens(synth.subseed(synth.MASTER_SEED, f"batch.bench.{i}"), cfg.vocab, args.prompt)
            toks.append(qg.qg_prefill(m, st, prompt))
            pos.append(len(prompt))
        return toks, pos

    bt = qg.Batch(m, states)  # one captured graph per step (qg_batch_step)
    toks, pos = prefill_all()
    for _ in range(args.warmup):
        toks = bt.step(toks, pos)
        pos = [p + 1 for p in pos]
    toks, pos = prefill_all()
    assert pos[0] + K <= cfg.max_seq_len
    ext = torch.cuda.ExternalStream(states[0].stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(ext)
    for _ in range(K):
        toks = bt.step(toks, pos)
        pos = [p + 1 for p in pos]
    e1.record(ext)
    e1.synchronize()
    dt = e0.elapsed_time(e1) / 1000.0
    bt.close()
    # one sequence through the captured single-sequence step
    one = states[0]
    one.reset()
    prompt = synth.tokens(synth.subseed(synth.MASTER_SEED, "batch.bench.0"), cfg.vocab, args.prompt)
    t1 = qg.qg_prefill(m, one, prompt)
    p1 = len(prompt)
    t1 = qg.qg_decode_token(m, one, t1, p1)
    ext1 = torch.cuda.ExternalStream(one.stream)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(ext1)
    for i in range(K):
        t1 = qg.qg_decode_token(m, one, t1, p1 + 1 + i)
    f1.record(ext1)
    f1.synchronize()
    d1 = f0.elapsed_time(f1) / 1000.0
    qg.qg_device_status()
    print(json.dumps({
        "mode": "batch", "workload": f"{args.workload}: {desc}", "kv_cache": KV_DESC[args.kv_format],
        "sequences": B, "steps": K, "prompt_tokens_each": args.prompt,
        "batch_tok_s": round(B * K / dt, 1), "batch_ms_per_step": round(1e3 * dt / K, 3),
        "single_tok_s": round(K / d1, 1), "single_ms_per_step": round(1e3 * d1 / K, 3),
        "ratio": round((B * K / dt) / (K / d1), 2),
        "path": ("small-batch GEMV (4 multiply-adds per weight read)" if B <= 4 else
                 "small-batch GEMV per group of 4 sequences" if B <= 8 else "prefill tensor-core GEMM tiles"),
    }), flush=True)


# GEMV shapes of the kernel mode: the building blocks at the model's shapes
# (planar layouts, the layers' own path), lm_head with its fused argmax, and
# the Q6_K GEMV on raw rows.
KERNEL_SHAPES = [
    ("q4k", 1024, 1024), ("q4k", 6144, 1024), ("q4k", 8224, 1024), ("q4k", 7168, 1024),
    ("q4k", 12352, 2560), ("q4k", 9216, 2560), ("q6k", 1024, 3584), ("q6k", 2560, 9216),
    ("lmhead", 248320, 1024), ("lmhead", 248320, 2560),
    ("q6k-rows", 2560, 9216), ("q6k-rows", 248320, 2560),  # qg_gemv_q6k on raw GGUF rows
]


def run_kernels(args):
    """One JSON line per GEMV shape: device time per launch in a graph of
    back-to-back launches (chained by programmatic dependent launch, as in the
    decode step) that rotate through enough weight copies to exceed 3x the
    129 MB L2, so every launch streams its weights from HBM."""
    import torch
    import quantized_gemv_gated_gb300 as qg
    peak, peak_kind = measured_peaks()
    stream = torch.cuda.Stream()
    shapes = KERNEL_SHAPES
    if args.shape:
        shapes = [sh for sh in KERNEL_SHAPES if f"{sh[0]}:{sh[1]}x{sh[2]}" in args.shape]
        if len(shapes) != len(set(args.shape)):
            raise SystemExit(f"--shape: not among {[f'{a}:{b}x{c}' for a, b, c in KERNEL_SHAPES]}")
    for kind, n, k in shapes:
        make = synth.q4k_tensor if kind == "q4k" else synth.q6k_tensor
        t = make(synth.subseed(synth.MASTER_SEED, f"kernel.{kind}.{n}.{k}"), n, k)
        src = torch.from_numpy(t.data).cuda()
        rows = kind == "q6k-rows"
        nbytes = t.data.size if rows else (qg.qg_q4k_planar_bytes if kind == "q4k" else qg.qg_q6k_planar_bytes)(n, k)
        copies = max(2, -(-3 * 129 * 2 ** 20 // nbytes))
        ws = []
        for _ in range(copies):
            if rows:
                ws.append(src.clone())
                continue
            w = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
            (qg.qg_q4k_to_planar if kind == "q4k" else qg.qg_q6k_to_planar)(src, w, n, k)
            ws.append(w)
        del src
        x = torch.from_numpy(synth.normal(synth.subseed(synth.MASTER_SEED, f"kernel.x.{k}"), k)).cuda()
        y = torch.empty(n, dtype=torch.float32, device="cuda")
        tok = torch.zeros(1, dtype=torch.int32, device="cuda")
        wsp = torch.zeros(2, dtype=torch.int64, device="cuda")

        def launch(w, st):
            if kind == "q4k":
                qg.qg_gemv_q4k_planar(w, x, y, n, k, st)
            elif kind == "q6k":
                qg.qg_gemv_q6k_planar(w, x, y, n, k, st)
            elif rows:
                qg.qg_gemv_q6k(w, x, y, n, k, st)
            else:
                qg.qg_lmhead_argmax(w, x, n, k, wsp, tok, st)

        with torch.cuda.stream(stream):
            for w in ws[:3]:
                launch(w, stream.cuda_stream)  # eager first launches set the kernels' attributes
        stream.synchronize()
        reps = max(copies, 64)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for r in range(reps):
                launch(ws[r % copies], stream.cuda_stream)
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(max(1, args.steps // 16)):
                g.replay()
            e1.record(stream)
        e1.synchronize()
        qg.qg_device_status()
        us = e0.elapsed_time(e1) * 1e3 / (max(1, args.steps // 16) * reps)
        algo = nbytes + 4 * k + (4 if kind == "lmhead" else 4 * n)
        gbs = algo / us / 1e3
        print(json.dumps({"kernel": f"{kind} {n}x{k}",
                          "layout": "raw GGUF rows" if rows else "planar (grouped, slice-major)",
                          "us_per_launch": round(us, 3), "bytes_per_launch": algo, "GB/s": round(gbs, 1),
                          "frac_of_peak": round(gbs / peak, 4), "peak_GB/s": peak, "peak_kind": peak_kind,
                          "weight_copies": copies, "launches_per_graph": reps}), flush=True)
        del ws, g
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="4b")
    ap.add_argument("--prompt", type=int, default=synth.PROMPT_LEN,
                    help="prompt tokens fed before the timed decode (default 850)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kv-format", choices=sorted(KV_FORMATS), default="f32",
                    help="KV cache format of the decode state (and of the oracle's, on the reference arm)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-API (e2e) measurement")
    ap.add_argument("--batch", type=int, default=0,
                    help="decode this many sequences in lockstep (qg_decode_batch) against one sequence (one JSON line)")
    ap.add_argument("--prefill", action="store_true",
                    help="time qg_prefill of the workload's prompt against token-by-token decode (one JSON line)")
    ap.add_argument("--kernels", action="store_true",
                    help="instead of the decode step: one JSON line per GEMV building block at the model's shapes")
    ap.add_argument("--shape", action="append", default=None, metavar="KIND:NxK",
                    help="with --kernels: only these shapes (e.g. q6k-rows:248320x2560); repeatable")
    ap.add_argument("--layer", action="store_true",
                    help="the one-layer workload through qg_deltanet_step: us per step (one JSON line)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.layer:
        run_layer(args)
        return
    if args.kernels:
        run_kernels(args)
        return
    if args.prefill:
        run_prefill(args)
        return
    if args.batch:
        run_batch(args)
        return
    rank, world, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
