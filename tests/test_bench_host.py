"""Host logic of bench.py without a GPU: the replica timing reduction over
ranks (gloo, world size 2), the per-token byte count, and the reference arm's
JSON line (the CPU oracle), including under torchrun with two ranks where
only rank 0 prints."""
import json
import os
import subprocess
import sys

import pytest

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402
import synth  # noqa: E402


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.max_over_ranks(1.5 + rank, world)
    bench.barrier(world)
    q.put((rank, t))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert res == [(0, 2.5), (1, 2.5)]


def test_bytes_per_token_closed_forms():
    # 0.8B: 553.63 MB fixed + 24,576 B per KV row read; 4B: 2,833.0 MB + 65,536 B
    c8, c4 = synth.CFG_0P8B, synth.CFG_4B
    assert bench.algorithmic_bytes(c8, 1) - bench.algorithmic_bytes(c8, 0) == 6 * 2 * 2 * 256 * 4
    assert bench.algorithmic_bytes(c4, 1) - bench.algorithmic_bytes(c4, 0) == 8 * 2 * 4 * 256 * 4
    assert abs(bench.algorithmic_bytes(c8, 0) / 1e6 - 553.63) < 0.01
    assert abs(bench.algorithmic_bytes(c4, 0) / 1e6 - 2833.03) < 0.01
    assert bench.lmhead_bytes(c8) == 248320 * 1024 // 256 * 210 + 1024 * 4


@pytest.mark.slow
def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "0.8b",
                          "--steps", "2", "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tok/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    # timed at the GPU arm's positions: right after the 850-token prompt
    assert d["config"]["timed_positions"] == [850, 851] and d["steps"] == 2
    assert d["cpu_baseline"]["cpu"] and d["cpu_baseline"]["cores"] >= 1


@pytest.mark.slow
def test_reference_arm_torchrun_world2_rank0_prints_only():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(29700 + os.getpid() % 200),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "0.8b", "--gpus", "2", "--steps", "2",
           "--warmup", "3"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1 and json.loads(lines[0])["n_gpus"] == 2


def test_kernel_bytes_add_up_to_the_token():
    """The per-kernel byte counts of the roofline, times their launches per
    token, add up to the whole token's algorithmic bytes."""
    for cfg in (synth.CFG_0P8B, synth.CFG_4B, synth.CFG_TINY):
        for kv in ("f32", "q8_0-q5_1"):
            for t in (1, 900):
                tot = sum(bench.kernel_launches(cfg, k) * bench.kernel_bytes(cfg, k, t, kv)
                          for k, _ in bench.KERNEL_KINDS)
                assert tot == bench.algorithmic_bytes(cfg, t, kv)
    assert [k for k, _ in bench.KERNEL_KINDS][-1] == "lmhead"


def test_byte_model_of_the_kv_formats():
    """Per token at KV length t, an attention layer moves 2 t kvd f32 values
    plus the new row (f32 cache), or t n_kv (272 + 192) bytes of records, the
    new row's records and its f32 V row written then read (quantized cache);
    everything else is the same."""
    import bench
    import synth
    cfg = synth.CFG_4B_LONG
    n_attn = sum(1 for k in cfg.kinds() if k == synth.ATTENTION)
    for t in (1, 8000):
        f = bench.algorithmic_bytes(cfg, t)
        q = bench.algorithmic_bytes(cfg, t, "q8_0-q5_1")
        per_f = 2 * t * cfg.kv_dim * 4 + 2 * cfg.kv_dim * 4
        per_q = t * cfg.n_kv_heads * 464 + cfg.n_kv_heads * 464 + 2 * cfg.kv_dim * 4
        assert f - q == n_attn * (per_f - per_q)
    assert bench.KV_FORMATS == {"f32": 0, "q8_0-q5_1": 1}


def test_bench_modes_are_registered():
    import subprocess
    import sys
    out = subprocess.run([sys.executable, "bench.py", "--help"], capture_output=True, text=True, timeout=120,
                         cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    assert out.returncode == 0
    for flag in ("--kv-format", "--prefill", "--batch", "--kernels", "--impl", "--layer"):
        assert flag in out.stdout


def test_traffic_records_apply_to_their_shapes_only():
    """ncu DRAM bytes are reported only for the shapes they were captured on
    (the 4B projections, shared by the 4b and 4b-long workloads) and only
    while the step kernels' sources are those of the capture."""
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        records = json.load(f)
    for kind in ("ffn_up", "ffn_down", "dn_in", "ssm_out", "delta", "lmhead"):
        e = records[kind]
        fresh = e["sources"] == bench.kernel_sources_hash()
        assert bench.ncu_traffic(kind, "4b") == (e["dram_bytes_read"] + e["dram_bytes_write"] if fresh else None)
        assert bench.ncu_traffic(kind, "4b-long") == bench.ncu_traffic(kind, "4b")
        assert bench.ncu_traffic(kind, "0.8b") is None
    assert bench.ncu_traffic("no-such-kernel", "4b") is None
