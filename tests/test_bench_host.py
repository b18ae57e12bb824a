"""Host-side logic of bench.py without a GPU: the multi-GPU replica path
(world size 2 over gloo, max-over-ranks timing, whole-job rate, per-rank
seeds), the algorithmic work model, and the reference arm (the float64
oracle on the host cores) on a toy workload."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [12.0, 20.0][rank]                 # rank 1 is slower
    ms = bench.max_over_ranks(local_ms, dist)
    rate = bench.whole_job_rate(world, 288, 10, ms / 1e3)
    dist.barrier()
    q.put((rank, ms, rate, bench.replica_seed(rank)))
    dist.destroy_process_group()


def test_replicas_world_size_two_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, rate, seed in res:
        assert ms == 20.0                          # every rank reports the slowest rank's time
        assert rate == pytest.approx(2 * 288 * 10 / 0.020)
    assert res[0][3] != res[1][3]                  # independent requests per replica


def test_single_process_rate():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_rate(1, 288, 20, 2.0) == pytest.approx(2880.0)


def test_work_model_counts_weights_once_and_scales_with_rows():
    cfg = synth.CONFIGS["1.5b"]
    w0 = bench.layer_work(cfg, 0)
    w50 = bench.layer_work(cfg, 50)
    # weight bytes of one layer appear exactly once across the GEMM families
    wb = sum(w0[f]["bytes"] for f in ("gemm_qkv", "gemm_gateup", "gemm_down")) + cfg.n_q_heads * 128 * cfg.d_model * 2
    assert bench.weight_bytes(cfg) / cfg.n_layers == pytest.approx(wb, rel=1e-9)
    assert w50["gemm_gateup"]["flops"] == pytest.approx(2 * 50 * 2 * cfg.d_model * cfg.d_ffn)
    assert w0["gemm_qkv"]["flops"] == 0
    assert bench.pass_work(cfg, [50] * cfg.n_layers)["flops"] > bench.pass_work(cfg, [10] * cfg.n_layers)["flops"]


def test_reference_arm_runs_the_oracle_on_a_toy_config():
    synth.CONFIGS["_toy"] = synth.small_config(name="toy", n_layers=2)
    try:
        r = subprocess.run([sys.executable, "-c",
                            "import sys, synth, bench; synth.CONFIGS['_toy'] = synth.small_config(name='toy', n_layers=2); "
                            "sys.argv = ['bench.py', '--impl', 'reference', '--config', '_toy', '--steps', '2', '--warmup', '1']; "
                            "bench.main()"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    finally:
        synth.CONFIGS.pop("_toy", None)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == bench.UNIT
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
