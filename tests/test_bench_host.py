"""Host-side logic of bench.py, without a GPU: the reference arm (the oracle
timed on bounded samples) prints the contract line, and the multi-rank
reduction (max over ranks, whole-job throughput) works over gloo."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "1", "--config", "tiny_b1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "cycles/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["steps"] == 2 and d["warmup"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r = bench.init_dist("gloo")
    t = 1.0 + rank                      # rank 1 is the slower one
    m = bench.max_over_ranks(t)
    v = bench.whole_job_value(100, w, m)
    bench.barrier()
    q.put((rank, m, v))
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, v in res:
        assert m == 2.0                 # the slowest rank's time
        assert v == pytest.approx(100 * 2 / 2.0)


def test_reference_arm_under_two_ranks_prints_only_on_rank_zero():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0", "--config", "tiny_b1"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_lm_head_roofline_picks_the_binding_resource():
    """The LM head is reported against the HBM peak when its bytes take longer
    than its flops (batch 1: 1.2 GB for 20 GFLOP) and against the bf16 tensor
    peak otherwise (batch 32: 637 GFLOP); both fractions are always given."""
    import bench
    from synthetic import CONFIG_BY_NAME
    hbm, tc = (6782.8, "measured"), (1915.7, "measured")
    b1 = bench.lm_head_roofline(CONFIG_BY_NAME["qwen3_8b_b1"], 1_244_791_040, 0.2, hbm, tc, 7)
    assert b1["bound"] == "hbm" and b1["unit"] == "GB/s" and b1["traffic"] == 7
    assert abs(b1["achieved"] - 1_244_791_040 / 0.2e-3 / 1e9) < 1e-9 * b1["achieved"]
    assert b1["frac"] == b1["hbm_frac"] and b1["peak"] == 6782.8
    flops = 2.0 * 32 * 16 * 4096 * 151936
    b32 = bench.lm_head_roofline(CONFIG_BY_NAME["qwen3_8b_b32_paged"], 1_248_862_208, 0.5, hbm,
                                 tc, None)
    assert b32["bound"] == "tensor" and b32["unit"] == "TFLOP/s"
    assert b32["flops_per_launch"] == flops and b32["peak"] == 1915.7
    assert abs(b32["achieved"] - flops / 0.5e-3 / 1e12) < 1e-9 * b32["achieved"]
    assert b32["frac"] == b32["tensor_frac"]
