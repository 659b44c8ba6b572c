"""Multi-process host logic of bench.py on CPU (gloo, world size 2): every
rank runs its own replica, the step time is the slowest rank's, the job
throughput counts every replica, and only rank 0 prints the reference arm."""
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 10.0 + 5.0 * rank                         # rank 1 is the slow one
    slowest = bench.max_over_ranks(ms)
    q.put((rank, slowest, bench.job_tflops(10**12, slowest, world)))
    dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, tf in res:
        assert slowest == 15.0
        assert abs(tf - 2 * 1e12 / 15e-3 / 1e12) < 1e-9   # two replicas' flops over the slowest time


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_tflops(2 * 10**12, 1000.0, 1) == 2.0


def test_reference_arm_prints_on_rank0_only(tmp_path):
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0", "--workload", "q8_0_256x256_t32"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "1", "--workload", "q8_0_256x256_t32"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    import json
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_cpu_sample_takes_the_rows_a_call_has():
    """The CPU baseline's sample asks for 1024 rows of dY; a call with fewer
    (the Q8_0 256x256, T = 32 workload) contributes all of its rows, and the
    one-shot baseline repeats so tiny a sample until a second has passed
    (the reference arm's per-step sample runs once)."""
    import bench
    from quantized_weight_out_gb300 import inputs
    wl = inputs.WORKLOADS["q8_0_256x256_t32"]
    f, dt, desc = bench.oracle_sample(wl, 1024)
    assert f == 2 * 32 * 256 * 256 and "1 pass" in desc
    f, dt, desc = bench.oracle_sample(wl, 1024, min_seconds=0.2)
    assert dt >= 0.2 and f % (2 * 32 * 256 * 256) == 0 and f > 2 * 32 * 256 * 256


def test_peak_follows_the_clock_record():
    """The burst peak for a short region or one without the power cap; the
    sustained peak only for a seconds-long region under sw_power_cap."""
    import bench
    peaks = {"bf16_tflops": 1926.9, "bf16_tflops_sustained": 1715.2, "hbm_gbs": 6800.7}
    assert bench.choose_peak(peaks, {"reasons": []}, 0.06) == (1926.9, "bf16_tflops")
    assert bench.choose_peak(peaks, {"reasons": []}, 5.0) == (1926.9, "bf16_tflops")
    assert bench.choose_peak(peaks, {"reasons": ["sw_power_cap"]}, 0.2)[1] == "bf16_tflops"
    assert bench.choose_peak(peaks, {"reasons": ["sw_power_cap"]}, 3.0) == (1715.2,
                                                                            "bf16_tflops_sustained")
    assert bench.choose_peak(peaks, None, 3.0)[1] == "bf16_tflops"


def test_reference_arm_and_cpu_baseline_share_sample_and_config():
    """Both CPU numbers time the same rows of every call, and the reference
    arm's config is the GPU arm's, key for key."""
    import bench
    from quantized_weight_out_gb300 import inputs
    assert bench.sample_rows(20, 5) == 1024
    assert bench.sample_rows(500, 3) == 64
    r = bench.sample_rows(100, 20)
    assert 64 <= r < 1024 and r % 64 == 0
    wl = inputs.WORKLOADS["layer7b_t8192"]
    c = bench.workload_config("layer7b_t8192", wl, 1)
    assert c["flops_per_step"] == sum(p.flops for p in wl)
    assert "no flush" in c["l2"]
    c1 = bench.workload_config("q8_0_256x256_t32", inputs.WORKLOADS["q8_0_256x256_t32"], 1)
    assert "clean lines" in c1["l2"]
