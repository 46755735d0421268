"""CPU checks of bench.py's host logic: the max-over-ranks timing and the
whole-job sum on two gloo ranks, argument rules, and the reference arm."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r processes (r+1)*100 queries in (1+r) seconds
    qps, slowest, total = bench.job_throughput((rank + 1) * 100.0, 1.0 + rank)
    bench.barrier()
    out[rank] = (qps, slowest, total)
    dist.destroy_process_group()


def test_two_rank_timing_reduction():
    import random
    port = 29500 + random.randint(0, 2000)
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for r in (0, 1):
        qps, slowest, total = res[r]
        assert slowest == 2.0 and total == 300.0
        assert qps == pytest.approx(150.0)      # all units over the slowest rank's time


def test_single_process_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_throughput(10.0, 2.0) == (5.0, 2.0, 10.0)


def test_argument_rules():
    sys.path.insert(0, ROOT)
    import bench
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.impl == "ours"
    with pytest.raises(SystemExit):
        bench.parse_args(["--warmup", "2"])


def test_accumulator_names():
    """The accumulator a backward resolves to and the arithmetic dtype the
    bench line reports for it."""
    sys.path.insert(0, ROOT)
    import bench
    r = bench.resolved_accumulator
    assert r("f32", "native", 0) == "fp32_buffer"
    assert r("bf16", "fp16_buffer", 1 << 20) == "fp16_buffer"
    assert r("f16", "fp16_buffer", 0) == "native"
    assert r("bf16", "auto", 0) == "native" and r("bf16", "auto", 64) == "fp32_buffer"
    assert r("bf16", "fp32_buffer", 64) == "fp32_buffer" and r("bf16", "native", 0) == "native"
    d = bench.arithmetic_dtype
    assert d("f32", "fp32_buffer") == "f32" and d("bf16", "fp32_buffer") == "f32"
    assert d("bf16", "fp16_buffer") == "f16" and d("bf16", "native") == "bf16"
    assert set(bench.ACCUM_MODES) == {"fp32_buffer", "native", "auto", "fp16_buffer"}
    assert bench.parse_args(["--accum", "fp16_buffer"]).accum == "fp16_buffer"
    assert bench.parse_args(["--no-accum-lines"]).no_accum_lines
    assert set(bench.LAUNCHES_PER_STEP) == {"fp32_buffer", "native", "fp16_buffer", "f32"}


def test_gather_roofline_counts_one_wavefront_per_corner_line():
    """bf16 D=32 (64-byte head vectors) and fp32 D=32 (128 bytes) take one
    line per corner; fp32 D=64 takes two. Encoder: 5,689,088 samples."""
    sys.path.insert(0, ROOT)
    import bench
    r = bench.gather_roofline(5689088, 32, 2, 0.105, 2070.0, 152)
    assert r["wavefronts_per_launch"] == 4 * 5689088
    assert r["peak"] == 314.6 and abs(r["achieved"] - 4 * 5689088 / 0.105e-3 / 1e9) < 0.1
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    assert bench.gather_roofline(100, 32, 4, 1.0, 2070.0, 152)["wavefronts_per_launch"] == 400
    assert bench.gather_roofline(100, 64, 4, 1.0, 2070.0, 152)["wavefronts_per_launch"] == 800


def test_traffic_figure_needs_matching_kernel_sources(tmp_path):
    sys.path.insert(0, ROOT)
    import bench
    h = bench.kernel_source_hash("msda_backward_kernel")
    assert len(h) == 16 and h != bench.kernel_source_hash("msda_forward_kernel")
    assert bench.profiled_traffic("no_such_kernel") is None


def test_traffic_figure_belongs_to_the_instantiation_run():
    """Each (kernel, dtype, accumulator) reads its own summary: the native
    backward never reports the fp32-workspace kernel's DRAM bytes, fp32 runs
    read the fp32 kernels' lines of their shared summary, and a run with no
    summary (fp16 data) reports none."""
    sys.path.insert(0, ROOT)
    import bench
    files = bench.PROFILE_FILES
    assert files[("msda_backward_kernel", "bf16", "native")] != \
        files[("msda_backward_kernel", "bf16", "fp32_buffer")]
    for k in ("msda_forward_kernel", "msda_backward_kernel"):
        assert bench.profiled_traffic(k, "f16", "native") is None
        f32 = bench.profiled_traffic(k, "f32", "fp32_buffer")
        assert f32 is None or f32 != bench.profiled_traffic(k, "bf16", "fp32_buffer")
    fwd = bench.profiled_traffic("msda_forward_kernel", "f32", "fp32_buffer")
    bwd = bench.profiled_traffic("msda_backward_kernel", "f32", "fp32_buffer")
    assert fwd is None or bwd is None or fwd != bwd
    for (k, _, _), name in files.items():
        assert os.path.exists(os.path.join(ROOT, "profiles", name)), name


def test_reference_arm_prints_its_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["unit"] == "queries/s"


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True,
                       timeout=120, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""
