"""Host-side checks of bench.py without a GPU: the reference arm's JSON line,
and the multi-rank path (replicas: barrier and max-over-ranks timing) as two
gloo ranks on the CPU."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(cmd, env_extra=None, timeout=240):
    env = dict(os.environ)
    env.update(env_extra or {})
    env.setdefault("OMP_NUM_THREADS", "2")
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)


def test_reference_arm_prints_one_json_line():
    r = _run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3",
              "--ref-macs", "2e7"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "gpt_projections_fp32_tf32"
    # the same config keys as the main line
    assert {"tokens", "d_model", "gemms_per_step", "parallelism", "l2"} <= set(d["config"])


def test_reference_arm_under_torchrun_two_ranks():
    r = _run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
              "--master-addr", "127.0.0.1", "--master-port", "29561", "bench.py", "--impl", "reference",
              "--gpus", "2", "--steps", "1", "--warmup", "3", "--ref-macs", "2e7"])
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout  # rank 0 alone prints
    assert json.loads(lines[0])["n_gpus"] == 2


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    t = bench.max_over_ranks(1.0 + rank, world, "cpu")
    out[rank] = t
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, 29562, out), nprocs=world, join=True)
        assert dict(out) == {0: 2.0, 1: 2.0}


def test_sweep_processes_merge_takes_the_median_process():
    """The per-shape result across processes is the median process's record
    (its time, TFLOP/s and fraction together), with every time kept."""
    import bench
    mk = lambda g, ms: {"gemm": g, "ms": ms, "tflops": 1.0 / ms, "roofline_frac": 0.5 / ms}
    runs = [[mk("a", 3.0), mk("b", 1.0)], [mk("a", 1.0), mk("b", 2.0)], [mk("a", 2.0), mk("b", 3.0)]]
    out = bench.merge_process_runs(runs)
    assert [x["gemm"] for x in out] == ["a", "b"]
    assert out[0]["ms"] == 2.0 and out[0]["tflops"] == 0.5 and out[0]["ms_processes"] == [1.0, 2.0, 3.0]
    assert out[1]["ms"] == 2.0 and out[1]["roofline_frac"] == 0.25
    with pytest.raises(ValueError):
        bench.merge_process_runs([[mk("a", 1.0)], [mk("b", 1.0)]])


def test_fp8_sweeps_time_the_k_major_form_against_the_fp8_peak():
    """The FP8 sweeps time B stored N x K (the form the kernels read in
    place, no transpose pass), one byte per operand element, against twice
    the measured bf16 tensor rate (the nominal FP8 / BF16 ratio)."""
    import bench
    for workload in ("large_fp8", "skinny_fp8"):
        cases = bench.sweep_cases(workload)
        assert cases and all(mode == "fp8" and c.transB and not c.transA for _, mode, c, *_ in cases)
    assert {(c.M, c.N, c.K) for _, _, c, *_ in bench.sweep_cases("large_fp8")} == \
        {(4096, 4096, 4096), (8192, 8192, 8192), (8192, 28672, 8192)}
    assert len(bench.sweep_cases("skinny_fp8")) == 9
    pk = bench.peaks()
    assert pk["fp8_tflops"] == 2 * pk["bf16_tflops"]
    assert pk["fp8_tflops_sustained"] == 2 * pk["bf16_tflops_sustained"]
    assert bench._elem_bytes("fp8") == 1


def test_default_line_times_every_other_config():
    """The default line carries configs 0, 2, 3 and 4 beside the GPT step,
    with the gates where the configurations set them: the tensor peak for
    TF32/BF16 squares of 4096 (both alpha/beta pairs) and both large BF16
    shapes, HBM for all 18 decode shapes."""
    import bench
    cases = bench.config_cases()
    assert {c[0] for c in cases} == {0, 2, 3, 4}
    labels = [c[2] for c in cases]
    assert len(set(labels)) == len(labels)
    assert sum(1 for c in cases if c[0] == 2) == 18 and sum(1 for c in cases if c[0] == 4) == 18
    tensor = sorted(c[2] for c in cases if c[1] == "tensor")
    assert len(tensor) == 6 and all("4096" in t or "8192" in t for t in tensor)
    assert all(c[1] == "hbm" for c in cases if c[0] == 4)
    assert all(c[1] is None for c in cases if c[3] == "fp32")
