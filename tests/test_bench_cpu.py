"""CPU checks of bench.py: the reference (oracle) arm's JSON line, and the
rank arithmetic of the multi-process path over gloo with world size 2."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "window48_L256", "--steps", "2", "--warmup", "3", "--cpu-rows", "64"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["unit"] == "TFLOP/s" and out["value"] > 0
    assert out["e2e"]["h2d_bytes_per_step"] == 0 and out["cpu_baseline"]["kind"] == "oracle"
    assert out["config"]["workload"] == "window48_L256"


def test_warmup_below_three_is_rejected():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--warmup", "2"], capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert r.returncode != 0


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    dev = torch.device("cpu")
    q.put((rank, bench.max_over_ranks(1.0 + rank, dist, dev), bench.sum_over_ranks(10.0 * (rank + 1), dist, dev)))
    dist.barrier()
    dist.destroy_process_group()


def test_rank_reductions_world_size_2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2.0, 30.0), (1, 2.0, 30.0)]


def test_traffic_is_reported_only_for_the_profiled_kernel_source(tmp_path, monkeypatch):
    # roofline.traffic comes from the committed ncu summary only while the
    # block-wise kernel's device code is the one that was profiled
    import shutil
    sys.path.insert(0, ROOT)
    import bench
    csrc = tmp_path / "sparse_mask_transformer_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in ("blockwise.cu", "blockwise_common.cuh", "sm100_ptx.cuh"):
        shutil.copy(os.path.join(ROOT, "sparse_mask_transformer_gb300", "csrc", f), csrc / f)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash()
    (tmp_path / "profiles" / "blockwise_wl.md").write_text(
        f"kernel_source_sha256: {h}\ntraffic_bytes_per_launch: 1.5e9\n")
    assert bench.profiled("wl", "traffic_bytes_per_launch") == 1.5e9
    assert bench.profiled("other", "traffic_bytes_per_launch") is None
    # host launch code below the marker does not change the device-code hash
    with open(csrc / "blockwise.cu", "a") as fh:
        fh.write("\n// host-side note\n")
    assert bench.profiled("wl", "traffic_bytes_per_launch") == 1.5e9
    # nor does a comment in the device code
    src = (csrc / "blockwise_common.cuh").read_text()
    (csrc / "blockwise_common.cuh").write_text(src + "\n// a note\n/* another */\n")
    assert bench.profiled("wl", "traffic_bytes_per_launch") == 1.5e9
    # a change to the device code does
    src = (csrc / "blockwise_common.cuh").read_text()
    (csrc / "blockwise_common.cuh").write_text(src + "\nconstexpr int kDeviceSideChange = 1;\n")
    assert bench.profiled("wl", "traffic_bytes_per_launch") is None


def test_run_for_keeps_stepping_for_the_given_time():
    sys.path.insert(0, ROOT)
    import time
    import bench
    calls = []
    t0 = time.perf_counter()
    n = bench.run_for(lambda: (calls.append(1), time.sleep(0.01)), 0.1)
    assert n == len(calls) >= 5 and time.perf_counter() - t0 >= 0.1


def test_clock_summary_reports_median_and_throttle_reasons():
    sys.path.insert(0, ROOT)
    import bench
    clk = bench.ClockSampler(0)
    act, no = "Active", "Not Active"
    clk.lines = [f"0, {mhz}, 2070, 900.0, 0x0, {no}, {no}, {no}, {cap}"
                 for mhz, cap in ((1980, no), (2070, act), (1995, no))] + ["garbage line"]
    out = clk.summary()
    assert out["sm_mhz"] == 1995 and out["sm_max_mhz"] == 2070 and out["samples"] == 3
    assert out["reasons"] == ["sw_power_cap"]
    clk.lines = []
    assert clk.summary()["reasons"] == ["unsampled"]


def test_l2_note_says_which_case_applies():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.l2_note(8_589_934_592, 402_653_184).startswith("inputs larger than L2")
    assert "warm L2" in bench.l2_note(65_536, 196_608)
