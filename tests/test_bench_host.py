"""Host-side logic of bench.py, on the CPU: the multi-rank reduction (two
gloo ranks), the whole-job throughput, the reference arm's rank gating and
JSON line, and the roofline units' choice of binding resource."""
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
import bench  # noqa: E402


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [3.0, 5.0][rank]                      # the slower rank's time wins
        m = bench.max_over_ranks(ms, dist, "cpu")
        out[rank] = (m, bench.job_throughput(1000, 4, world, m))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    port = 29500 + os.getpid() % 1000
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == res[1]
    m, v = res[0]
    assert m == 5.0
    assert v == pytest.approx(1000 * 4 * 2 / 0.005)   # every rank's rows over the slowest time


def test_single_process_reduction_is_identity():
    assert bench.max_over_ranks(2.5) == 2.5
    assert bench.job_throughput(16384, 10, 1, 8.0) == pytest.approx(16384 * 10 / 0.008)


def _run_reference(env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--workload", "tiny", "--steps", "1", "--warmup", "0"],
                          capture_output=True, text=True, env=env, timeout=300)


def test_reference_arm_other_ranks_exit_quietly():
    r = _run_reference({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_reference_arm_rank0_prints_one_line():
    r = _run_reference({"RANK": "0", "WORLD_SIZE": "1"})
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_roofline_units_pick_the_binding_resource():
    peak_f, peak_b = 1701.9e12, 6790.3e9
    c = {"T": 2048, "d": 2048, "f": 768, "E": 64, "k": 8}
    u = bench.kernel_units(c, touched=64)
    R = 2048 * 8
    # GEMM1 FLOPs and bytes written out
    kind, flop, nbytes = u["gemm1_swiglu"]
    assert kind == "flop" and flop == 2.0 * R * 2048 * 2 * 768
    assert nbytes == 64 * 2048 * 1536 * 2 + R * 2048 * 2 + R * 3 * 768 * 2
    # dW1 writes make wgrad1 HBM-bound on this workload, GEMM1 too (weights of 64 experts)
    for name in ("wgrad1", "gemm1_swiglu"):
        _, flop, nbytes = u[name]
        assert nbytes / peak_b > flop / peak_f
    # with 2048 rows per expert the forward GEMMs are compute-bound
    big = bench.kernel_units({"T": 16384, "d": 2048, "f": 768, "E": 8, "k": 1}, touched=8)
    _, flop, nbytes = big["gemm1_swiglu"]
    assert flop / peak_f > nbytes / peak_b
    # memory-only kernels carry no FLOPs
    assert u["merge"][0] is None and u["merge"][1] == 0.0


def test_recorded_traffic_follows_the_kernel_code_not_its_comments():
    real = {n: open(os.path.join(ROOT, "mixture_experts_layer_stable_gb300", "csrc", n)).read()
            for n in os.listdir(os.path.join(ROOT, "mixture_experts_layer_stable_gb300", "csrc"))}
    base = bench.src_digest("ring_forward", real.__getitem__)
    # a comment edit keeps the digest (and so the recorded ncu bytes)
    commented = dict(real, **{"ring.cu": "// note\n" + real["ring.cu"].replace("\n", "  // x\n", 3)})
    assert bench.src_digest("ring_forward", commented.__getitem__) == base
    # a code edit in the kernel's own translation unit or in a header it
    # includes does not
    for name in ("ring.cu", "ptx.cuh", "rowops.cuh"):
        edited = dict(real, **{name: real[name] + "\nstatic int moe_digest_probe;\n"})
        assert bench.src_digest("ring_forward", edited.__getitem__) != base
    # a header the grouped GEMMs do not include does not matter to them
    edited = dict(real, **{"rowops.cuh": real["rowops.cuh"] + "\nstatic int moe_digest_probe;\n"})
    assert bench.src_digest("wgrad1", edited.__getitem__) == bench.src_digest("wgrad1", real.__getitem__)
    # another translation unit does not matter to this kernel
    other = dict(real, **{"sched.cu": real["sched.cu"] + "\nstatic int moe_digest_probe;\n"})
    assert bench.src_digest("ring_forward", other.__getitem__) == base
    assert bench.src_digest("wgrad1", other.__getitem__) == bench.src_digest("wgrad1", real.__getitem__)


def test_clock_sampler_keeps_samples_of_the_load_window():
    import time as _t
    t0 = _t.mktime(_t.strptime("2026/12/03 05:39:00", "%Y/%m/%d %H:%M:%S"))
    lines = ["2026/12/03 05:39:00.100, 0, 300, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "2026/12/03 05:39:01.200, 0, 1980, 2070, 900.5, 0x4, Not Active, Not Active, Not Active, Active",
             "2026/12/03 05:39:01.300, 0, 2000, 2070, 910.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "garbage line"]
    all_ = bench.ClockSampler.parse(lines)
    assert all_["samples"] == 3 and all_["sm_mhz"] == 1980
    win = bench.ClockSampler.parse(lines, since=t0 + 1.0)
    assert win["samples"] == 2 and win["sm_mhz"] == 1990 and win["sm_max_mhz"] == 2070
    assert win["reasons"] == ["sw_power_cap"]
