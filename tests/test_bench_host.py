"""Host-side logic of bench.py, on CPU: the clock summary, the sample FLOP
count, and the N>1 plumbing (barrier + max over ranks) with two gloo ranks."""
import glob
import json
import os
import socket
import subprocess
import sys
import textwrap

import bench
from tiled_attention_10_gb300.inputs import WORKLOADS, Workload

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_clock_summary_flags_throttle_reasons():
    rows = [["t", "0", "1900", "2070", "900.0", "0x0", "Not Active", "Not Active", "Not Active", "Active"],
            ["t", "0", "1500", "2070", "1300.0", "0x4", "Not Active", "Not Active", "Not Active", "Active"],
            ["t", "0", "600", "2070", "90.0", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"]]
    c = bench.ClockSampler.summarize(rows)
    assert c["sm_mhz"] == 1700.0          # median of the two samples under load
    assert c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]
    assert bench.ClockSampler.summarize([])["samples"] == 0


def test_peak_choice_follows_run_length_and_power_cap():
    # a short burst at full clock compares against the burst GEMM figure; a
    # region over a second, or one that ran under the power cap, against the
    # sustained one
    assert not bench.use_sustained_peak(200.0, {"reasons": []})
    assert not bench.use_sustained_peak(200.0, {})
    assert bench.use_sustained_peak(1500.0, {"reasons": []})
    assert bench.use_sustained_peak(200.0, {"reasons": ["sw_power_cap"]})


def test_recorded_traffic_is_tied_to_each_kernels_sources():
    # a committed ncu record counts only while the sources it was taken on are
    # unchanged: the forward's records against the forward's files, the
    # backward's against the backward's
    fwd, bwd = bench.kernel_source_sha(), bench.kernel_source_sha(bench.BWD_SOURCES)
    assert fwd != bwd and len(fwd) == len(bwd) == 16
    for kernel, sources, sha in (("fa_fwd", bench.FWD_SOURCES, fwd),
                                 ("fa_bwd_dkdv", bench.BWD_SOURCES, bwd)):
        for path in glob.glob(os.path.join(ROOT, "profiles", f"{kernel}_*.ncu.json")):
            rec = json.load(open(path))
            workload = os.path.basename(path)[len(kernel) + 1:-len(".ncu.json")]
            got = bench.recorded_traffic(workload, kernel, sources)
            assert got == (rec["dram_bytes_per_launch"] if rec["kernel_sha"] == sha else None)
    assert bench.recorded_traffic("no_such_workload") is None


def test_sample_flops_matches_nominal_formula_on_full_problem():
    w = Workload("t", 1, 1, 64, 64, 128, "bf16", "BNSD", False)
    assert bench.sample_flops(w, 1, 64) == w.flops
    wc = Workload("t", 1, 1, 64, 64, 128, "bf16", "BNSD", True)
    # exact causal work (diagonal included) vs the nominal half
    assert bench.sample_flops(wc, 1, 64) == 4 * 128 * (64 * 65 // 2)
    assert abs(bench.sample_flops(wc, 1, 64) / wc.flops - 65 / 64) < 1e-12


def test_headline_flops():
    w = WORKLOADS["bf16_4x32x4096x128"]
    assert w.flops == 4 * 4 * 32 * 4096 * 4096 * 128


def test_reference_arm_prints_one_line(capsys):
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3",
                       "--workload", "fp16_1x8x512x64"]) == 0
    import json
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "TFLOP/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_two_rank_max_over_ranks_gloo():
    code = textwrap.dedent(f"""
        import os, sys
        sys.path.insert(0, {ROOT!r})
        import torch.distributed as dist
        import bench
        rank = int(os.environ["RANK"])
        dist.init_process_group("gloo")
        bench.barrier(2)
        m = bench.max_over_ranks(1.5 + rank, 2)
        assert m == 2.5, m
        dist.destroy_process_group()
        print("rank", rank, "ok")
    """)
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True))
    outs = [p.communicate(timeout=120)[0] for p in procs]
    assert all(p.returncode == 0 for p in procs), outs
    assert all("ok" in o for o in outs)
