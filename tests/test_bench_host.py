"""Host-side logic of bench.py, on the CPU.

The benchmark's numbers are only as good as the bookkeeping around them:
  - the clock record must flag a throttled or clock-locked run (the samples
    taken inside the timed region, the throttle reasons that were active);
  - the ncu summaries must add up launches, times, shares and DRAM bytes per
    kernel from ncu's CSV log, converting its units;
  - the DRAM traffic figure may only be reported while the GEMM's sources are
    the ones it was captured on.
None of this needs a GPU: nvidia-smi and ncu output is fed in as text.
"""
import argparse
import json
import os
import shutil

import pytest

import bench


# ------------------------------------------------------------- clocks ---
def sampler(lines, t0, t1):
    """A ClockSampler holding the given (time, nvidia-smi line) samples, no subprocess."""
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    cs.proc = object()
    cs.samples = list(lines)
    cs.t0, cs.t1 = t0, t1
    return cs


def smi(sm, smax, hw="Not Active", hw_thermal="Not Active", sw_thermal="Not Active", power_cap="Not Active"):
    return f"0, {sm}, {smax}, 700.5, 0x0000000000000000, {hw}, {hw_thermal}, {sw_thermal}, {power_cap}"


def test_clock_summary_uses_only_the_timed_region():
    lines = [(0.5, smi(1000, 2070, hw="Active")),      # before the region: ignored
             (1.1, smi(2070, 2070)), (1.2, smi(2055, 2070)), (1.3, smi(2070, 2070)),
             (3.0, smi(900, 2070, sw_thermal="Active"))]  # after the region: ignored
    s = sampler(lines, 1.0, 2.0).summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == []


def test_clock_summary_reports_every_active_reason_once():
    lines = [(1.1, smi(1400, 2070, power_cap="Active")), (1.2, smi(1380, 2070, hw="Active", power_cap="Active")),
             (1.3, smi(1300, 2070, hw_thermal="Active")), (1.4, "garbage line"), (1.5, smi("[N/A]", 2070))]
    s = sampler(lines, 1.0, 2.0).summary()
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap"]
    assert s["samples"] == 3  # the malformed and the non-numeric lines are skipped
    assert s["sm_mhz"] == 1380.0


def test_clock_summary_without_nvidia_smi():
    cs = sampler([], 0.0, 1.0)
    cs.proc = None
    s = cs.summary()
    assert s["samples"] == 0 and s["sm_mhz"] is None and s["reasons"] == ["nvidia-smi unavailable"]


def test_clock_summary_short_region_takes_the_nearest_samples():
    lines = [(float(i), smi(2000 + i, 2070)) for i in range(6)]
    s = sampler(lines, 10.0, 10.001).summary()  # no sample inside: the last three
    assert s["samples"] == 3 and s["sm_mhz"] == 2004.0


# ------------------------------------------------------- ncu summaries ---
HEADER = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size",'
          '"Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"')


def ncu_row(i, kernel, metric, unit, value):
    return (f'"{i}","9","python3.12","127.0.0.1","{kernel}","1","13","(160, 1, 1)","(456, 1, 1)","0","10.3",'
            f'"Command line profiler metrics","{metric}","{unit}","{value}"')


@pytest.fixture
def fake_root(tmp_path, monkeypatch):
    os.makedirs(tmp_path / "profiles")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "feedc0de")
    return tmp_path


def write_csv(path, rows):
    with open(path, "w") as f:
        f.write("==PROF== Connected to process 9\n==PROF== Disconnected from process 9\n")
        f.write(HEADER + "\n" + "\n".join(rows) + "\n")


def test_summarize_ncu_launch_list_and_traffic(fake_root):
    # kernel names as ncu prints them (an anonymous namespace shows as "unnamed>::")
    gemm = "void k_verify_gemm<0, 64, 2, 0>(GemmArgs)"
    act = "void unnamed>::k_rotate_quant_act<1, 1024>(const float *, int, int, const unsigned int *, signed char *)"
    rows = []
    for i in range(3):  # three GEMM launches: 30 MB read + 0.5 MB written each, 10 us each
        rows += [ncu_row(2 * i, gemm, "dram__bytes_read.sum", "Mbyte", "30.00"),
                 ncu_row(2 * i, gemm, "dram__bytes_write.sum", "Kbyte", "500"),
                 ncu_row(2 * i, gemm, "gpu__time_duration.sum", "usecond", "10.00")]
        rows += [ncu_row(2 * i + 1, act, "dram__bytes_read.sum", "byte", "262,144"),
                 ncu_row(2 * i + 1, act, "dram__bytes_write.sum", "byte", "0"),
                 ncu_row(2 * i + 1, act, "gpu__time_duration.sum", "nsecond", "2500")]
    csv = fake_root / "launches.csv"
    write_csv(csv, rows)
    args = argparse.Namespace(summarize_ncu=str(csv), ncu_name="unit", ncu_command="ncu ... (test)")
    assert bench.summarize_ncu(args) == 0
    md = (fake_root / "profiles" / "launches_unit.md").read_text()
    assert "| `k_verify_gemm<0, 64, 2, 0>` | 3 | 30.0 | 80.0% | 90.0 | 1.5 |" in md
    assert "| `k_rotate_quant_act<1, 1024>` | 3 | 7.5 | 20.0% | 0.8 | 0.0 |" in md
    assert "Command: `ncu ... (test)`" in md
    rec = json.loads((fake_root / "profiles" / "k_verify_gemm_unit_traffic.json").read_text())
    assert rec["launches"] == 3 and rec["kernel_source_hash"] == "feedc0de"
    assert rec["dram_bytes_per_launch"] == pytest.approx(30.5e6)


def test_summarize_ncu_time_only_writes_no_traffic_record(fake_root):
    gemm = "void k_verify_gemm<0, 64, 2, 0>(GemmArgs)"
    csv = fake_root / "t.csv"
    write_csv(csv, [ncu_row(0, gemm, "gpu__time_duration.sum", "msecond", "0.011")])
    bench.summarize_ncu(argparse.Namespace(summarize_ncu=str(csv), ncu_name="t", ncu_command=""))
    assert "| 1 | 11.0 | 100.0% |" in (fake_root / "profiles" / "launches_t.md").read_text()
    assert not (fake_root / "profiles" / "k_verify_gemm_t_traffic.json").exists()


# ------------------------------------------------- traffic record gate ---
def test_traffic_record_only_for_the_sources_it_was_taken_on(fake_root, monkeypatch):
    path = fake_root / "profiles" / "k_verify_gemm_decoder_9b_traffic.json"
    path.write_text(json.dumps({"dram_bytes_per_launch": 30.3e6, "kernel_source_hash": "feedc0de"}))
    assert bench.gemm_traffic_record()["dram_bytes_per_launch"] == 30.3e6
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0ther")
    assert bench.gemm_traffic_record() is None
    path.write_text("not json")
    assert bench.gemm_traffic_record() is None


def test_kernel_source_hash_follows_the_gemm_sources(tmp_path, monkeypatch):
    here = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "quantized_speculative_verify_gb300", "csrc")
    csrc = tmp_path / "quantized_speculative_verify_gb300" / "csrc"
    shutil.copytree(here, csrc)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    assert h0 == bench.kernel_source_hash()
    # a kernel outside the GEMM does not change it
    with open(csrc / "k_attn.cu", "a") as f:
        f.write("\n// unrelated\n")
    assert bench.kernel_source_hash() == h0
    # the GEMM's launcher in the API file does
    api = (csrc / "hq_api.cu").read_text()
    i = api.index("cudaError_t launch_verify_gemm(")
    (csrc / "hq_api.cu").write_text(api[:i] + api[i:].replace("MIN_TILES = 4", "MIN_TILES = 5", 1))
    h1 = bench.kernel_source_hash()
    assert h1 != h0
    # so does the register-resident kernel and the code both GEMMs share
    for f in ("k_gemm_rs.cuh", "gemm_common.cuh"):
        with open(csrc / f, "a") as fh:
            fh.write("\n// changed\n")
        assert bench.kernel_source_hash() != h1
        h1 = bench.kernel_source_hash()


def test_gemm_kernel_name_follows_the_library_dispatch():
    assert bench.gemm_kernel_name("w4", 16) == bench.gemm_kernel_name("w8", 32) == "k_verify_gemm_rs"
    assert bench.gemm_kernel_name("w4", 33) == bench.gemm_kernel_name("w8", 128) == "k_verify_gemm"


# ------------------------------------------------------ reference arm ---
def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the CPU oracle) prints one JSON line on the
    same metric, unit and workload as the GPU arm, with its own cpu_baseline
    and an e2e entry that moves no bytes."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["config"]["workload"] == bench.WORKLOAD
    assert line["steps"] == 1 and line["warmup"] == 1 and line["value"] > 0
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == line["value"] and cpu["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_do_no_work(capsys):
    class OtherRank:
        rank = 1

    args = argparse.Namespace(steps=1, warmup=1, gpus=2)
    assert bench.run_reference(args, OtherRank()) == 0
    assert capsys.readouterr().out == ""
