"""bench.py's JSON line, checked on the CPU through its reference arm (the
float64 oracle on the host cores; no GPU needed): the keys and types every
line carries, the warm-up floor, and that ranks other than 0 of a multi-rank
launch exit without work or output."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*argv, env=None):
    e = dict(os.environ)
    e.update(env or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *argv], cwd=ROOT,
                       env=e, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return r.stdout


def _line(out):
    lines = [l for l in out.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out
    return json.loads(lines[0])


@pytest.mark.parametrize("workload,unit,dtype", [
    ("c1", "positions/s", "f64"), ("s2", "tokens/s", "f64"), ("c3t", "positions/s", "f64"),
    ("kvp", "sequences/s", "int64"), ("dynk", "sequences/s", "int64")])
def test_reference_line_carries_the_contract_keys(workload, unit, dtype):
    d = _line(_bench("--impl", "reference", "--workload", workload, "--steps", "1",
                     "--warmup", "1", "--ref-sample", "2"))
    assert d["impl"] == "reference"
    assert isinstance(d["metric"], str) and d["metric"]
    assert d["unit"] == unit and d["value"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == 1
    assert d["warmup"] == 3  # raised to the floor of three warm-up steps
    assert d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["dtype"] == dtype and d["data"] == "synthetic"
    cfg = d["config"]
    assert isinstance(cfg["workload"], str) and cfg["workload"]
    assert not {"model", "seq_len", "global_batch"} & set(cfg)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == unit
    assert cb["cores"] >= 1 and isinstance(cb["sample"], str) and cb["sample"]
    e2e = d["e2e"]
    assert e2e == {"value": d["value"], "unit": unit, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_without_work():
    out = _bench("--impl", "reference", "--workload", "c1", "--steps", "1", "--warmup", "3",
                 "--ref-sample", "2", env={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert out.strip() == ""


def test_clock_sampler_reads_clocks_and_throttle_reasons():
    """The clocks object of the JSON line: the median SM clock under load, the
    maximum, and every throttle reason reported active in any sample."""
    sys.path.insert(0, ROOT)
    import bench
    cs = bench.ClockSampler(0)
    cs.proc = type("P", (), {"terminate": lambda self: None, "wait": lambda self, timeout=None: 0,
                             "kill": lambda self: None})()
    cs.lines = [
        "2070, 2070, 0x0, Not Active, Not Active, Not Active, Not Active",
        "1980, 2070, 0x4, Not Active, Not Active, Not Active, Active",
        "2070, 2070, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage",
        "[N/A], 2070, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    clk = cs.stop()
    assert clk["sm_mhz"] == 2070.0 and clk["sm_max_mhz"] == 2070.0
    assert clk["reasons"] == ["sw_power_cap"] and clk["samples"] == 3
    cs.lines = ["2070, 2070, 0x0, Active, Not Active, Active, Not Active"]
    assert bench.ClockSampler.stop(cs)["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_traffic_is_reported_only_for_the_captured_source(monkeypatch):
    """roofline.traffic comes from an ncu capture and is dropped (None) as soon
    as the kernel source differs from the one the capture was taken on."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.traffic_for("c2", 123.0) == 123.0  # an explicit override
    assert bench.traffic_for("no-such-workload", None) is None
    src, digest, value = bench.MEASURED_TRAFFIC["c2"]
    monkeypatch.setitem(bench.MEASURED_TRAFFIC, "c2", (src, "0" * 16, value))
    assert bench.traffic_for("c2", None) is None


def test_no_cluster_multicast_in_the_sources():
    """No kernel of the library uses a cluster-multicast form (TMA loads or
    tcgen05 commits): the LM head's CTA pairs stage their own rows and their
    own half of each W tile, so nothing restricts a process or a replica run
    to one GPU."""
    import glob
    srcs = glob.glob(os.path.join(ROOT, "speculative_decoding_verification_47_gb300", "csrc", "*"))
    assert srcs
    for p in srcs:
        with open(p) as f:
            text = f.read()
        assert "multicast" not in text, p


PROFILE_OF = {"c2": "verify_kernel_c2.md", "c1": "verify_kernel_c1.md", "c3": "verify_kernel_c3_topp.md",
              "c3t": "verify_kernel_c3t.md", "s2": "sample_kernel_s2.md", "c4": "lmhead_gemm_c4.md"}


def test_bench_traffic_matches_the_committed_profiles():
    """Each workload's roofline.traffic in bench.py and the ncu summary under
    profiles/ describe the same capture: the same source file and hash, and
    DRAM read + write equal to the bench figure."""
    import re
    sys.path.insert(0, ROOT)
    import bench

    def mbytes(value, unit):
        return float(value) * {"byte": 1e-6, "Kbyte": 1e-3, "Mbyte": 1.0, "Gbyte": 1e3}[unit]

    for workload, name in PROFILE_OF.items():
        src, digest, value = bench.MEASURED_TRAFFIC[workload]
        text = open(os.path.join(ROOT, "profiles", name)).read()
        m = re.search(r"csrc/(\S+), sha256 prefix ([0-9a-f]{16})", text)
        assert m, name
        assert (m.group(1), m.group(2)) == (src, digest), (workload, m.groups(), src, digest)
        rd = re.search(r"DRAM read\s+([0-9.]+) (\w+)", text)
        wr = re.search(r"DRAM write\s+([0-9.]+) (\w+)", text)
        got = mbytes(*rd.groups()) + mbytes(*wr.groups())
        assert abs(got - value / 1e6) < 1e-3, (workload, got, value / 1e6)
