"""The benchmark's reference arm (the oracle on the host cores) prints the one JSON line the
measurement contract asks for; it needs no GPU, so its keys and types are checked here."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def reference_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    return json.loads(out.stdout.strip().splitlines()[-1])


def test_reference_line_keys(reference_line):
    d = reference_line
    sys.path.insert(0, ROOT)
    import bench
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["data"] == "synthetic"
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 0
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["vs_baseline"] is None
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_clock_record_uses_the_timed_region():
    """The clock record of the GPU line: the median over the samples taken inside the timed region
    when there are at least three, else over the loaded window that continues it (and it says
    which); throttle reasons seen anywhere in the loaded window are reported."""
    sys.path.insert(0, ROOT)
    import bench
    c = bench.ClockSampler(0)
    line = lambda mhz, pc="Not Active": f"{mhz}, 2070, 900.0, Not Active, Not Active, Not Active, {pc}"
    c.lines = [(0.5, line(900)), (1.1, line(2070)), (1.2, line(2060)), (1.3, line(2070)), (1.9, line(2000, "Active")),
               (3.0, line(1000))]
    s = c.summary(1.0, 1.5, 2.0)
    assert s["samples"] == 3 and s["samples_loaded"] == 4 and s["sm_mhz"] == 2070.0
    assert s["window"] == "timed region" and s["reasons"] == ["sw_power_cap"] and s["sm_max_mhz"] == 2070.0
    short = c.summary(1.0, 1.15, 2.0)
    assert short["samples"] == 1 and short["window"].startswith("timed region and")
    assert short["sm_mhz"] == float(np.median([2070, 2060, 2070, 2000]))


def test_traffic_record_follows_the_gemm_code(tmp_path):
    """The committed DRAM-traffic ratio is used only while gemm.cu's code is the one it was captured
    with: its digest ignores comments and white space and changes with any code token."""
    sys.path.insert(0, ROOT)
    import bench
    src = os.path.join(ROOT, "bit_exact_speculative_gb300", "csrc", "gemm.cu")
    assert bench.traffic_ratio_from_profile(src) is not None     # the record matches the code as committed
    code = open(src).read()
    a = tmp_path / "a.cu"
    a.write_text("// a new comment\n/* and a block\n comment */\n" + code.replace("\n", "\n  "))
    assert bench.code_digest(str(a)) == bench.code_digest(src)
    b = tmp_path / "b.cu"
    b.write_text(code.replace("constexpr int STAGES = 4;", "constexpr int STAGES = 5;"))
    assert bench.code_digest(str(b)) != bench.code_digest(src)
    assert bench.traffic_ratio_from_profile(str(b)) is None
