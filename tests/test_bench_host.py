"""Host-side logic of bench.py, on the CPU: the kernel sources its traffic
lookup hashes, the lookup itself, the peak file, the algorithmic work of each
operation, the launch count per plan, and the reference arm's JSON line."""

import json
import os
import re
import subprocess
import sys

import pytest
import torch

import bench
import permute_grouped_gemm_gb300 as pgg
from workloads import WORKLOADS, make_inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from permute_grouped_gemm_gb300 import build as pbuild
    pbuild.build()
    return pgg.load()


def test_kernel_sources_exist_and_hash():
    for kernel, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.isfile(os.path.join(ROOT, f)), (kernel, f)
        h = bench.kernel_hash(kernel)
        assert len(h) == 16 and h == bench.kernel_hash(kernel)


def test_recorded_traffic_needs_the_current_source_hash(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the hashed sources are read relative to ROOT as well: give it the real ones
    for files in bench.KERNEL_SOURCES.values():
        for f in files:
            dst = tmp_path / f
            dst.parent.mkdir(parents=True, exist_ok=True)
            dst.write_bytes(open(os.path.join(ROOT, f), "rb").read())
    k = "gmm_dx_owner_kernel"
    assert bench.recorded_traffic(k, "uniform-bf16") is None  # no summary
    good = bench.kernel_hash(k)
    (prof / f"{k}_uniform-bf16.md").write_text(
        f"kernel_source_hash: {good}\ndram_bytes_per_launch: 123456 (read 1 + write 2)\n")
    assert bench.recorded_traffic(k, "uniform-bf16") == 123456
    (prof / f"{k}_uniform-bf16.md").write_text(
        "kernel_source_hash: 0000000000000000\ndram_bytes_per_launch: 123456\n")
    assert bench.recorded_traffic(k, "uniform-bf16") is None  # stale counters are not used


def test_peaks_from_the_measured_file_or_the_fallback(tmp_path, monkeypatch):
    peaks, src = bench.load_peaks()
    assert peaks["bf16_tflops"] > 0 and peaks["hbm_gbs"] > 0
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.load_peaks()
    assert src == "fallback" and peaks == bench.FALLBACK_PEAKS


def test_algorithmic_work_and_launch_counts(lib):
    w = WORKLOADS["uniform-bf16"]
    inp = make_inputs(w, device="cpu")
    dev = torch.device("cpu")
    M, N, K, G, B = w.M, w.N, w.K, w.G, w.batch
    dx = bench.OPS["dx"](inp, pgg, dev)
    flops, nbytes = dx.algorithmic()
    assert flops == 2 * M * N * K
    # d_y and d_x once, the weight of the non-empty experts once, plus the indices
    assert nbytes >= M * N * 2 + G * K * N * 2 + B * K * 4
    assert dx.kernel == "gmm_dx_owner_kernel" and dx.launches == 5
    for op in ("dw", "fwd"):
        o = bench.OPS[op](inp, pgg, dev)
        assert o.algorithmic()[0] == 2 * M * N * K
        assert getattr(o, "launches", 4) == 4
    un = bench.OPS["unperm"](inp, pgg, dev)
    flops, nbytes = un.algorithmic()
    assert flops == 3 * M * N
    assert nbytes == B * N * 2 + 2 * M * N * 2 + 2 * M * 2 + M * 8
    tiny = bench.OPS["dx"](make_inputs(WORKLOADS["tiny-fp32"], device="cpu"), pgg, dev)
    assert tiny.kernel == "gmm_dx_kernel" and tiny.launches == 4


@pytest.mark.parametrize("op", ["dx", "dw", "fwd", "unperm"])
def test_reference_arm_prints_one_json_line(op):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--op", op, "--workload", "tiny-fp32", "--steps", "1", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["unit"] in ("TFLOP/s", "GB/s")
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"] == "tiny-fp32"


def test_clock_summary_covers_only_the_samples_of_its_window():
    c = bench.ClockSampler(0)
    c.samples = [(1.0, 2070.0, 2070.0, (), 300.0),
                 (2.0, 1700.0, 2070.0, ("sw_power_cap",), 1390.0),
                 (3.0, 1800.0, 2070.0, (), 1200.0),
                 (9.0, 900.0, 2070.0, ("hw_slowdown",), 200.0)]
    s = c.summary(1.5, 3.5)
    assert s["samples"] == 2 and s["sm_mhz"] == 1750.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 1390.0
    assert c.summary()["samples"] == 4
    assert c.summary(4.0, 5.0) == {"sm_mhz": None, "sm_max_mhz": None,
                                   "reasons": ["no samples"], "samples": 0, "source": "none"}


def test_reason_bits_name_the_nvml_clock_event_reasons():
    # nvmlClocksEventReason* bit values of the public NVML header
    assert bench._REASON_BITS[0x4] == "sw_power_cap"
    assert bench._REASON_BITS[0x8] == "hw_slowdown"
    assert bench._REASON_BITS[0x20] == "sw_thermal_slowdown"
    assert bench._REASON_BITS[0x40] == "hw_thermal_slowdown"


def test_kernel_source_hashes_cover_the_headers_each_kernel_includes():
    # a profile's recorded hash must change when any device header its kernel
    # includes changes, so every included .cuh is in the kernel's source list
    for kernel, files in bench.KERNEL_SOURCES.items():
        with open(os.path.join(ROOT, files[0])) as f:
            included = set(re.findall(r'#include "([^"]+\.cuh)"', f.read()))
        listed = {os.path.basename(x) for x in files[1:]}
        assert included <= listed, (kernel, sorted(included - listed))


def test_profile_summaries_match_the_current_kernel_sources():
    # every ncu summary that records a kernel source hash was taken on the
    # current source of that kernel, or says that it was not
    import glob
    import os
    import re
    import bench

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    checked = 0
    for path in sorted(glob.glob(os.path.join(root, "profiles", "*.md"))):
        text = open(path).read()
        m = re.search(r"kernel_source_hash:\s*([0-9a-f]{16})", text)
        if not m:
            continue
        name = os.path.basename(path)[: -len(".md")]
        kernel = name[: name.rindex("_")]
        assert kernel in bench.KERNEL_SOURCES, (path, kernel)
        if "capture_of_earlier_source: yes" in text:
            continue
        assert m.group(1) == bench.kernel_hash(kernel), (
            f"{os.path.basename(path)} records {m.group(1)}, the source now hashes to "
            f"{bench.kernel_hash(kernel)}: re-take it or mark it as a capture of an earlier source")
        checked += 1
    assert checked >= 5
