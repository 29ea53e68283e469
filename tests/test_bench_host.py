"""Host-side logic of bench.py that needs no GPU: the clock-sample summary
(median SM clock, throttle reasons), the workload config it reports, and the
rule that the committed DRAM-traffic record is used only while the fused
kernel's source still hashes to the recorded value."""
import hashlib
import json
import os
import shutil

import bench
import workloads as wl

CSRC = ("gdr_fused.cu", "gdr_fused_common.cuh", "gdr_sm100.cuh")


def _row(sm, mx, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    return ["0", str(sm), str(mx), "900.0", "0x0", hw, hwt, swt, cap]


def test_clock_summary_median_max_and_reasons():
    c = bench.ClockSampler(0)
    c.rows = [_row(2070, 2070), _row(1980, 2070, cap="Active"), _row(2055, 2070), _row("[N/A]", "[N/A]")]
    s = c.summary()
    assert s["sm_mhz"] == 2055.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 4
    assert s["reasons"] == ["sw_power_cap"]
    c.rows.append(_row(1500, 2070, hw="Active", swt="Active"))
    assert bench.ClockSampler.summary(c)["reasons"] == ["hw_slowdown", "sw_power_cap", "sw_thermal_slowdown"]


def test_clock_summary_without_samples():
    s = bench.ClockSampler(0).summary()
    assert s == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}


def test_config_names_the_bench_workload():
    class A:
        algo, gpus = "auto", 1
    cfg = bench.config_of(wl.GDN_BF16_LARGE, A())
    assert cfg["workload"] == "gdn_bf16_B4_T32768_H32_K128"
    assert (cfg["B"], cfg["T"], cfg["H"], cfg["HV"], cfg["K"], cfg["V"]) == (4, 32768, 32, 32, 128, 128)
    assert cfg["use_qk_l2norm"] and cfg["gate"] == "scalar" and cfg["varlen_lengths"] is None
    assert "larger than L2" in cfg["l2_flush"] and cfg["parallelism"] == "replicas1"


def _fake_root(tmp_path, digest):
    src = os.path.join(bench.ROOT, "chunked_gated_delta_08_gb300", "csrc")
    dst = tmp_path / "chunked_gated_delta_08_gb300" / "csrc"
    dst.mkdir(parents=True)
    for f in CSRC:
        shutil.copy(os.path.join(src, f), dst / f)
    (tmp_path / "profiles").mkdir()
    rec = {"kernel_source_sha256": digest, "traffic_bytes_per_launch_bench_workload": 123456789}
    (tmp_path / "profiles" / "gdr_fused_kernel_traffic.json").write_text(json.dumps(rec))
    return str(tmp_path)


def test_traffic_record_only_while_the_source_matches(tmp_path, monkeypatch):
    h = hashlib.sha256()
    src = os.path.join(bench.ROOT, "chunked_gated_delta_08_gb300", "csrc")
    for f in CSRC:
        with open(os.path.join(src, f), "rb") as fh:
            h.update(fh.read())
    monkeypatch.setattr(bench, "ROOT", _fake_root(tmp_path, h.hexdigest()))
    assert bench.recorded_traffic(wl.GDN_BF16_LARGE, "gdr_fused") == 123456789
    assert bench.recorded_traffic(wl.GDN_BF16_LARGE, "chunked") is None
    assert bench.recorded_traffic(wl.KDA_BF16_VARLEN, "gdr_fused") is None
    # one byte of kernel source changed: the record no longer describes the kernel
    p = tmp_path / "chunked_gated_delta_08_gb300" / "csrc" / "gdr_fused.cu"
    p.write_bytes(p.read_bytes() + b"\n")
    assert bench.recorded_traffic(wl.GDN_BF16_LARGE, "gdr_fused") is None
