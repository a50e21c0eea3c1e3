"""The benchmark's own arithmetic on the CPU: the algorithmic bytes and flop
counts behind the reported roofline fractions, against the totals tabulated
for the workloads (14 bytes per bf16 element of optimizer state; standard
Newton-Schulz count T (4 m^2 n + 2 m^3) per slice) and against closed forms
of the symmetric-aware count T (3 m^2 n + m^3)."""
import pytest
import torch

import bench
import synth


@pytest.mark.parametrize("name,gbytes,gflop", [("skinny_74x24x10240", 0.2546, 8.74),
                                               ("stacks_experts", 8.63, 20980),
                                               ("dense_24L", 68.0, 513334),
                                               ("moe_24L", 52.4, 150448)])
def test_workload_bytes_and_flops_match_the_tables(name, gbytes, gflop):
    w = synth.workload(name)
    nbytes, flops, flops_sym, skinny_bytes, per_el = bench.workload_work(w)
    assert per_el == 14
    assert nbytes / 1e9 == pytest.approx(gbytes, rel=3e-3)
    assert flops / 1e9 == pytest.approx(gflop, rel=6e-4)
    # the symmetric-aware count is never more than the standard one, and at
    # least half of it (3 m^2 n + m^3 >= (4 m^2 n + 2 m^3) / 2)
    assert flops / 2 <= flops_sym <= flops


def test_symmetric_count_closed_forms():
    w = synth.Workload("t", ((24, 10240), (3, 64, 128), (4096, 11008)), torch.bfloat16, 1e-2)
    _, flops, flops_sym, skinny_bytes, _ = bench.workload_work(w)
    T = w.ns_steps
    std = T * ((4 * 24 * 24 * 10240 + 2 * 24 ** 3) + 3 * (4 * 64 * 64 * 128 + 2 * 64 ** 3)
               + (4 * 4096 * 4096 * 11008 + 2 * 4096 ** 3))
    sym = T * ((3 * 24 * 24 * 10240 + 24 ** 3) + 3 * (3 * 64 * 64 * 128 + 64 ** 3)
               + (3 * 4096 * 4096 * 11008 + 4096 ** 3))
    assert flops == std and flops_sym == sym
    # the fused kernel's groups (m <= 64) carry the bytes of the HBM roofline
    assert skinny_bytes == 14 * (24 * 10240 + 3 * 64 * 128)


def test_fp32_parameters_take_20_bytes_per_element():
    w = synth.workload("fp32_24x1024")
    nbytes, _, _, _, per_el = bench.workload_work(w)
    assert per_el == 20 and nbytes == 20 * 24 * 1024


def test_peaks_come_from_the_measured_file_when_present():
    pk = bench.peaks()
    assert pk["src"] in ("measured", "fallback")
    assert pk["hbm"] > 1000 and pk["tc"] > pk["tc_sustained"] > 100


def test_source_digest_ignores_comments_only(tmp_path):
    import bench
    a = tmp_path / "a.cu"
    a.write_text("// header\nint f(int x) {  /* twice */ return 2 * x; }\n")
    b = tmp_path / "b.cu"
    b.write_text("/* another\n header */\nint f(int x) {\n  return 2 * x;  // doubled\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("int f(int x) { return 3 * x; }\n")
    assert bench.source_digest(str(a)) == bench.source_digest(str(b))
    assert bench.source_digest(str(a)) != bench.source_digest(str(c))


def test_profile_value_needs_a_matching_digest(tmp_path, monkeypatch):
    import bench
    prof = tmp_path / "profiles"
    src = tmp_path / "newton_schulz_05_gb300" / "csrc"
    prof.mkdir()
    src.mkdir(parents=True)
    (src / "k.cu").write_text("__global__ void k() {}\n")
    digest = bench.source_digest(str(src / "k.cu"))
    (prof / "k.txt").write_text("source digest: %s\ndram bytes per launch: 1234\n" % digest)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profile_value("k.txt", "k.cu", "dram bytes per launch") == 1234.0
    (src / "k.cu").write_text("__global__ void k() { int x = 0; }\n")
    assert bench.profile_value("k.txt", "k.cu", "dram bytes per launch") is None


@pytest.mark.parametrize("clocks,rejected", [
    ({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 10}, False),
    ({"sm_mhz": 1490.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 10}, False),
    ({"sm_mhz": 1900.0, "sm_max_mhz": 2070.0, "reasons": ["hw_slowdown"], "samples": 10}, True),
    ({"sm_mhz": 1900.0, "sm_max_mhz": 2070.0, "reasons": ["sw_thermal_slowdown"], "samples": 5}, True),
    ({"sm_mhz": 1000.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 10}, True),
    ({"sm_mhz": 1000.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 2}, False),
    ({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}, False),
])
def test_clock_record_rejection_rule(clocks, rejected):
    # without a process group the decision is this rank's own
    assert bench.clock_rejected(clocks, torch.device("cpu")) is rejected
