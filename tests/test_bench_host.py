"""Host-side logic of the benchmark, on CPU: the DRAM-traffic lookup in the committed ncu
summary (reported only while the kernel sources hash to the captured version), the fallback
peaks, the parser of the nvidia-smi clock samples that decides whether a run was throttled, and
the default run's warm-up and workload."""
import json

import pytest

import bench


def _summary(tmp_path, sha, per_unit):
    p = tmp_path / "summary.md"
    p.write_text(f"# kernel\n\nkernel_source_sha256: {sha}\ndram_bytes_per_unit: {per_unit}\n")
    return str(p)


def test_traffic_scales_with_the_units_while_the_sources_match(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", _summary(tmp_path, bench.kernel_source_hash(), 1236.9))
    assert bench.profiled_traffic(1000) == pytest.approx(1236900.0)


def test_traffic_is_null_after_a_source_change_or_without_a_summary(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", _summary(tmp_path, "0123456789abcdef", 1236.9))
    assert bench.profiled_traffic(1000) is None
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", str(tmp_path / "absent.md"))
    assert bench.profiled_traffic(1000) is None


def test_source_hash_follows_every_source_file(tmp_path, monkeypatch):
    a, b = tmp_path / "a.cu", tmp_path / "b.cuh"
    a.write_text("kernel")
    b.write_text("header")
    monkeypatch.setattr(bench, "KERNEL_SOURCES", [str(a), str(b)])
    h0 = bench.kernel_source_hash()
    assert len(h0) == 16 and h0 == bench.kernel_source_hash()
    b.write_text("header changed")
    assert bench.kernel_source_hash() != h0


def test_peaks_fall_back_without_a_readable_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_peaks() == (bench.FALLBACK_PEAKS, "fallback")
    f = tmp_path / "MEASURED_PEAKS.json"
    f.write_text(json.dumps({"hbm_gbs": 6807.9, "bf16_tflops": 1906.3,
                             "bf16_tflops_sustained": 1738.4, "gpu_name": "GB300"}))
    assert bench.load_peaks() == ({"hbm_gbs": 6807.9, "bf16_tflops": 1906.3,
                                   "bf16_tflops_sustained": 1738.4}, "measured")
    f.write_text(json.dumps({"hbm_gbs": 6807.9}))          # a peak missing
    assert bench.load_peaks()[1] == "fallback"
    f.write_text("{ not json")
    assert bench.load_peaks()[1] == "fallback"


class _Exited:
    def terminate(self):
        pass

    def wait(self):
        return 0


def _stopped_sampler(tmp_path, lines):
    s = bench.ClockSampler.__new__(bench.ClockSampler)    # no nvidia-smi: feed its output
    s.file = open(tmp_path / "clocks.csv", "w+")
    s.file.write("\n".join(lines) + "\n")
    s.file.flush()
    s.proc = _Exited()
    return s.stop()


def test_clock_samples_give_the_median_clock_and_the_active_reasons(tmp_path):
    # fields: clocks.sm, clocks.max.sm, power.draw, hw_slowdown, hw_thermal_slowdown,
    # sw_thermal_slowdown, sw_power_cap
    r = _stopped_sampler(tmp_path, [
        "1980, 2070, 1100.5, Not Active, Not Active, Not Active, Active",
        "2070, 2070, 900.0, Not Active, Not Active, Not Active, Not Active",
        "1935, 2070, 1390.2, Not Active, Not Active, Not Active, Active",
        "[N/A], 2070, 1000.0, Not Active, Active, Not Active, Not Active",   # unreadable clock
        "short line",
    ])
    assert r == {"sm_mhz": 1980.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_a_thermal_slowdown_is_reported(tmp_path):
    r = _stopped_sampler(tmp_path, ["1500, 2070, 1000.0, Not Active, Active, Not Active, Not Active"])
    assert r["reasons"] == ["hw_thermal_slowdown"] and r["sm_mhz"] == 1500.0


def test_default_run_is_the_long_text_workload_with_enough_warmup():
    args = bench.parse_args([])
    assert args.warmup >= 3 and args.steps >= 1 and args.gpus == 1 and args.impl == "ours"
    w = bench.workload(args)
    assert (w.name, w.B, w.H, w.N, w.d) == ("long_text", 2, 16, 16384, 128)
    w = bench.workload(bench.parse_args(["--workload", "vit_b16_batch", "--shape", "1,16,8192,128"]))
    assert (w.B, w.H, w.N, w.d) == (1, 16, 8192, 128) and w.name.startswith("vit_b16_batch")


def test_error_norms_of_the_sample_check():
    np = pytest.importorskip("numpy")
    rng = np.random.default_rng(5)
    ref = {"o": rng.normal(size=(1, 1, 40, 8)), "lse": rng.normal(size=(1, 1, 40)) + 3.0,
           "dq": rng.normal(size=(1, 1, 40, 8)), "dk": rng.normal(size=(1, 1, 40, 8)),
           "dv": rng.normal(size=(1, 1, 40, 8))}
    ref["o"][0, 0, 7, 3] = 3.0                       # one large output, where a bf16 step is 2^-6
    got = {k: v.copy() for k, v in ref.items()}
    got["o"][0, 0, 7, 3] += 2.0 ** -6                # exactly one step off there
    got["o"][0, 0, 1, 1] += 1e-3
    got["lse"][0, 0, 2] += 4e-5 * 4.0
    got["dq"] *= 1.004
    e = bench.error_norms(got, ref)
    assert e["o_max_abs"] == pytest.approx(2.0 ** -6) and e["o_ref_at_max"] == 3.0
    assert e["o_max_abs_in_bf16_steps"] == pytest.approx(1.0)
    assert e["o_elems_over_1e-2"] == 1
    assert e["lse_rel"] == pytest.approx(4e-5 * 4.0 / np.abs(ref["lse"]).max())
    assert e["dq_rel_fro"] == pytest.approx(0.004)
    assert e["dk_rel_fro"] == 0.0 and e["dv_rel_fro"] == 0.0
    assert 0 < e["o_rel_fro"] < 1e-2


def test_both_arms_describe_the_workload_alike():
    w = bench.workload(bench.parse_args([]))
    c = bench.workload_config(w, 4)
    assert c == {"workload": "long_text", "B": 2, "H": 16, "N": 16384, "d_k": 128, "seq_len": 16384,
                 "global_batch": 8, "parallelism": "independent batches x4", "qk_std": 2.0}
