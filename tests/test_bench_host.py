"""bench.py's host-side helpers on the CPU: the roofline denominators (the
measured-peaks file or the fallbacks), the DRAM traffic taken from a
recorded ncu capture (scaled to the launch, and dropped once the kernel's
sources change), and the summary of the nvidia-smi clock samples taken
during a timed region."""
import datetime
import json
import os
import time

import pytest

import bench


def _sources(root, files):
    csrc = root / "paged_kv_attention_working_gb300" / "csrc"
    csrc.mkdir(parents=True, exist_ok=True)
    for name, text in files.items():
        (csrc / name).write_text(text)


def test_traffic_is_scaled_to_the_launch_and_dropped_when_sources_change(tmp_path, monkeypatch):
    _sources(tmp_path, {"k.cu": "kernel v1", "h.cuh": "helpers"})
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"kern w": {"source_sha256": bench.kernel_sources_sha(["k.cu", "h.cuh"]),
                      "dram_bytes_per_launch": 1000, "algorithmic_per_launch": 500}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.traffic("kern w", ["k.cu", "h.cuh"], 500) == 1000
    # a capture of a smaller case of the workload, scaled to the full launch
    assert bench.traffic("kern w", ["k.cu", "h.cuh"], 2000) == 4000
    assert bench.traffic("another kernel", ["k.cu", "h.cuh"], 500) is None
    # the hash covers the files in the order given
    assert bench.traffic("kern w", ["h.cuh", "k.cu"], 500) is None
    (tmp_path / "paged_kv_attention_working_gb300" / "csrc" / "k.cu").write_text("kernel v2")
    assert bench.traffic("kern w", ["k.cu", "h.cuh"], 500) is None


def test_traffic_without_a_recorded_capture_is_none(tmp_path, monkeypatch):
    _sources(tmp_path, {"k.cu": "kernel"})
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic("kern w", ["k.cu"], 1) is None


@pytest.mark.parametrize("content, hbm, tensor", [
    (None, (bench.FALLBACK_HBM_GBS, "fallback"), (bench.FALLBACK_BF16_TFLOPS, "fallback")),
    ({"hbm_gbs": 6698.0, "bf16_tflops": 1929.0, "bf16_tflops_sustained": 1743.5},
     (6698.0, "measured"), (1929.0, "measured")),
    ({"hbm_gbs": {"value": 6500}, "bf16_TFLOPs": {"value": 1800.5}}, (6500.0, "measured"), (1800.5, "measured")),
    ({"hbm_gbs": 0, "bf16_tflops": "n/a"},
     (bench.FALLBACK_HBM_GBS, "fallback"), (bench.FALLBACK_BF16_TFLOPS, "fallback")),
    ("{not json", (bench.FALLBACK_HBM_GBS, "fallback"), (bench.FALLBACK_BF16_TFLOPS, "fallback")),
])
def test_peaks_are_measured_when_the_file_has_them(tmp_path, monkeypatch, content, hbm, tensor):
    if content is not None:
        text = content if isinstance(content, str) else json.dumps(content)
        (tmp_path / "MEASURED_PEAKS.json").write_text(text)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.peaks() == hbm
    assert bench.tensor_peak() == tensor


class _StoppedSampler:
    def terminate(self):
        pass

    def wait(self):
        pass


def test_clock_summary_keeps_samples_inside_the_timed_region():
    c = bench.Clocks(0)
    c.proc = _StoppedSampler()
    t0 = time.time()

    def row(dt, sm, mx, hw="Not Active", thermal="Not Active", power="Not Active"):
        ts = datetime.datetime.fromtimestamp(t0 + dt).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return f"{ts}, 0, {sm}, {mx}, 900.5, 0x0, {hw}, {thermal}, Not Active, {power}\n"

    c.f.write(row(-5.0, 1000, 2070, hw="Active"))     # before the region: ignored
    c.f.write(row(0.1, 1980, 2070, power="Active"))
    c.f.write(row(0.3, 2070, 2070))
    c.f.write(row(0.5, "[N/A]", 2070))                  # unreadable clock: not counted
    c.f.write(row(0.7, 2070, 2070))
    c.f.write(row(9.0, 1200, 2070, thermal="Active"))  # after the region: ignored
    c.f.flush()
    s = c.stop(t0, t0 + 1.0)
    assert s["sm_mhz"] == 2070.0
    assert s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    assert s["samples"] == 4
    assert not os.path.exists(c.f.name)


def test_clock_summary_without_nvidia_smi():
    c = bench.Clocks(0)
    c.proc = None
    s = c.stop(0.0, 1.0)
    assert s["sm_mhz"] is None and s["reasons"] == ["nvidia-smi unavailable"]
    assert not os.path.exists(c.f.name)


def test_recorded_captures_match_the_workloads_algorithmic_work():
    """profiles/traffic.json scales each capture by the algorithmic work of
    the launch it measured; that work must still be what bench.py computes
    for the same workload (a change to a workload generator would otherwise
    scale the recorded traffic wrongly)."""
    from paged_kv_attention_working_gb300 import workloads as wl

    with open(os.path.join(os.path.dirname(bench.__file__), "profiles", "traffic.json")) as f:
        rec = json.load(f)
    w8 = wl.llama8b_decode(num_layers=32)
    assert bench.decode_attend_bytes(w8)[1] == rec["decode_kernel llama8b_decode"]["algorithmic_per_launch"]
    # the 70B capture ran 64 of the 256 working sets (8 dedup groups)
    w70 = bench.llama70b_workload(64)
    assert bench.decode_attend_bytes(w70)[1] == rec["decode_kernel llama70b_fp8"]["algorithmic_per_launch"]
    for name in ("mixed_batch", "mixed_batch_e4m3"):
        if f"prefill_kernel {name}" not in rec:    # no capture of the current kernel recorded
            continue
        w = wl.mixed_batch(name=name, kv_dtype=wl.KV_E4M3 if name.endswith("e4m3") else wl.KV_BF16)
        main_segs = [op for op in w.ops if op[0] == "pass"][1][1]
        chunks = [s for s in main_segs if s[0].startswith("c")]
        assert bench.prefill_chunk_flops(w, chunks) == rec[f"prefill_kernel {name}"]["algorithmic_per_launch"]


def test_shared_prefix_bytes_count_each_group_once():
    """The dedup groups' shared prefix is counted once per group: 56 of the 64
    working sets reuse their group's 2048-token prefix, so the batch's K/V
    bytes are those of the unshared batch less 56 prefixes."""
    from paged_kv_attention_working_gb300 import workloads as wl

    w = bench.llama70b_workload(64)
    plain = wl.llama70b_fp8(n_ws=64, prefix_groups=8)
    per_key = w.num_kv_heads * w.head_dim * 1 * 2      # e4m3 K and V
    assert bench.decode_attend_bytes(plain)[0] - bench.decode_attend_bytes(w)[0] == 56 * 2048 * per_key
