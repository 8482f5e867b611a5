"""Host logic of bench.py that needs no GPU: the roofline denominators, the
DRAM-traffic record keyed on the attend kernel's source, and the parsing of
the nvidia-smi clock samples taken during the timed region."""
import json
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _fake_root(tmp_path, source_text=b"__global__ void k() {}\n", record=None):
    csrc = tmp_path / "mla_absorbed_latent_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "attend_tc.cu").write_bytes(source_text)
    (tmp_path / "profiles").mkdir()
    if record is not None:
        (tmp_path / "profiles" / "attend_traffic.json").write_text(json.dumps(record))
    return tmp_path


def _record(source_text, **over):
    d = {"source": "attend_tc.cu", "source_digest": bench.source_digest(source_text.decode()), "kind": "tcgen05",
         "fmt": "bf16", "workload_name": "v3_paged", "cache_bytes": 603979776, "dram_bytes_per_launch": 617000000}
    d.update(over)
    return d


def test_traffic_is_reported_for_the_captured_source(tmp_path, monkeypatch):
    src = b"__global__ void attend() {}\n"
    monkeypatch.setattr(bench, "ROOT", str(_fake_root(tmp_path, src, _record(src))))
    assert bench.kernel_traffic("tcgen05", "bf16", "v3_paged", 603979776) == 617000000


@pytest.mark.parametrize("change", ["source", "kind", "fmt", "workload", "size", "missing"])
def test_traffic_is_dropped_when_it_no_longer_describes_the_kernel(tmp_path, monkeypatch, change):
    src = b"__global__ void attend() {}\n"
    rec = _record(src)
    if change == "source":
        rec["source_digest"] = bench.source_digest((src + b"__device__ int edited;\n").decode())
    elif change == "kind":
        rec["kind"] = "cuda-core"
    elif change == "fmt":
        rec["fmt"] = "int8"
    root = _fake_root(tmp_path, src, None if change == "missing" else rec)
    monkeypatch.setattr(bench, "ROOT", str(root))
    workload, size = ("v3_ragged", 603979776) if change == "workload" else ("v3_paged", 150994944) if change == "size" \
        else ("v3_paged", 603979776)
    assert bench.kernel_traffic("tcgen05", "bf16", workload, size) is None


def test_digest_follows_code_not_comments():
    a = "__global__ void k(int* x) {\n  x[0] = 1;  // one\n}\n"
    b = "/* the kernel */\n__global__ void k(int* x) {   x[0] = 1;\n\n  // set the first element\n}"
    c = "__global__ void k(int* x) {\n  x[0] = 2;  // one\n}\n"
    assert bench.source_digest(a) == bench.source_digest(b)
    assert bench.source_digest(a) != bench.source_digest(c)


def test_peaks_measured_and_fallback(tmp_path, monkeypatch):
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
        d = json.load(f)
    hbm, tf, tf_sus, src = bench.load_peaks()
    assert src == "measured" and hbm == float(d["hbm_gbs"]) and tf == float(d["bf16_tflops"])
    assert tf_sus == float(d.get("bf16_tflops_sustained", d["bf16_tflops"]))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))  # no peaks file there
    assert bench.load_peaks() == (6800.0, 1900.0, 1700.0, "fallback")


class _FakeProc:
    def __init__(self, text):
        self.text = text

    def terminate(self):
        pass

    def kill(self):
        pass

    def communicate(self, timeout=None):
        return self.text, ""


def test_clock_samples_median_max_and_reasons():
    # index, sm, max sm, power, active mask, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap
    rows = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1200.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 10.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    cs = bench.ClockSampler(0)
    cs.proc = _FakeProc("\n".join(rows) + "\n")
    got = cs.stop()
    assert got == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_clock_samples_flag_thermal_slowdown():
    rows = ["0, 1400, 2070, 1390.0, 0x28, Active, Not Active, Active, Not Active"]
    cs = bench.ClockSampler(0)
    cs.proc = _FakeProc("\n".join(rows) + "\n")
    got = cs.stop()
    assert got["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"] and got["sm_mhz"] == 1400.0


def test_clock_sampler_without_nvidia_smi_reports_nothing():
    cs = bench.ClockSampler(0)
    assert cs.stop() is None


def test_producer_roofline_picks_the_binding_ceiling():
    """A 32,768-token chunk at hidden 7168 does ~525 FLOP per byte: tensor-bound on
    these peaks; a 64-token decode-time append (~57 FLOP/B) is bound by HBM."""
    peaks = (6677.8, 1939.3, 1751.0, "measured")
    flops, nbytes = bench.project_work(32768, 7168, "bf16")
    assert flops == 2.0 * 32768 * 576 * 7168
    assert nbytes == 576 * 7168 * 2 + 32768 * 7168 * 2 + 32768 * 1152
    r = bench.project_roofline(flops, nbytes, 0.25, peaks)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(flops / 0.25e-3 / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / 1939.3)
    flops, nbytes = bench.project_work(64, 7168, "int8")
    assert nbytes == 576 * 7168 * 2 + 64 * 7168 * 2 + 64 * 624
    r = bench.project_roofline(flops, nbytes, 0.01, peaks)
    assert r["bound"] == "hbm" and r["frac"] == pytest.approx(nbytes / 1e-5 / 1e9 / 6677.8)


def test_parity_stats_of_the_timed_output():
    rng = np.random.default_rng(3)
    ref = {b: rng.standard_normal((16, 128)) for b in (0, 5)}
    good = {b: r + 1e-4 * rng.standard_normal(r.shape) for b, r in ref.items()}
    st = bench.parity_stats(good, ref)
    assert st["rows"] == 2 and st["within_tolerance"] and st["max_abs_err"] < 1e-3
    bad = dict(good)
    bad[5] = ref[5] * 1.05          # 5 % off: elementwise within 2e-2 + 1e-2|ref| fails somewhere
    st = bench.parity_stats(bad, ref)
    assert not st["within_tolerance"] and st["worst_head_rel_rms"] == pytest.approx(0.05, rel=1e-6)
    zero = {0: np.zeros((16, 128))}  # an all-zero output does not pass on rows with real values
    assert not bench.parity_stats(zero, {0: ref[0]})["within_tolerance"]
    assert bench.parity_stats({}, ref) is None
