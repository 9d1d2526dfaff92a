"""Host logic of the benchmark, on the CPU.

The clock record (median SM clock, the largest maximum clock and power, and the throttle
reasons seen during the timed region) is parsed from nvidia-smi's CSV; a stand-in
`nvidia-smi` on PATH prints canned samples, so nothing here queries or changes a GPU. The
LSE kernel's DRAM traffic is read from the committed ncu record only while the kernel's
sources hash to the value the record was taken on."""
import importlib.util
import os
import stat
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SAMPLES = [
    "0, 1900, 2070, 900.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
    "0, 1950, 2070, 950.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
    "0, 2000, 2070, 1000.0, 0x0000000000000008, Active, Not Active, Not Active, Not Active",
    "0, [N/A], 2070, [N/A], 0x0, Not Active, Not Active, Not Active, Not Active",
]


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _fake_smi(tmp_path, lines):
    exe = tmp_path / "nvidia-smi"
    body = "".join(f"echo '{ln}'\n" for ln in lines)
    exe.write_text("#!/bin/sh\n" + body + "exec sleep 30\n")
    exe.chmod(exe.stat().st_mode | stat.S_IXUSR)
    return str(tmp_path)


def _sample(monkeypatch, tmp_path, lines):
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, lines) + os.pathsep + os.environ["PATH"])
    sampler = _bench().ClockSampler(0).start()
    time.sleep(0.5)
    return sampler.stop()


def test_median_clock_maxima_and_reasons(monkeypatch, tmp_path):
    rec = _sample(monkeypatch, tmp_path, SAMPLES)
    assert rec["samples"] == 4
    assert rec["sm_mhz"] == 1950.0  # median of the three numeric samples
    assert rec["sm_max_mhz"] == 2070.0
    assert rec["power_w_max"] == 1000.0
    assert rec["reasons"] == ["hw_slowdown", "sw_power_cap"]


def test_no_samples_is_reported(monkeypatch, tmp_path):
    rec = _sample(monkeypatch, tmp_path, [])
    assert rec["sm_mhz"] is None and rec["reasons"] == ["no samples"]


def test_traffic_record_is_keyed_on_the_kernel_sources(monkeypatch):
    bench = _bench()
    assert bench.profiled_traffic("bf16") is not None and bench.profiled_traffic("bf16") > 0
    assert bench.profiled_traffic("no-such-precision") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.profiled_traffic("bf16") is None


def _profile_commands():
    """Every `python bench.py ...` command line in the committed profile summaries (the
    backslash continuations joined)."""
    import glob
    out = []
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        text = open(path).read().replace("\\\n", " ")
        for line in text.splitlines():
            if "bench.py" not in line:
                continue
            for part in line.split("&&"):
                words = part.split()  # the commands quote nothing
                while words and words[0] != "python":
                    words.pop(0)  # drop an ncu prefix and its options
                if words[:2] == ["python", "bench.py"]:
                    out.append((os.path.basename(path), words[2:]))
    return out


def test_profile_commands_are_valid_bench_invocations(monkeypatch):
    """The commands the profile summaries were made with run committed files only and still
    parse with the benchmark's current options (warm-up and step rules included)."""
    cmds = _profile_commands()
    names = {name for name, _ in cmds}
    assert len(names) == len([p for p in os.listdir(os.path.join(ROOT, "profiles"))
                              if p.endswith(".md")])
    bench = _bench()
    for name, argv in cmds:
        monkeypatch.setattr("sys.argv", ["bench.py", *argv])
        bench.parse_args()  # exits (SystemExit) on an unknown flag or a broken rule


def test_clock_matched_fraction_and_peak_sources(monkeypatch, tmp_path):
    """The clock-matched fraction rescales the peak from the clock it was measured at to
    the run's clock; the tf32 peak comes from the measured record when present, else from
    the bf16 peak times the nominal ratio, and says which; unit-count peaks use the
    sampled clock, or the maximum clock when there are no samples."""
    b = _bench()
    assert b.clock_matched(0.98, 1725.0, 1462.0) == 0.98 * 1462.0 / 1725.0
    assert b.clock_matched(0.98, None, 1462.0) is None
    assert b.clock_matched(0.98, 1725.0, None) is None
    peaks = {"bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0,
             "clocks_under_load": {"sm_mhz_median": 1440.0}}
    assert b.peak_clock_mhz(peaks) == 1440.0
    assert b.peak_clock_mhz({}) is None
    monkeypatch.setattr(b, "TF32_PEAK_FILE", str(tmp_path / "absent.json"))
    pk, mhz, src = b.load_tf32_peak(peaks, "measured")
    assert pk == 1700.0 * 1.1 / 2.25 and mhz == 1440.0 and "nominal" in src
    rec = tmp_path / "tf32.json"
    rec.write_text('{"tf32_tflops_sustained": 900.0, "clocks_sustained": {"sm_mhz": 1500.0}}')
    monkeypatch.setattr(b, "TF32_PEAK_FILE", str(rec))
    pk, mhz, src = b.load_tf32_peak(peaks, "measured")
    assert pk == 900.0 and mhz == 1500.0 and "measured" in src
    hz, label = b.run_clock_hz({"sm_mhz": 1700.0}, peaks)
    assert hz == 1.7e9 and "sampled" in label
    hz, label = b.run_clock_hz({"sm_mhz": None}, peaks)
    assert hz == 2.07e9 and "maximum" in label
