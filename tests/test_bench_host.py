"""Host-side pieces of bench.py on CPU: the clock-record parser, the choice
of FP8 peak, the staleness rule of the recorded DRAM traffic, the
threaded oracle runner, and the host-link ceiling of the end-to-end leg."""
import json
import threading

import pytest

import bench


def _sampler(lines):
    c = bench.ClockSampler("0")
    c.lines = lines
    return c.summary()


def test_clock_summary_uses_loaded_samples_and_reports_throttle_reasons():
    idle = "1500, 2070, 120.5, Not Active, Not Active, Not Active, Not Active"
    busy = "2070, 2070, 950.0, Not Active, Not Active, Not Active, Not Active"
    capped = "1605, 2070, 1390.0, Not Active, Not Active, Not Active, Active"
    s = _sampler([idle, busy, busy, capped, "garbage", "1, 2, three, a, b, c, d"])
    assert s["samples"] == 3                      # the idle sample is not "under load"
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    assert s["power_w_max"] == 1390.0
    hot = "1800, 2070, 1000.0, Active, Not Active, Active, Not Active"
    assert _sampler([hot])["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert _sampler([]) is None
    # no sample above the load threshold: all samples count
    assert _sampler([idle])["samples"] == 1


def test_fp8_peak_burst_and_sustained(tmp_path, monkeypatch):
    peaks = tmp_path / "peaks.json"
    peaks.write_text(json.dumps({"bf16_tflops": 1932.5, "bf16_tflops_sustained": 1759.5}))
    monkeypatch.setattr(bench, "PEAKS_FILE", str(peaks))
    assert bench.fp8_peak(sustained=False) == (3865.0, "measured bf16_tflops x 2")
    assert bench.fp8_peak(sustained=True) == (3519.0, "measured bf16_tflops_sustained x 2")
    monkeypatch.setattr(bench, "PEAKS_FILE", str(tmp_path / "absent.json"))
    assert bench.fp8_peak(sustained=False)[1].startswith("fallback")


def test_recorded_traffic_is_dropped_when_the_kernel_sources_change(tmp_path, monkeypatch):
    rec = tmp_path / "traffic.json"
    key = "dequant_1x128_bf16"
    rec.write_text(json.dumps({key: {"dram_bytes_per_launch": 123, "sources_sha": bench.sources_sha(key)}}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(rec))
    assert bench.measured_traffic(key) == 123
    rec.write_text(json.dumps({key: {"dram_bytes_per_launch": 123, "sources_sha": "0" * 16}}))
    assert bench.measured_traffic(key) is None
    assert bench.measured_traffic("no_such_kernel") is None


def test_oracle_parallel_runs_exactly_the_requested_steps():
    class Counter:
        def __init__(self):
            self.n, self.lock, self.threads = 0, threading.Lock(), set()

        def run(self):
            with self.lock:
                self.n += 1
                self.threads.add(threading.get_ident())

    c = Counter()
    runs, el = bench.oracle_parallel(c, 4, reps=37)
    assert runs == 37 and c.n == 37 and el >= 0.0
    c2 = Counter()
    runs, el = bench.oracle_parallel(c2, 3, seconds=0.05)
    assert runs == c2.n >= 1 and el >= 0.05


def test_cpu_model_names_x86_and_arm_hosts():
    x86 = "processor\t: 0\nvendor_id\t: GenuineIntel\nmodel name\t: Intel(R) Xeon(R) Platinum 8480+\n"
    assert bench.cpu_model(x86) == "Intel(R) Xeon(R) Platinum 8480+"
    grace = "processor\t: 0\nBogoMIPS\t: 2000.00\nCPU implementer\t: 0x41\nCPU architecture: 8\nCPU part\t: 0xd4f\n"
    assert bench.cpu_model(grace) == "Arm Neoverse-V2"
    other = "CPU implementer\t: 0x61\nCPU part\t: 0x023\n"
    assert bench.cpu_model(other) == "implementer 0x61 part 0x023"
    assert bench.cpu_model("") == "unknown"
    assert isinstance(bench.cpu_model(), str)


def test_reference_arm_prints_one_complete_line(monkeypatch, capsys):
    """`bench.py --impl reference` at rank 0: the CPU oracle on the bounded
    sample of the step, one JSON line with the contract's keys."""
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    assert bench.main(["--impl", "reference", "--steps", "2", "--warmup", "1"]) == 0
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 2
    assert d["config"]["workload"] == bench.WORKLOAD
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["sample"] and cb["cpu_model"]
    # every step runs one sample on each of the threads it reports
    assert cb["cores"] == bench._oracle_threads()
    assert d["config"]["sample_bytes_per_step"] == bench.OracleSample().bytes * cb["cores"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_link_ceiling_two_phase():
    """Both directions share the link at half its concurrent rate until the
    smaller transfer ends; the rest of the larger one runs at its one-way
    rate; the result is the step's bytes over that time."""
    import bench
    # 10 GB up and 20 GB down, 50 GB/s each while both run, then 10 GB down
    # alone at 50 GB/s: 0.2 s + 0.2 s for a 30 GB step
    assert bench.link_ceiling(30e9, 10e9, 20e9, 100.0, 50.0, 100.0) == pytest.approx(75.0)
    # the upload is the larger one: its rest runs at the upload rate
    # (0.2 s shared + 10 GB at 25 GB/s = 0.6 s)
    assert bench.link_ceiling(30e9, 20e9, 10e9, 25.0, 400.0, 100.0) == pytest.approx(50.0)
    # equal transfers never leave the shared phase
    assert bench.link_ceiling(2e9, 1e9, 1e9, 999.0, 999.0, 100.0) == pytest.approx(100.0)


def test_host_memory_available_and_the_e2e_check(tmp_path):
    """MemAvailable, capped by what a cgroup limit leaves; e2e runs only when
    every local rank's pinned buffers fit in 60% of it."""
    import bench
    meminfo = "MemTotal:       500000000 kB\nMemAvailable:   400000000 kB\n"
    lim, cur = tmp_path / "memory.max", tmp_path / "memory.current"
    lim.write_text("max\n")
    cur.write_text("123\n")
    assert bench.host_memory_available(meminfo, (str(lim), str(cur))) == 400000000 * 1024
    lim.write_text(str(100 * 2 ** 30) + "\n")
    cur.write_text(str(40 * 2 ** 30) + "\n")
    assert bench.host_memory_available(meminfo, (str(lim), str(cur))) == 60 * 2 ** 30
    assert bench.host_memory_available("", (str(tmp_path / "none"), str(cur))) is None
    assert isinstance(bench.host_memory_available(), (int, type(None)))
    step = 50.3e9  # the benchmark step's pinned inputs and results
    assert bench.e2e_fits(step, 1, 400e9)
    assert not bench.e2e_fits(step, 8, 400e9)
    assert bench.e2e_fits(step, 8, None)
