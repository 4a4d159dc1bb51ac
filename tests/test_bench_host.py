"""bench.py's host-side pieces that need no GPU: the reference arm (the CPU
oracle timed on a bounded sample) prints the contract's JSON line, and the
oracle sample runs on FP8 rows as on bf16 rows."""
import json

from synth import workloads as W


def test_reference_arm_prints_the_contract_line(capsys):
    import bench
    bench.main(["--impl", "reference", "--workload", "resolve", "--steps", "2", "--warmup", "1"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "rows/s" and line["value"] > 0
    assert line["higher_is_better"] is True and line["steps"] == 2 and line["warmup"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "rows/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_oracle_sample_on_both_row_formats():
    import bench
    w = W.make("tiny")
    for fp8 in (False, True):
        rows, secs, steps = bench.oracle_sample(w, seconds=1e9, units=1, steps_cap=3, skip=1,
                                                fp8=fp8)
        assert steps == 2 and rows == 2 * w.K and secs > 0


def test_clock_sampler_summarises_samples_and_throttle_reasons(tmp_path):
    """The clocks record: median SM clock under load, the maximum, and every
    throttle reason seen Active (from nvidia-smi's CSV, here written by hand)."""
    import bench

    class _Done:  # stands in for the nvidia-smi process
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    csv = tmp_path / "clocks.csv"
    csv.write_text(
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n"
        "0, 1980, 2070, 1390.5, 0x4, Not Active, Not Active, Not Active, Active\n"
        "0, 2070, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
        "garbled line\n")
    s = bench.ClockSampler(0)
    s.proc, s.path = _Done(), str(csv)
    rec = s.stop()
    assert rec == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "samples": 3,
                   "reasons": ["sw_power_cap"]}
    assert not csv.exists()  # the sample file is removed


def test_clock_sampler_without_nvidia_smi_says_so():
    import bench
    s = bench.ClockSampler(0)
    s.wait_ready(timeout_s=0.01)  # no process: returns at once (plus its short settle)
    assert s.stop() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
