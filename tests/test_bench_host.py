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
