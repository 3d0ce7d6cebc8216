"""The benchmark's native line on a GPU, at a small row count: one JSON line with every key the
contract asks for, the dominant kernel's roofline against the measured peak, and the end-to-end
and CPU-baseline legs filled in."""
import json

import pytest

import bench

pytestmark = pytest.mark.gpu


def test_native_line_keeps_the_contract(capsys):
    rc = bench.main(["--rows", "65536", "--steps", "3", "--warmup", "3", "--no-fp8", "--no-dgrad", "--no-gateup",
                     "--no-adam", "--cpu-seconds", "1"])
    assert rc == 0
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "clocks",
                "gpu_launches"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 3 and line["warmup"] == 3 and line["value"] > 0
    assert line["gpu_launches"] == 2 * 3                   # fwd + bwd per timed step
    rf = line["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and 0 < rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"])
    e2e = line["e2e"]
    assert e2e["h2d_bytes_per_step"] == 65536 * (4 * 3072 + 2 * 3072 + 4)
    assert e2e["d2h_bytes_per_step"] == 65536 * (2 * 3072 + 4 * 3072 + 4)
    assert 0 < e2e["value"] < line["value"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(line["clocks"])
