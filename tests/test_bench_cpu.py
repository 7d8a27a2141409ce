"""bench.py on the host: the reference arm's JSON line (the oracle timed on
the host cores, the fields the benchmark contract names) and argument checks.
No GPU is touched."""
import json

import pytest


def test_reference_arm_prints_one_contract_line(capsys):
    import bench
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0", "--ref-iters", "1"])
    lines = [ln for ln in capsys.readouterr().out.strip().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["higher_is_better"] is True and line["n_gpus"] == 1 and line["steps"] == 1
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"] == bench.WORKLOAD


def test_own_arm_rejects_fewer_than_three_warmup_steps():
    import bench
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_no_prelaunch_switch_is_accepted_by_the_parser(monkeypatch):
    import bench
    seen = {}
    monkeypatch.setattr(bench, "run_ours", lambda args: seen.setdefault("args", args) and None)
    bench.main(["--no-prelaunch", "--steps", "1", "--warmup", "3"])
    assert seen["args"].no_prelaunch is True and seen["args"].steps == 1
