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
    # the same workload description as the GPU arm's, key for key
    import workloads
    c = workloads.scene_case()
    want = bench.workload_config(c, line["config"]["tree_depth"], line["config"]["tree_nodes"], 1, 2, 1)
    assert line["config"] == want


def test_reference_tree_shape_is_the_librarys(oracle_mod):
    """The reference arm reports the oracle tree's depth and node count in the
    shared config; they equal the library's tree's (node-for-node builds)."""
    import icp_nearest_neighbour_gb300 as nn
    import workloads
    nn.load(build_if_missing=True)
    c = workloads.scene_case()
    info = nn.kdtree_info(nn.kdtree_build(c.target, c.leaf_size))
    ot = oracle_mod.KDTree(c.target, c.leaf_size)
    assert (info["depth"], info["n_nodes"]) == (ot.depth, ot.n_nodes)


def test_traffic_capture_is_used_only_for_the_kernel_it_measured(tmp_path, monkeypatch):
    import bench
    prof = tmp_path / "traffic.md"
    monkeypatch.setattr(bench, "TRAFFIC_PROFILE", str(prof))
    assert bench.measured_traffic()[0] is None
    prof.write_text("# capture\ntraffic: kernel_source_sha256_16=0123456789abcdef "
                    "dram_bytes_per_launch=4.1e6 lts_bytes_per_launch=2.0e8\n")
    got, why = bench.measured_traffic()
    assert got is None and "stale" in why
    prof.write_text(f"traffic: kernel_source_sha256_16={bench.kernel_source_hash()} "
                    "dram_bytes_per_launch=4.1e6 lts_bytes_per_launch=2.0e8\n")
    got, _ = bench.measured_traffic()
    assert got == {"dram_bytes": 4.1e6, "l2_bytes": 2.0e8}


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


def test_algorithmic_work_constants_follow_the_yardstick():
    """The bench divides the oracle's counted work by kernel time; its
    constants must be what the yardstick counts today (scene registration and
    the 1M x 1M mixture query)."""
    import bench
    from oracle import yardstick
    sc = yardstick.work("scene")
    assert abs(sc["bytes_per_query"] - bench.ICP_BYTES_PER_QUERY) < 0.01
    assert abs(sc["fp32_flops_per_query"] - bench.ICP_FP32_FLOPS_PER_QUERY) < 0.1
    g = yardstick.work("gmm")
    assert abs(g["bytes_per_query"] - bench.GMM_BYTES_PER_QUERY) < 0.01
    assert abs(g["fp32_flops_per_query"] - bench.GMM_FP32_FLOPS_PER_QUERY) < 0.1
