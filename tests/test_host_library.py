"""CPU-only checks of libicpnn: it loads, exports every symbol the header
declares, and its host parts (tree build, Kabsch solve, argument checking)
match the oracle.  No GPU is touched here."""
import math
import os
import re

import numpy as np
import pytest

import workloads as W
from conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    import icp_nearest_neighbour_gb300 as nn
    nn.load(build_if_missing=True)
    return nn


def test_library_exports_every_declared_symbol(lib):
    import glob
    header = "".join(open(h).read() for h in sorted(glob.glob(os.path.join(ROOT, "include", "*.h"))))
    declared = set(re.findall(r"\b(icpnn_[a-z_0-9]+)\s*\(", header))
    assert {"icpnn_kdtree_build", "icpnn_kdtree_build_device", "icpnn_kdtree_upload", "icpnn_nn_query",
            "icpnn_icp_align", "icpnn_probe_l2_read"} <= declared
    handle = lib.load()
    for name in sorted(declared):
        assert hasattr(handle, name), name
    assert handle.icpnn_version() >= 100


def _leaf_sets(ex):
    out = []
    for i in range(len(ex["left"])):
        if ex["left"][i] < 0:
            out.append(sorted(ex["leaf_index"][ex["start"][i]:ex["end"][i]].tolist()))
    return out


def _tree_clouds():
    rng = np.random.default_rng(31)
    g = W.grid_cloud(8, 0.5)
    return {
        "uniform": (W.uniform_cloud(5000, 1), 8),
        "grid_ties": (g, 1),
        "duplicates": (np.vstack([g, g[:100], g[:100]]), 4),
        "flat": (np.c_[rng.uniform(-1, 1, (3000, 2)), np.zeros(3000)].astype(np.float32), 12),
        "single": (np.array([[1.0, 2.0, 3.0]], np.float32), 8),
        "scene": (W.scene_case(20_000, 10).target, 12),
        "tiny_case": (W.tiny_case().target, 8),
        # the root's variance is first summed about the first point: far from
        # the rest it leaves too little precision and the sum is taken again
        "outlier_first": (np.vstack([[[4e4, -3e4, 2e4]], W.uniform_cloud(3000, 5)]).astype(np.float32), 8),
        "all_same": (np.tile(np.float32([[0.3, -1.7, 2.5]]), (200, 1)), 4),
        "two_flat_axes": (np.c_[rng.uniform(-1, 1, 2000), np.full(2000, 0.7), np.full(2000, -2.0)].astype(np.float32), 6),
    }


@pytest.mark.parametrize("name", list(_tree_clouds()))
def test_tree_matches_oracle_tree(lib, oracle_mod, name):
    pts, leaf = _tree_clouds()[name]
    t = lib.kdtree_build(pts, leaf)
    o = oracle_mod.KDTree(pts, leaf)
    ex, oex = lib.kdtree_export(t), o.export()
    info = lib.kdtree_info(t)
    assert info["n_nodes"] == o.n_nodes and info["depth"] == o.depth
    for k in ("split_val", "split_dim", "left", "right", "start", "end"):
        np.testing.assert_array_equal(ex[k], oex[k], err_msg=k)
    # which points share a leaf is unique; their order inside a leaf is not
    assert _leaf_sets(ex) == _leaf_sets(oex)
    assert sorted(ex["leaf_index"].tolist()) == list(range(len(pts)))


@pytest.mark.parametrize("name", ["uniform", "grid_ties", "flat", "scene"])
def test_round_robin_tree_matches_oracle_tree(lib, oracle_mod, name):
    pts, leaf = _tree_clouds()[name]
    t = lib.kdtree_build(pts, leaf, round_robin=True)
    o = oracle_mod.KDTree(pts, leaf, round_robin=True)
    ex, oex = lib.kdtree_export(t), o.export()
    for k in ("split_val", "split_dim", "left", "right", "start", "end"):
        np.testing.assert_array_equal(ex[k], oex[k], err_msg=k)
    assert _leaf_sets(ex) == _leaf_sets(oex)


def _big_tree_clouds():
    """Clouds large enough that the top nodes are split chunk-parallel and by
    binned selection, with the distributions that stress it: surface samples,
    tight clusters (most of a node in one bin), heavy coordinate ties, and a
    zero-spread axis."""
    rng = np.random.default_rng(77)
    centres = rng.uniform(-30, 30, (5, 3))
    clustered = W.gaussian_mixture(90_000, rng, centres, np.array([0.001, 0.01, 0.5, 2.0, 0.0001]))
    coarse = np.round(rng.normal(size=(70_000, 3)) * 4).astype(np.float32) * 0.25
    flat = np.c_[rng.uniform(-5, 5, (60_000, 2)), np.zeros(60_000)].astype(np.float32)
    return {
        "scene100k": (W.scene_case().target, 12),
        "lidar": (W.lidar_case().target, 8),
        "clustered": (clustered, 10),
        "coarse_ties": (coarse, 4),
        "flat": (flat, 16),
    }


@pytest.mark.parametrize("round_robin", [False, True])
@pytest.mark.parametrize("name", list(_big_tree_clouds()))
def test_large_tree_matches_oracle_tree(lib, oracle_mod, name, round_robin):
    pts, leaf = _big_tree_clouds()[name]
    t = lib.kdtree_build(pts, leaf, round_robin=round_robin)
    o = oracle_mod.KDTree(pts, leaf, round_robin=round_robin)
    ex, oex = lib.kdtree_export(t), o.export()
    for k in ("split_val", "split_dim", "left", "right", "start", "end"):
        np.testing.assert_array_equal(ex[k], oex[k], err_msg=k)
    assert _leaf_sets(ex) == _leaf_sets(oex)
    # repeated builds give the same leaf order, whatever the thread timing
    np.testing.assert_array_equal(lib.kdtree_export(lib.kdtree_build(pts, leaf, round_robin=round_robin))
                                  ["leaf_index"], ex["leaf_index"])


def test_concurrent_builds_give_the_same_tree(lib):
    """Several host threads build at once: their parallel regions share the
    library's worker pool (nested, interleaved) and every tree still comes
    out the same, leaf order included."""
    import threading
    pts = W.scene_case(60_000, 3).target
    ref = lib.kdtree_export(lib.kdtree_build(pts, 12))
    errors = []

    def worker():
        try:
            for _ in range(6):
                ex = lib.kdtree_export(lib.kdtree_build(pts, 12))
                for k in ("split_val", "split_dim", "start", "end", "leaf_index"):
                    np.testing.assert_array_equal(ex[k], ref[k], err_msg=k)
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(e)

    threads = [threading.Thread(target=worker) for _ in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors[0]


def test_builds_of_changing_sizes_reuse_host_blocks_safely(lib):
    """The tree's host arrays come from a cache of freed blocks, handed out
    again to requests they can hold: trees of alternating sizes, built and
    freed in turn, must come out exactly as the first build of each size."""
    small = W.uniform_cloud(1500, 11)
    big = W.scene_case(40_000, 3).target
    ref = {k: lib.kdtree_export(lib.kdtree_build(c, 8)) for k, c in (("s", small), ("b", big))}
    for _ in range(4):
        for k, c in (("b", big), ("s", small), ("s", small), ("b", big)):
            t = lib.kdtree_build(c, 8)
            ex = lib.kdtree_export(t)
            for f in ("split_val", "split_dim", "start", "end", "leaf_index"):
                np.testing.assert_array_equal(ex[f], ref[k][f], err_msg=f)
            t.free()


def test_tree_depth_cap(lib, oracle_mod):
    pts = W.uniform_cloud(3000, 4)
    t = lib.kdtree_build(pts, 1, max_depth=5)
    o = oracle_mod.KDTree(pts, 1, max_depth=5)
    assert lib.kdtree_info(t)["depth"] == 5
    assert _leaf_sets(lib.kdtree_export(t)) == _leaf_sets(o.export())


def test_tree_build_rejects_bad_input(lib):
    pts = W.uniform_cloud(100, 2)
    for args, status in [((pts, 0), "INVALID_ARG"), ((pts, 65), "INVALID_ARG"),
                         ((pts, 8, 21), "TREE_DEPTH"), ((np.zeros((0, 3), np.float32), 8), "INVALID_ARG")]:
        with pytest.raises(lib.IcpnnError) as e:
            lib.kdtree_build(*args)
        assert e.value.status == status
    bad = pts.copy()
    bad[17, 1] = np.nan
    with pytest.raises(lib.IcpnnError) as e:
        lib.kdtree_build(bad, 8)
    assert e.value.status == "NONFINITE" and "17" in str(e.value)
    bad[17, 1] = np.inf
    with pytest.raises(lib.IcpnnError):
        lib.kdtree_build(bad, 8)


def test_device_build_checks_arguments_before_touching_a_device(lib):
    """icpnn_kdtree_build_device validates like the host build, before any CUDA call."""
    pts = W.uniform_cloud(100, 2)
    for args, status in [((pts, 0), "INVALID_ARG"), ((pts, 65), "INVALID_ARG"),
                         ((pts, 8, 21), "TREE_DEPTH"), ((np.zeros((0, 3), np.float32), 8), "INVALID_ARG")]:
        with pytest.raises(lib.IcpnnError) as e:
            lib.kdtree_build_device(*args)
        assert e.value.status == status


def _moments_from_pairs(S, Q):
    S = np.asarray(S, np.float64)
    Q = np.asarray(Q, np.float64)
    mu_s, mu_q = S.mean(0), Q.mean(0)
    return {"n_accepted": len(S), "mu_src": mu_s, "mu_tgt": mu_q, "H": (S - mu_s).T @ (Q - mu_q)}


def test_kabsch_matches_oracle_on_random_pairs(lib, oracle_mod):
    rng = np.random.default_rng(41)
    for trial in range(50):
        n = int(rng.integers(3, 400))
        S = rng.normal(size=(n, 3)) * rng.uniform(0.1, 30, size=3)
        R_true = W.axis_angle_matrix(W.random_unit_vector(rng), rng.uniform(0, math.pi))
        Q = S @ R_true.T + rng.normal(size=3) * 5 + rng.normal(size=(n, 3)) * rng.uniform(0, 2)
        if trial % 5 == 0:
            Q[:, 0] = -Q[:, 0]                       # mirrored: exercises the reflection guard
        T = lib.kabsch(_moments_from_pairs(S, Q))
        R_o, t_o, _ = oracle_mod.kabsch(S, Q)
        np.testing.assert_allclose(T[:3, :3], R_o, atol=1e-9)
        np.testing.assert_allclose(T[:3, 3], t_o, atol=1e-9 * (1 + np.abs(t_o).max()))
        assert abs(np.linalg.det(T[:3, :3]) - 1) < 1e-12
        np.testing.assert_array_equal(T[3], [0, 0, 0, 1])


@pytest.mark.parametrize("case", ["A", "B"])
def test_kabsch_hand_fixture(lib, case):
    from conftest import read_fixture
    rows = read_fixture("kabsch_hand.txt")
    pairs = np.array([[float(v) for v in r[2:8]] for r in rows if r[0] == "pair" and r[1] == case])
    exp = np.array([float(v) for v in [r for r in rows if r[0] == "expect" and r[1] == case][0][2:]])
    T = lib.kabsch(_moments_from_pairs(pairs[:, :3], pairs[:, 3:]))
    np.testing.assert_allclose(T[:3, :3], exp[:9].reshape(3, 3), atol=1e-12)
    np.testing.assert_allclose(T[:3, 3], exp[9:], atol=1e-12)


def test_kabsch_degenerate(lib):
    with pytest.raises(lib.IcpnnError) as e:
        lib.kabsch({"n_accepted": 2, "mu_src": np.zeros(3), "mu_tgt": np.zeros(3), "H": np.eye(3)})
    assert e.value.status == "DEGENERATE"
    line = np.outer(np.arange(10.0), [1.0, 2.0, 3.0])
    with pytest.raises(lib.IcpnnError) as e:
        lib.kabsch(_moments_from_pairs(line, line + 1))
    assert e.value.status == "DEGENERATE"


def test_probe_entry_points_check_arguments_without_a_device(lib):
    """The test helpers behind the pre-launched passes validate on the host:
    the command-delay and collect-delay injectors take their settings (and
    are switched off again), the command-wait probe needs an uploaded tree."""
    for probe in (lib.probe_delay_commands, lib.probe_delay_collect):
        for bad in ((-1, 1, 0), (0, -1, 0), (0, 1, 10_000_000_001)):
            with pytest.raises(lib.IcpnnError) as e:
                probe(*bad)
            assert e.value.status == "INVALID_ARG"
        probe(2, 1, 1000)
        probe(0, 0, 0)
    t = lib.kdtree_build(W.uniform_cloud(100, 3), 8)
    with pytest.raises(lib.IcpnnError) as e:
        lib.probe_command_wait(t, W.uniform_cloud(10, 4), 1_000_000, 0)
    assert e.value.status == "NOT_UPLOADED"
    assert lib.NO_PRELAUNCH == 16


def test_query_without_upload_is_an_error(lib):
    t = lib.kdtree_build(W.uniform_cloud(100, 3), 8)
    q = W.uniform_cloud(10, 4)
    with pytest.raises(lib.IcpnnError) as e:
        lib.nn_query(t, q, np.empty(10, np.int32), np.empty(10, np.float32))
    assert e.value.status == "NOT_UPLOADED"
    with pytest.raises(lib.IcpnnError) as e:
        lib.icp_align(t, q, 5, 1e-6)
    assert e.value.status == "NOT_UPLOADED"
    with pytest.raises(lib.IcpnnError) as e:
        lib.icp_align(t, q, 5, 1e-6, prelaunch=False)
    assert e.value.status == "NOT_UPLOADED"


def test_product_path_has_no_oracle_or_fallback():
    """The package must not import the oracle, and must fail loudly without its
    compiled library (no CPU fallback)."""
    pkg = os.path.join(ROOT, "icp_nearest_neighbour_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cpp", ".h", ".cuh")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"\boracle\b", text.replace("the oracle", "")), f
    src = open(os.path.join(pkg, "__init__.py")).read()
    assert "raise RuntimeError" in src
