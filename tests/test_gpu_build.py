"""The device tree build (icpnn_kdtree_build_device) against the oracle's
tree and the host build: the same split axes, split values and leaf ranges
node for node, the same points in every leaf, and the same search results.

The tree of "Implementing ICP with CUDA-KDTree" (pwwt.cn/news/5235220),
sections 2.2, 2.3, 4.2 and 5.1: axis of largest variance (or round robin),
median split by (coordinate, index)."""
import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nn():
    import torch
    import icp_nearest_neighbour_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    m.load(build_if_missing=True)
    return m


def _leaf_sets(ex):
    out = []
    for i in range(len(ex["left"])):
        if ex["left"][i] < 0:
            out.append(sorted(ex["leaf_index"][ex["start"][i]:ex["end"][i]].tolist()))
    return out


def _clouds():
    rng = np.random.default_rng(131)
    g = W.grid_cloud(8, 0.5)
    centres = rng.uniform(-30, 30, (5, 3))
    clustered = W.gaussian_mixture(60_000, rng, centres, np.array([0.001, 0.01, 0.5, 2.0, 0.0001]))
    coarse = np.round(rng.normal(size=(50_000, 3)) * 4).astype(np.float32) * 0.25
    flat = np.c_[rng.uniform(-5, 5, (40_000, 2)), np.zeros(40_000)].astype(np.float32)
    same = np.tile(np.array([[0.1, -2.5, 7.0]], np.float32), (300, 1))
    signed_zero = np.zeros((500, 3), np.float32)
    signed_zero[::2, 0] = -0.0
    signed_zero[:, 1] = rng.uniform(-1, 1, 500)
    return {
        "uniform": (W.uniform_cloud(5000, 1), 8),
        "grid_ties": (g, 1),
        "duplicates": (np.vstack([g, g[:100], g[:100]]), 4),
        "single": (np.array([[1.0, 2.0, 3.0]], np.float32), 8),
        "two": (np.array([[1.0, 2.0, 3.0], [1.0, 2.0, 3.0]], np.float32), 1),
        "tiny_case": (W.tiny_case().target, 8),
        "scene100k": (W.scene_case().target, 12),
        "lidar": (W.lidar_case().target, 16),
        "clustered": (clustered, 10),
        "coarse_ties": (coarse, 4),
        "flat": (flat, 16),
        "all_same": (same, 4),
        "signed_zero": (signed_zero, 2),
    }


@pytest.mark.parametrize("round_robin", [False, True])
@pytest.mark.parametrize("name", list(_clouds()))
def test_device_tree_matches_oracle_tree(nn, oracle_mod, name, round_robin):
    pts, leaf = _clouds()[name]
    t = nn.kdtree_build_device(pts, leaf, round_robin=round_robin)
    o = oracle_mod.KDTree(pts, leaf, round_robin=round_robin)
    ex, oex = nn.kdtree_export(t), o.export()
    info = nn.kdtree_info(t)
    assert info["n_nodes"] == o.n_nodes and info["depth"] == o.depth
    for k in ("split_val", "split_dim", "left", "right", "start", "end"):
        np.testing.assert_array_equal(ex[k], oex[k], err_msg=k)
    assert _leaf_sets(ex) == _leaf_sets(oex)
    assert sorted(ex["leaf_index"].tolist()) == list(range(len(pts)))


@pytest.mark.parametrize("max_depth", [0, 3, 5])
def test_device_tree_depth_cap(nn, oracle_mod, max_depth):
    pts = W.uniform_cloud(3000, 4)
    t = nn.kdtree_build_device(pts, 1, max_depth=max_depth)
    o = oracle_mod.KDTree(pts, 1, max_depth=max_depth)
    ex, oex = nn.kdtree_export(t), o.export()
    assert nn.kdtree_info(t)["depth"] == max_depth
    for k in ("split_val", "split_dim", "left", "right", "start", "end"):
        np.testing.assert_array_equal(ex[k], oex[k], err_msg=k)
    assert _leaf_sets(ex) == _leaf_sets(oex)


def test_device_tree_from_device_memory_and_search(nn, oracle_mod):
    """A device-resident cloud, then exact queries on the tree without any
    host copy of it."""
    import torch
    c = W.scene_case(40_000, 20_000)
    t = nn.kdtree_build_device(torch.from_numpy(c.target).cuda(), 12)
    q = torch.from_numpy(c.source).cuda()
    idx = torch.empty(len(c.source), dtype=torch.int32, device="cuda")
    d2 = torch.empty(len(c.source), dtype=torch.float32, device="cuda")
    nn.nn_query(t, q, idx, d2, 1)
    torch.cuda.synchronize()
    i_o, d_o = oracle_mod.KDTree(c.target, 12).query(c.source)
    np.testing.assert_array_equal(idx.cpu().numpy(), i_o)
    np.testing.assert_array_equal(d2.cpu().numpy().view(np.uint32), d_o.view(np.uint32))


def test_registration_on_device_tree_equals_host_tree(nn):
    """The same tree gives the same registration, bit for bit."""
    import torch
    c = W.scene_case(60_000, 60_000)
    th = nn.kdtree_build(c.target, 12)
    nn.kdtree_upload(th)
    td = nn.kdtree_build_device(c.target, 12)
    src = torch.from_numpy(c.source).cuda()
    rh = nn.icp_align(th, src, 30, 1e-5, 1.0, trace=True)
    rd = nn.icp_align(td, src, 30, 1e-5, 1.0, trace=True)
    assert rh["iters"] == rd["iters"]
    np.testing.assert_array_equal(rh["T"], rd["T"])
    assert rh["final_mse"] == rd["final_mse"]
    for a, b in zip(rh["trace"], rd["trace"]):
        np.testing.assert_array_equal(a["T"], b["T"])
        assert a["mse"] == b["mse"] and a["n_accepted"] == b["n_accepted"]


def test_device_build_errors(nn):
    pts = W.uniform_cloud(1000, 2)
    bad = pts.copy()
    bad[317, 2] = np.inf
    with pytest.raises(nn.IcpnnError) as e:
        nn.kdtree_build_device(bad, 8)
    assert e.value.status == "NONFINITE" and "317" in str(e.value)
    for args, status in [((pts, 0), "INVALID_ARG"), ((pts, 65), "INVALID_ARG"), ((pts, 8, 21), "TREE_DEPTH")]:
        with pytest.raises(nn.IcpnnError) as e:
            nn.kdtree_build_device(*args)
        assert e.value.status == status


def test_device_tree_uploads_to_host_copy_on_demand(nn, oracle_mod):
    """Export after a device build fetches the host copy; a second export and
    an upload on the same device change nothing."""
    pts = W.uniform_cloud(20000, 17)
    t = nn.kdtree_build_device(pts, 12)
    ex1 = nn.kdtree_export(t)
    nn.kdtree_upload(t)
    ex2 = nn.kdtree_export(t)
    for k in ex1:
        np.testing.assert_array_equal(ex1[k], ex2[k])


def test_l2_probe_runs_and_checks_its_arguments(nn):
    import torch
    x = torch.ones(1 << 20, dtype=torch.float32, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    nn.probe_l2_read(x, 4, sink)
    torch.cuda.synchronize()
    assert int(sink.item()) == 0
    with pytest.raises(nn.IcpnnError):
        nn.probe_l2_read(x[:3], 1, sink)      # 12 bytes: not a multiple of 16


def test_device_tree_matches_host_tree_at_4M_points(nn):
    """The large workload's 4M-point target (leaf 16, depth 18): device build
    against the host build, node for node (two independent implementations;
    the host build is pinned to the oracle on the smaller clouds)."""
    c = W.large_case()
    th = nn.kdtree_build(c.target, c.leaf_size)
    td = nn.kdtree_build_device(c.target, c.leaf_size)
    eh, ed = nn.kdtree_export(th), nn.kdtree_export(td)
    for k in ("split_val", "split_dim", "left", "right", "start", "end"):
        np.testing.assert_array_equal(ed[k], eh[k], err_msg=k)
    # same point sets per leaf: indices sorted within each leaf's range
    leaves = np.flatnonzero(eh["left"] < 0)
    order = np.argsort(eh["start"][leaves])
    sizes = (eh["end"] - eh["start"])[leaves][order]
    leaf_of_pos = np.repeat(np.arange(len(leaves)), sizes)
    assert len(leaf_of_pos) == len(c.target)
    def per_leaf_sorted(li):
        return li[np.lexsort((li, leaf_of_pos))]
    np.testing.assert_array_equal(per_leaf_sorted(ed["leaf_index"]), per_leaf_sorted(eh["leaf_index"]))
