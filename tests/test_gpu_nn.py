"""GPU parity of the nearest-neighbour query (icpnn_nn_query) against the
oracle: indices and squared distances must be bit-identical.

The exact nearest neighbour of "Implementing ICP with CUDA-KDTree"
(pwwt.cn/news/5235220), section 3.2, with ties resolved to the lowest index.
"""
import numpy as np
import pytest

import workloads as W
from conftest import read_fixture

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nn():
    import torch
    import icp_nearest_neighbour_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    m.load(build_if_missing=True)
    return m


def gpu_nn(nn, tree, q, flags=1, host=False):
    import torch
    q = np.ascontiguousarray(q, np.float32).reshape(-1, 3)
    n = len(q)
    if host:
        idx = np.full(n, -7, np.int32)
        d2 = np.full(n, -7.0, np.float32)
        nn.nn_query(tree, q, idx, d2, flags)
        return idx, d2
    qd = torch.from_numpy(q).cuda()
    idx = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    d2 = torch.full((n,), -7.0, dtype=torch.float32, device="cuda")
    nn.nn_query(tree, qd, idx, d2, flags)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), d2.cpu().numpy()


def assert_nn_equal(idx_g, d2_g, idx_o, d2_o):
    np.testing.assert_array_equal(idx_g, idx_o)
    nan_g, nan_o = np.isnan(d2_g), np.isnan(d2_o)
    np.testing.assert_array_equal(nan_g, nan_o)
    np.testing.assert_array_equal(d2_g[~nan_g].view(np.uint32), d2_o[~nan_o].view(np.uint32))


def make_tree(nn, pts, leaf, max_depth=-1):
    t = nn.kdtree_build(pts, leaf, max_depth)
    nn.kdtree_upload(t)
    return t


@pytest.mark.parametrize("leaf", [1, 2, 8])
def test_hand_fixture(nn, leaf):
    rows = read_fixture("nn_hand.txt")
    tgt = np.array([[float(v) for v in r[2:5]] for r in rows if r[0] == "target"], np.float32)
    q = np.array([[float(v) for v in r[1:4]] for r in rows if r[0] == "query"], np.float32)
    exp_idx = np.array([int(r[5]) for r in rows if r[0] == "query"], np.int32)
    exp_d2 = np.array([float(r[6]) for r in rows if r[0] == "query"], np.float32)
    t = make_tree(nn, tgt, leaf)
    for flags in (0, 1):
        idx, d2 = gpu_nn(nn, t, q, flags)
        assert_nn_equal(idx, d2, exp_idx, exp_d2)


def _clouds():
    rng = np.random.default_rng(3)
    g = W.grid_cloud(9, 0.5, origin=(-2.0, -2.0, -2.0))
    q_lat = W.grid_cloud(17, 0.25, origin=(-2.0, -2.0, -2.0))
    dup = np.vstack([g, g[rng.permutation(len(g))[:200]]])
    clustered = W.gaussian_mixture(6000, rng, rng.uniform(-5, 5, (6, 3)), rng.uniform(0.05, 0.5, 6))
    flat = W.uniform_cloud(4000, 5)
    flat[:, 2] = 0.0
    line = np.zeros((300, 3), np.float32)
    line[:, 0] = np.repeat(np.arange(100, dtype=np.float32), 3)
    return {
        "grid": (g, q_lat),
        "dup": (dup, q_lat),
        "clustered": (clustered, W.uniform_cloud(9000, 9, -6, 6)),
        "flat": (flat, W.uniform_cloud(5000, 13)),
        "line": (line, W.uniform_cloud(3000, 17, -5, 105)),
        "far_queries": (W.uniform_cloud(3000, 19), W.uniform_cloud(2000, 20, 50, 60)),
    }


@pytest.mark.parametrize("name", list(_clouds()))
@pytest.mark.parametrize("leaf", [1, 8, 16, 64])
def test_tie_heavy_clouds_match_brute_force(nn, oracle_mod, name, leaf):
    ref, q = _clouds()[name]
    t = make_tree(nn, ref, leaf)
    i_o, d_o = oracle_mod.nn_brute(ref, q)
    for flags in (0, 1):
        assert_nn_equal(*gpu_nn(nn, t, q, flags), i_o, d_o)


@pytest.mark.parametrize("nq", [1, 2, 31, 33, 255, 257, 2047, 2049, 65537])
def test_ragged_query_counts(nn, oracle_mod, nq):
    ref = W.uniform_cloud(20000, 101)
    q = W.uniform_cloud(nq, 102 + nq, -1.2, 1.2)
    t = make_tree(nn, ref, 12)
    ot = oracle_mod.KDTree(ref, 12)
    i_o, d_o = ot.query(q)
    for flags in (0, 1):
        assert_nn_equal(*gpu_nn(nn, t, q, flags), i_o, d_o)


def test_edge_cases(nn, oracle_mod):
    # single-point tree
    one = np.array([[0.5, -1.0, 2.0]], np.float32)
    t1 = make_tree(nn, one, 8)
    q = W.uniform_cloud(1000, 3)
    assert_nn_equal(*gpu_nn(nn, t1, q), *oracle_mod.nn_brute(one, q))
    # depth-capped tree: leaves of ~n/8 points
    ref = W.uniform_cloud(5000, 4)
    t2 = make_tree(nn, ref, 1, max_depth=3)
    assert nn.kdtree_info(t2)["depth"] == 3
    assert_nn_equal(*gpu_nn(nn, t2, q), *oracle_mod.nn_brute(ref, q))
    # depth 0: the whole cloud in one leaf
    t3 = make_tree(nn, ref[:64], 64)
    assert nn.kdtree_info(t3)["depth"] == 0
    assert_nn_equal(*gpu_nn(nn, t3, q), *oracle_mod.nn_brute(ref[:64], q))
    # non-finite queries match nothing; finite neighbours are unaffected
    qb = q.copy()
    qb[5, 0] = np.nan
    qb[6, 2] = np.inf
    qb[7, 1] = -np.inf
    idx, d2 = gpu_nn(nn, t2, qb)
    assert (idx[5:8] == -1).all() and np.isnan(d2[5:8]).all()
    assert_nn_equal(idx, d2, *oracle_mod.nn_brute(ref, qb))
    # queries on the target points themselves: d2 = 0, lowest duplicate index
    dup = np.vstack([ref, ref[::7]])
    t4 = make_tree(nn, dup, 8)
    idx, d2 = gpu_nn(nn, t4, dup)
    assert (d2 == 0).all()
    expect = np.arange(len(dup))
    expect[len(ref):] = np.arange(0, len(ref), 7)
    np.testing.assert_array_equal(idx, expect)
    # n = 0 is a no-op
    import torch
    e = torch.empty((0, 3), dtype=torch.float32, device="cuda")
    nn.nn_query(t2, e, torch.empty(0, dtype=torch.int32, device="cuda"),
                torch.empty(0, dtype=torch.float32, device="cuda"))


def test_host_and_device_buffers_agree(nn, oracle_mod):
    ref = W.uniform_cloud(30000, 6)
    q = W.uniform_cloud(20000, 7)
    t = make_tree(nn, ref, 12)
    i_h, d_h = gpu_nn(nn, t, q, host=True)
    i_d, d_d = gpu_nn(nn, t, q, host=False)
    assert_nn_equal(i_h, d_h, i_d, d_d)
    assert_nn_equal(i_h, d_h, *oracle_mod.nn_brute(ref, q))


def test_kernels_actually_launch(nn):
    before = nn.launch_count()
    ref = W.uniform_cloud(5000, 8)
    t = make_tree(nn, ref, 8)
    gpu_nn(nn, t, W.uniform_cloud(3000, 9), flags=1)
    assert nn.launch_count() - before >= 4   # bbox, Morton, sort passes, gather, search


# --------------------------------------------------------- full workloads ---

def _full_query_case(name):
    if name == "gmm":
        c = W.gmm_case()
        return c.reference, c.queries, c.leaf_size
    c = W.CASES[name]()
    return c.target, c.source, c.leaf_size


@pytest.mark.parametrize("name", ["tiny", "scene", "lidar", "gmm"])
def test_full_workloads_every_query(nn, oracle_mod, name):
    """Every query of the full-size workloads, in both orders."""
    ref, q, leaf = _full_query_case(name)
    t = make_tree(nn, ref, leaf)
    ot = oracle_mod.KDTree(ref, leaf)
    i_o, d_o = ot.query(q)
    for flags in (0, 1):
        assert_nn_equal(*gpu_nn(nn, t, q, flags), i_o, d_o)


def test_large_workload_every_query(nn, large_oracle):
    """4M-point target, all 2M queries, both query orders, against the oracle."""
    c = large_oracle["case"]
    t = make_tree(nn, c.target, c.leaf_size)
    i_o, d_o = large_oracle["identity_nn"]
    for flags in (0, 1):
        idx, d2 = gpu_nn(nn, t, c.source, flags)
        assert_nn_equal(idx, d2, i_o, d_o)
    assert (i_o >= 0).all() and np.isfinite(d_o).all()


@pytest.mark.parametrize("name", ["grid", "clustered", "line"])
def test_round_robin_trees_match_brute_force(nn, oracle_mod, name):
    ref, q = _clouds()[name]
    t = nn.kdtree_build(ref, 4, round_robin=True)
    nn.kdtree_upload(t)
    assert_nn_equal(*gpu_nn(nn, t, q, 0), *oracle_mod.nn_brute(ref, q))
