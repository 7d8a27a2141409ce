"""The kernels' float32 arithmetic pinned to the pages' reading on the GPU,
without the oracle in between ("Implementing ICP with CUDA-KDTree", section
3.2 leaf-loop distance and section 2.1 / 3.3 transform).

Expected values come from exact rational arithmetic rounded to binary32 by
definition (tests/test_oracle_rounding.py); the inputs are seeded so that
other association orders and fused multiply-adds give different bits on
many of them.

* nn_query: each query has its own reference point within 35 m and every
  other one at least 200 m away, so the returned dist2 is the
  distance of that one pair, which must carry the reading's bits.
* icp_step: the target holds exactly the reading's transform of every source
  point (on a 4 m lattice), so a kernel transform that deviates in a single
  bit leaves a non-zero dist2.
"""
import numpy as np
import pytest

from test_oracle_rounding import (as_f32, d2_alternatives, d2_reading, tf_alternatives,
                                  tf_reading)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nn():
    import torch
    import icp_nearest_neighbour_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    m.load(build_if_missing=True)
    return m


def _isolated_pairs(seed=91, side=14, spacing=300.0):
    rng = np.random.default_rng(seed)
    g = np.arange(side) * spacing
    base = np.stack(np.meshgrid(g, g, g, indexing="ij"), -1).reshape(-1, 3)
    n = len(base)
    q = (base + rng.uniform(-40, 40, (n, 3))).astype(np.float32)
    scale = 10.0 ** rng.uniform(-3, 1, (n, 3))
    r = (q + rng.standard_normal((n, 3)) * scale).astype(np.float32)
    return r, q


def test_nn_query_distance_is_the_readings(nn):
    import torch
    r, q = _isolated_pairs()
    want = [d2_reading(r[i], q[i]) for i in range(len(r))]
    alts = [d2_alternatives(r[i], q[i]) for i in range(len(r))]
    for name in alts[0]:
        assert sum(a[name] != w for a, w in zip(alts, want)) >= 20, name
    exp = np.array([as_f32(v) for v in want], np.float32)
    tree = nn.kdtree_build(r, 8)
    nn.kdtree_upload(tree)
    for flags in (0, nn.MORTON_SORT):
        idx = torch.empty(len(q), dtype=torch.int32, device="cuda")
        d2 = torch.empty(len(q), dtype=torch.float32, device="cuda")
        nn.nn_query(tree, torch.from_numpy(q).cuda(), idx, d2, flags)
        np.testing.assert_array_equal(idx.cpu().numpy(), np.arange(len(q)))
        np.testing.assert_array_equal(d2.cpu().numpy().view(np.uint32), exp.view(np.uint32))


def _lattice_source(seed, side=20, spacing=4.0):
    rng = np.random.default_rng(seed)
    g = (np.arange(side) - side / 2) * spacing
    s = np.stack(np.meshgrid(g, g, g, indexing="ij"), -1).reshape(-1, 3)
    s = s + rng.uniform(-1, 1, s.shape) * 10.0 ** rng.uniform(-3, 0, s.shape)
    return s.astype(np.float32)


def _rotation(rng):
    axis = rng.standard_normal(3)
    axis /= np.linalg.norm(axis)
    ang = rng.uniform(-np.pi, np.pi)
    K = np.array([[0, -axis[2], axis[1]], [axis[2], 0, -axis[0]], [-axis[1], axis[0], 0]])
    return np.eye(3) + np.sin(ang) * K + (1 - np.cos(ang)) * (K @ K)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_icp_pass_transform_is_the_readings(nn, seed):
    import torch
    rng = np.random.default_rng(seed)
    R = _rotation(rng).astype(np.float32)
    t = rng.uniform(-5, 5, 3).astype(np.float32)
    s = _lattice_source(100 + seed)
    p = [tf_reading(R, t, s[i]) for i in range(len(s))]
    for name in tf_alternatives(R, t, s[0]):
        diff = sum(tf_alternatives(R, t, s[i])[name] != p[i] for i in range(0, len(s), 4))
        assert diff >= 20, name
    target = np.array([[as_f32(v) for v in row] for row in p], np.float32)
    tree = nn.kdtree_build(target, 8)
    nn.kdtree_upload(tree)
    n = len(s)
    idx = torch.empty(n, dtype=torch.int32, device="cuda")
    d2 = torch.empty(n, dtype=torch.float32, device="cuda")
    m = nn.icp_step(tree, torch.from_numpy(s).cuda(), R, t, float("inf"), idx, d2)
    np.testing.assert_array_equal(idx.cpu().numpy(), np.arange(n))
    assert np.all(d2.cpu().numpy().view(np.uint32) == 0)
    assert m["n_accepted"] == n and m["sum_d2"] == 0.0
