"""GPU voxel-grid downsampling (icpnn_voxel_downsample) against the oracle:
bit-identical centroids in the same voxel order ("Implementing ICP with
CUDA-KDTree", section 4.3)."""
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


def gpu_vox(nn, pts, v, host=False):
    import torch
    if host:
        return nn.voxel_downsample(np.ascontiguousarray(pts, np.float32), v)
    out = nn.voxel_downsample(torch.from_numpy(np.ascontiguousarray(pts, np.float32)).cuda(), v)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def assert_same(a, b):
    assert a.shape == b.shape
    np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))


def test_hand_fixture(nn):
    rows = read_fixture("voxel_hand.txt")
    pts = np.array([[float(v) for v in r[1:4]] for r in rows if r[0] == "point"], np.float32)
    exp = np.array([[float(v) for v in r[1:4]] for r in rows if r[0] == "expect"]).astype(np.float32)
    for host in (False, True):
        assert_same(gpu_vox(nn, pts, 0.5, host), exp)


def _clouds():
    rng = np.random.default_rng(23)
    normal = (rng.normal(size=(20000, 3)) * np.array([2.0, 1.0, 0.5])).astype(np.float32)
    normal[::97] = normal[1::97]
    wide = rng.uniform(-5000, 5000, size=(50000, 3)).astype(np.float32)      # 2^60 keys: two-stage sort
    grid = W.grid_cloud(20, 0.5, origin=(-5.0, -5.0, -5.0))                   # points on voxel faces
    holes = normal.copy()
    holes[::13, 1] = np.nan
    holes[::29, 2] = np.inf
    return {
        "normal_0.37": (normal, 0.37),
        "normal_0.05": (normal, 0.05),
        "wide_0.01": (wide, 0.01),
        "grid_0.5": (grid, 0.5),
        "nonfinite_0.2": (holes, 0.2),
        "same_voxel": (np.tile(np.array([[0.01, 0.02, 0.03]], np.float32), (3000, 1)), 1.0),
        "single": (np.array([[1.5, -2.5, 3.25]], np.float32), 0.1),
    }


@pytest.mark.parametrize("name", list(_clouds()))
def test_clouds_match_oracle(nn, oracle_mod, name):
    pts, v = _clouds()[name]
    assert_same(gpu_vox(nn, pts, v), oracle_mod.voxel_downsample(pts, v))


@pytest.mark.parametrize("name,v", [("large", 0.1), ("lidar", 0.2), ("scene", 0.05)])
def test_workload_targets(nn, oracle_mod, name, v):
    pts = W.CASES[name]().target
    assert_same(gpu_vox(nn, pts, v), oracle_mod.voxel_downsample(pts, v))


def test_empty_and_all_nonfinite(nn):
    assert gpu_vox(nn, np.zeros((0, 3), np.float32), 0.1, host=True).shape == (0, 3)
    assert gpu_vox(nn, np.full((7, 3), np.nan, np.float32), 0.1).shape == (0, 3)


def test_errors(nn):
    pts = W.uniform_cloud(100, 3)
    for bad in (0.0, -1.0, float("inf")):
        with pytest.raises(nn.IcpnnError) as e:
            gpu_vox(nn, pts, bad)
        assert e.value.status == "INVALID_ARG"
    huge = pts.copy()
    huge[5] = 1e30
    with pytest.raises(nn.IcpnnError) as e:
        gpu_vox(nn, huge, 1e-3)
    assert e.value.status == "INVALID_ARG" and "2^40" in str(e.value)
    # the library stays usable
    assert_same(gpu_vox(nn, pts, 0.5), gpu_vox(nn, pts, 0.5, host=True))
