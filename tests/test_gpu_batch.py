"""Multi-frame registration (icpnn_icp_align_batch): several sources against
one resident target, several frames in flight ("Implementing ICP with
CUDA-KDTree", section 3.4).  Every frame must equal a single-frame
icpnn_icp_align of it bit for bit, whatever the number of frames in flight,
and the single-frame path is itself held to the oracle (test_gpu_icp.py); one
frame is also compared with the oracle directly here."""
import math

import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def setup():
    import torch
    import icp_nearest_neighbour_gb300 as nn
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    nn.load(build_if_missing=True)
    c, srcs, gts = W.scene_frames(6)
    tree = nn.kdtree_build(c.target, c.leaf_size)
    nn.kdtree_upload(tree)
    dsrcs = [torch.from_numpy(s).cuda() for s in srcs]
    return nn, c, tree, srcs, dsrcs


@pytest.mark.parametrize("residual", [False, True])
def test_batch_equals_single_frames(setup, residual):
    nn, c, tree, srcs, dsrcs = setup
    dmax = c.max_corr_dist[0]
    single = [nn.icp_align(tree, s, c.max_iter, c.eps, dmax, residual_reject=residual, prelaunch=False)
              for s in dsrcs]
    for mc, pre in ((1, True), (3, True), (8, True), (3, False)):
        b = nn.icp_align_batch(tree, dsrcs, c.max_iter, c.eps, dmax, residual_reject=residual,
                               max_concurrent=mc, prelaunch=pre)
        for f, ref in enumerate(single):
            assert b["status"][f] == 0
            np.testing.assert_array_equal(b["T"][f], ref["T"])
            assert b["iters"][f] == ref["iters"]
            assert b["final_mse"][f] == ref["final_mse"]


def test_batch_host_sources_and_initial_transforms(setup):
    nn, c, tree, srcs, dsrcs = setup
    inits = np.stack([np.eye(4)] * 3)
    inits[1, :3, 3] = [0.1, -0.2, 0.05]
    b = nn.icp_align_batch(tree, [srcs[0], dsrcs[1], srcs[2]], 10, 0.0, 1.0, init_T=inits)
    for f, s in enumerate([dsrcs[0], dsrcs[1], dsrcs[2]]):
        ref = nn.icp_align(tree, s, 10, 0.0, 1.0, init_T=inits[f])
        np.testing.assert_array_equal(b["T"][f], ref["T"])


def test_batch_reports_the_failing_frame(setup):
    import torch
    nn, c, tree, srcs, dsrcs = setup
    far = torch.from_numpy(srcs[1] + np.float32(500.0)).cuda()
    with pytest.raises(nn.IcpnnError) as e:
        nn.icp_align_batch(tree, [dsrcs[0], far, dsrcs[2]], 5, 0.0, 0.5)
    assert e.value.status == "DEGENERATE" and "frame 1" in str(e.value)
    res = e.value.result
    assert list(res["status"]) == [0, -4, 0]
    ref = nn.icp_align(tree, dsrcs[2], 5, 0.0, 0.5)
    np.testing.assert_array_equal(res["T"][2], ref["T"])


def test_batch_frame_matches_oracle(setup, oracle_mod):
    nn, c, tree, srcs, dsrcs = setup
    b = nn.icp_align_batch(tree, dsrcs[:4], c.max_iter, c.eps, c.max_corr_dist[0])
    ot = oracle_mod.KDTree(c.target, c.leaf_size)
    ref = oracle_mod.icp_align(ot, srcs[3], c.max_iter, c.eps, c.max_corr_dist[0])
    assert abs(int(b["iters"][3]) - ref["iters"]) <= 1
    if int(b["iters"][3]) == ref["iters"]:
        M = b["T"][3][:3, :3].T @ ref["T"][:3, :3]
        ang = math.atan2(np.linalg.norm([M[2, 1] - M[1, 2], M[0, 2] - M[2, 0], M[1, 0] - M[0, 1]]) / 2,
                         (np.trace(M) - 1) / 2)
        assert ang <= 1e-4
        assert np.linalg.norm(b["T"][3][:3, 3] - ref["T"][:3, 3]) <= 1e-5 * c.extent
