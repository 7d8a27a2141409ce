"""icpnn_icp_step_noalloc: the ICP correspondence pass for callers that cannot
allocate device memory (a host application that owns every device buffer,
a process whose memory is reserved by another allocator, a real-time loop
that cannot stop for cudaMalloc / cudaFree).  Its only scratch is a fixed
array inside the library, shared by every call.

Checked through the C ABI against the ordinary pass, icpnn_icp_step, on two
calls in a row (the second call runs on whatever the first left in the shared
scratch): per-point indices and distances bit for bit, moments within the
tolerances the other ICP tests use.  This file is collected last.
"""
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
    c = W.scene_case()
    tree = nn.kdtree_build(c.target, c.leaf_size)
    nn.kdtree_upload(tree)
    return nn, c, tree, torch.from_numpy(c.source).cuda()


def _outputs(n):
    import torch
    return (torch.full((n,), -7, dtype=torch.int32, device="cuda"),
            torch.full((n,), -7.0, dtype=torch.float32, device="cuda"))


def _close(a, b, extent):
    assert a["n_accepted"] == b["n_accepted"] and a["n_nonfinite"] == b["n_nonfinite"] == 0
    assert abs(a["mse"] - b["mse"]) <= 1e-6 * abs(b["mse"])
    scale = max(np.abs(b["mu_src"]).max(), np.abs(b["mu_tgt"]).max(), extent)
    assert np.abs(a["mu_src"] - b["mu_src"]).max() <= 1e-5 * scale
    assert np.abs(a["mu_tgt"] - b["mu_tgt"]).max() <= 1e-5 * scale
    assert np.linalg.norm(a["H"] - b["H"]) <= 1e-5 * np.linalg.norm(b["H"])


def test_noalloc_pass_matches_icp_step_on_two_calls_in_a_row(setup):
    import torch
    nn, c, tree, src = setup
    n = len(c.source)
    cases = [(np.eye(4), c.max_corr_dist[0]), (c.T_gt, 0.3)]
    rt = [(T[:3, :3].astype(np.float32), T[:3, 3].astype(np.float32), d) for T, d in cases]

    refs = []
    for R, t, d in rt:
        idx, d2 = _outputs(n)
        m = nn.icp_step(tree, src, R, t, d, idx, d2)
        refs.append((m, idx.cpu().numpy(), d2.cpu().numpy()))

    outs = []
    for R, t, d in rt:                       # back to back: call 1, then call 2
        idx, d2 = _outputs(n)
        m = nn.icp_step_noalloc(tree, src, R, t, d, idx, d2)
        outs.append((m, idx, d2))
    torch.cuda.synchronize()

    for (m_ref, i_ref, d_ref), (m, idx, d2) in zip(refs, outs):
        np.testing.assert_array_equal(idx.cpu().numpy(), i_ref)
        np.testing.assert_array_equal(d2.cpu().numpy().view(np.uint32), d_ref.view(np.uint32))
        _close(m, m_ref, c.extent)


def test_noalloc_limits(setup):
    import torch
    nn, c, tree, src = setup
    R = np.eye(3, dtype=np.float32)
    t = np.zeros(3, np.float32)
    big = torch.zeros((nn.NOALLOC_MAX_POINTS + 1, 3), dtype=torch.float32, device="cuda")
    with pytest.raises(nn.IcpnnError) as e:
        nn.icp_step_noalloc(tree, big, R, t)
    assert e.value.status == "INVALID_ARG" and str(nn.NOALLOC_MAX_POINTS) in str(e.value)
    with pytest.raises(nn.IcpnnError) as e:
        nn.icp_step_noalloc(tree, c.source, R, t)      # host buffer: would need a staging copy
    assert e.value.status == "INVALID_ARG"
    # a rejected call leaves the shared scratch usable
    m = nn.icp_step_noalloc(tree, src, R, t, c.max_corr_dist[0])
    _close(m, nn.icp_step(tree, src, R, t, c.max_corr_dist[0]), c.extent)


def test_noalloc_pass_at_its_largest_size(setup):
    """n = NOALLOC_MAX_POINTS uses the scratch array to its last partial
    record and counter word: the same results as icp_step, twice in a row."""
    import torch
    nn, c, tree, _ = setup
    n = nn.NOALLOC_MAX_POINTS
    reps = -(-n // len(c.source))
    jitter = np.repeat(np.arange(reps, dtype=np.float32) * np.float32(1e-3), len(c.source))[:, None]
    pts = np.ascontiguousarray((np.tile(c.source, (reps, 1)) + jitter)[:n], np.float32)
    src = torch.from_numpy(pts).cuda()
    R = c.T_gt[:3, :3].astype(np.float32)
    t = c.T_gt[:3, 3].astype(np.float32)
    idx_r, d2_r = _outputs(n)
    ref = nn.icp_step(tree, src, R, t, c.max_corr_dist[0], idx_r, d2_r)
    for _ in range(2):
        idx, d2 = _outputs(n)
        m = nn.icp_step_noalloc(tree, src, R, t, c.max_corr_dist[0], idx, d2)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(idx.cpu().numpy(), idx_r.cpu().numpy())
        np.testing.assert_array_equal(d2.cpu().numpy().view(np.uint32), d2_r.cpu().numpy().view(np.uint32))
        _close(m, ref, c.extent)
