"""GPU parity of the fused ICP pass (icpnn_icp_step) and of the whole
registration (icpnn_icp_align) against the oracle.

"Implementing ICP with CUDA-KDTree" (pwwt.cn/news/5235220): section 2.1
(objective and SVD step), 3.3 (loop on the original source with the
accumulated transform), 4.4 (maximum correspondence distance), 4.6 (stopping
rule).

Tolerances:
  * per-point indices and squared distances: bit-identical;
  * accepted-pair counts: identical (the accept test is an exact float
    comparison on bit-identical distances);
  * mse: 1e-6 relative (float32 partial sums per warp, float-float pairs above);
  * centroids: 1e-5 of max(|mu|, scene extent); H: 1e-5 relative in the
    Frobenius norm;
  * transforms: 1e-4 rad rotation and 1e-5 * scene extent translation.
"""
import math

import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu

ROT_TOL = 1e-4
TRANS_TOL = 1e-5


@pytest.fixture(scope="module")
def nn():
    import torch
    import icp_nearest_neighbour_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    m.load(build_if_missing=True)
    return m


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def rot_angle(Ra, Rb):
    """Angle of Ra^T Rb, robust near zero (from the skew part)."""
    M = np.asarray(Ra).T @ np.asarray(Rb)
    s = np.linalg.norm([M[2, 1] - M[1, 2], M[0, 2] - M[2, 0], M[1, 0] - M[0, 1]]) / 2
    c = (np.trace(M) - 1) / 2
    return math.atan2(s, c)


def check_moments(m, st, extent):
    assert m["n_accepted"] == st["n_accepted"]
    if st["n_accepted"] == 0:
        return
    assert abs(m["mse"] - st["mse"]) <= 1e-6 * abs(st["mse"]) + 1e-30
    scale = max(np.abs(st["mu_s"]).max(), np.abs(st["mu_q"]).max(), extent)
    assert np.abs(m["mu_src"] - st["mu_s"]).max() <= 1e-5 * scale
    assert np.abs(m["mu_tgt"] - st["mu_q"]).max() <= 1e-5 * scale
    assert np.linalg.norm(m["H"] - st["H"]) <= 1e-5 * np.linalg.norm(st["H"])


def check_transform(Ta, Tb, extent):
    assert rot_angle(Ta[:3, :3], Tb[:3, :3]) <= ROT_TOL
    assert np.linalg.norm(Ta[:3, 3] - Tb[:3, 3]) <= TRANS_TOL * extent


def lib_step(nn, tree, src, T, dmax):
    import torch
    R32 = np.asarray(T)[:3, :3].astype(np.float32)
    t32 = np.asarray(T)[:3, 3].astype(np.float32)
    n = len(src)
    idx = torch.empty(n, dtype=torch.int32, device="cuda")
    d2 = torch.empty(n, dtype=torch.float32, device="cuda")
    m = nn.icp_step(tree, dev(src), R32, t32, dmax, idx, d2)
    return m, idx.cpu().numpy(), d2.cpu().numpy()


def setup(nn, oracle_mod, case):
    t = nn.kdtree_build(case.target, case.leaf_size)
    nn.kdtree_upload(t)
    return t, oracle_mod.KDTree(case.target, case.leaf_size)


@pytest.mark.parametrize("name", ["tiny", "scene"])
def test_step_parity(nn, oracle_mod, name):
    c = W.CASES[name]()
    t, ot = setup(nn, oracle_mod, c)
    for T in (np.eye(4), c.T_gt):
        for dmax in (c.max_corr_dist[0], math.inf, 0.05):
            m, idx, d2 = lib_step(nn, t, c.source, T, dmax)
            st = oracle_mod.icp_step(ot, c.source, T, dmax)
            np.testing.assert_array_equal(idx, st["idx"])
            np.testing.assert_array_equal(d2.view(np.uint32), st["d2"].view(np.uint32))
            check_moments(m, st, c.extent)
            assert m["n_nonfinite"] == 0


def test_step_host_source_and_no_per_point_outputs(nn, oracle_mod):
    c = W.tiny_case()
    t, ot = setup(nn, oracle_mod, c)
    R = c.T_gt[:3, :3].astype(np.float32)
    tt = c.T_gt[:3, 3].astype(np.float32)
    m_host = nn.icp_step(t, c.source, R, tt, 0.1)
    m_dev = nn.icp_step(t, dev(c.source), R, tt, 0.1)
    for k in ("n_accepted", "mse"):
        assert m_host[k] == m_dev[k]
    np.testing.assert_array_equal(m_host["H"], m_dev["H"])
    check_moments(m_dev, oracle_mod.icp_step(ot, c.source, c.T_gt, 0.1), c.extent)


@pytest.mark.parametrize("name", ["scene", "lidar"])
def test_radius_seeded_pass_gives_identical_moments(nn, oracle_mod, name):
    """Without per-point outputs the search starts from the rejection radius;
    the accepted pairs, and so every moment bit, must not change."""
    c = W.CASES[name]()
    t, ot = setup(nn, oracle_mod, c)
    src = dev(c.source)
    for T in (np.eye(4), c.T_gt):
        R32 = T[:3, :3].astype(np.float32)
        t32 = T[:3, 3].astype(np.float32)
        for dmax in (c.max_corr_dist[0], 0.05, 0.3, math.inf):
            full, _, _ = lib_step(nn, t, c.source, T, dmax)
            seeded = nn.icp_step(t, src, R32, t32, dmax)
            for k in ("n_accepted", "sum_d2", "mse"):
                assert full[k] == seeded[k] or (math.isnan(full[k]) and math.isnan(seeded[k]))
            np.testing.assert_array_equal(full["H"], seeded["H"])
            np.testing.assert_array_equal(full["mu_src"], seeded["mu_src"])


@pytest.mark.parametrize("nsrc", [1, 3, 255, 257, 4099])
def test_step_ragged_sizes(nn, oracle_mod, nsrc):
    c = W.tiny_case()
    t, ot = setup(nn, oracle_mod, c)
    src = np.ascontiguousarray(c.source[:nsrc])
    m, idx, d2 = lib_step(nn, t, src, c.T_gt, math.inf)
    st = oracle_mod.icp_step(ot, src, c.T_gt, math.inf)
    np.testing.assert_array_equal(idx, st["idx"])
    np.testing.assert_array_equal(d2.view(np.uint32), st["d2"].view(np.uint32))
    check_moments(m, st, c.extent)


def _trace_parity(nn, oracle_mod, c, t, ot, src, dmax, res, sample_iters=None):
    """Feed each iteration's transform to the oracle: same pairs, same mse,
    and a solve that lands on the library's next transform."""
    tr = res["trace"]
    ks = range(len(tr)) if sample_iters is None else sample_iters
    for k in ks:
        st = oracle_mod.icp_step(ot, src, tr[k]["T"], dmax)
        assert tr[k]["n_accepted"] == st["n_accepted"], k
        assert abs(tr[k]["mse"] - st["mse"]) <= 1e-6 * st["mse"], k
        T_next = oracle_mod.solve_from_step(st, src, ot)
        T_lib = tr[k + 1]["T"] if k + 1 < len(tr) else res["T"]
        check_transform(T_lib, T_next, c.extent)


@pytest.mark.parametrize("name", ["tiny", "scene", "lidar"])
def test_align_parity(nn, oracle_mod, name):
    c = W.CASES[name]()
    t, ot = setup(nn, oracle_mod, c)
    dmax = c.max_corr_dist[0]
    res = nn.icp_align(t, dev(c.source), c.max_iter, c.eps, dmax, trace=True)
    _trace_parity(nn, oracle_mod, c, t, ot, c.source, dmax, res)
    # the reported error is the oracle's pass under the returned transform
    fin = oracle_mod.icp_step(ot, c.source, res["T"], dmax)
    assert abs(res["final_mse"] - fin["mse"]) <= 1e-6 * fin["mse"]
    assert res["final_n_accepted"] == fin["n_accepted"]
    assert res["overlap"] == fin["n_accepted"] / len(c.source)
    ref = oracle_mod.icp_align(ot, c.source, c.max_iter, c.eps, dmax)
    # independent end-to-end runs: the same transform.  The iteration count
    # may differ by one when |delta mse| lands within rounding of eps; the
    # library's transform is then compared with the oracle run for exactly the
    # library's number of iterations.
    assert abs(res["iters"] - ref["iters"]) <= 1
    if res["iters"] != ref["iters"]:
        ref = oracle_mod.icp_align(ot, c.source, res["iters"], 0.0, dmax)
        assert ref["iters"] == res["iters"]
    check_transform(res["T"], ref["T"], c.extent)
    # when both transforms round to the same float32 (R, t) the final passes
    # are the same computation on both sides
    if all(np.array_equal(a, b) for a, b in zip(oracle_mod.as_kernel_rt(res["T"]),
                                                oracle_mod.as_kernel_rt(ref["T"]))):
        assert abs(res["final_mse"] - ref["final_mse"]) <= 1e-6 * ref["final_mse"]
    R = res["T"][:3, :3]
    np.testing.assert_allclose(R.T @ R, np.eye(3), atol=1e-12)
    assert abs(np.linalg.det(R) - 1) < 1e-12


def test_overlap_ratio_and_warning(nn, oracle_mod):
    """Page section 6: warn when the overlap after registration is below 80%.
    Overlap = pairs accepted under the returned transform / source points.
    The scene registration overlaps fully; the LiDAR scans (25% of each
    sector unseen by the other, returns thinning out with range beyond the
    0.5 m gate) stay near one half, and the call warns."""
    import warnings
    c = W.scene_case()
    t = nn.kdtree_build(c.target, c.leaf_size)
    nn.kdtree_upload(t)
    with warnings.catch_warnings():
        warnings.simplefilter("error", nn.LowOverlapWarning)
        res = nn.icp_align(t, dev(c.source), c.max_iter, c.eps, c.max_corr_dist[0])
    assert res["overlap"] >= nn.OVERLAP_WARN_RATIO and not res["low_overlap"]
    c = W.lidar_case()
    t, ot = setup(nn, oracle_mod, c)
    with pytest.warns(nn.LowOverlapWarning):
        res = nn.icp_align(t, dev(c.source), c.max_iter, c.eps, c.max_corr_dist[0])
    assert res["low_overlap"] and res["overlap"] < nn.OVERLAP_WARN_RATIO
    fin = oracle_mod.icp_step(ot, c.source, res["T"], c.max_corr_dist[0])
    assert res["final_n_accepted"] == fin["n_accepted"]
    b = nn.icp_align_batch(t, [dev(c.source)], c.max_iter, c.eps, c.max_corr_dist[0])
    assert b["final_n_accepted"][0] == res["final_n_accepted"]


def _residual_case(name):
    if name == "tiny_outliers":
        c = W.tiny_case()
        src, _ = W.with_outliers(c.source, 0.05, 0.15, 11)
        return c, src, math.inf
    c = W.CASES[name]()
    return c, c.source, c.max_corr_dist[0]


@pytest.mark.parametrize("name", ["tiny_outliers", "scene"])
def test_residual_rejection_parity(nn, oracle_mod, name):
    """Section 4.4 residual rejection: each iteration's transform fed to the
    oracle reproduces the correspondence pass exactly, the residual variance
    to 1e-5, the kept set up to pairs whose residual sits within rounding of
    the 3-sigma threshold (the two sides sum the residuals in different
    orders), and the re-solve lands on the library's next transform."""
    c, src, dmax = _residual_case(name)
    t, ot = setup(nn, oracle_mod, c)
    res = nn.icp_align(t, dev(src), c.max_iter, c.eps, dmax, trace=True, residual_reject=True)
    tr = res["trace"]
    ks = range(len(tr)) if name == "tiny_outliers" else sorted({0, 1, 5, len(tr) // 2, len(tr) - 1})
    for k in ks:
        st = oracle_mod.icp_step(ot, src, tr[k]["T"], dmax)
        assert tr[k]["n_accepted"] == st["n_accepted"], k
        assert abs(tr[k]["mse"] - st["mse"]) <= 1e-6 * st["mse"], k
        T1 = oracle_mod.solve_from_step(st, src, ot)
        rr = oracle_mod.residual_reject(st, src, ot, T1, 3.0)
        assert abs(tr[k]["sigma2"] - rr["sigma2"]) <= 1e-5 * rr["sigma2"], k
        assert abs(tr[k]["n_inliers"] - rr["n_kept"]) <= 2, k
        if name == "tiny_outliers":
            assert tr[k]["n_inliers"] < tr[k]["n_accepted"], k
        T_lib = tr[k + 1]["T"] if k + 1 < len(tr) else res["T"]
        check_transform(T_lib, rr["T"], c.extent)
    if name == "tiny_outliers":
        plain = nn.icp_align(t, dev(src), c.max_iter, c.eps, dmax)
        assert rot_angle(res["T"][:3, :3], c.T_gt[:3, :3]) < rot_angle(plain["T"][:3, :3], c.T_gt[:3, :3])


@pytest.mark.parametrize("name", ["tiny_outliers", "scene"])
def test_persistent_residual_registration_matches_ordinary_launches(nn, name):
    """The persistent kernel runs each iteration's residual passes itself (the
    threshold handed over on the GPU); the registration is bit-identical to
    one with ordinary launches, also when one residual command arrives after
    the kernel gave up waiting for it (80 ms late: the host falls back)."""
    c, src, dmax = _residual_case(name)
    t = nn.kdtree_build(c.target, c.leaf_size)
    nn.kdtree_upload(t)
    s = dev(src)
    kw = dict(trace=True, residual_reject=True, warn_overlap=False)
    a = nn.icp_align(t, s, c.max_iter, c.eps, dmax, prelaunch=False, **kw)
    b = nn.icp_align(t, s, c.max_iter, c.eps, dmax, **kw)
    nn.probe_delay_commands(3, 1, 80_000_000)     # the second iteration's residual command
    try:
        d = nn.icp_align(t, s, c.max_iter, c.eps, dmax, **kw)
    finally:
        nn.probe_delay_commands(0, 0, 0)
    for r in (b, d):
        np.testing.assert_array_equal(a["T"], r["T"])
        assert a["iters"] == r["iters"] and a["final_mse"] == r["final_mse"]
        for ra, rb in zip(a["trace"], r["trace"]):
            assert (ra["mse"], ra["n_accepted"], ra["n_inliers"], ra["sigma2"]) == \
                (rb["mse"], rb["n_accepted"], rb["n_inliers"], rb["sigma2"])


def test_tiny_recovers_ground_truth(nn):
    c = W.tiny_case()
    t = nn.kdtree_build(c.target, c.leaf_size)
    nn.kdtree_upload(t)
    res = nn.icp_align(t, dev(c.source), c.max_iter, c.eps, c.max_corr_dist[0])
    assert res["iters"] < c.max_iter
    assert rot_angle(res["T"][:3, :3], c.T_gt[:3, :3]) < 3e-4
    assert np.linalg.norm(res["T"][:3, 3] - c.T_gt[:3, 3]) < 5e-4


def test_align_is_deterministic(nn):
    c = W.scene_case()
    t = nn.kdtree_build(c.target, c.leaf_size)
    nn.kdtree_upload(t)
    a = nn.icp_align(t, dev(c.source), 10, 0.0, 1.0, trace=True)
    b = nn.icp_align(t, dev(c.source), 10, 0.0, 1.0, trace=True)
    np.testing.assert_array_equal(a["T"], b["T"])
    assert [r["mse"] for r in a["trace"]] == [r["mse"] for r in b["trace"]]


def test_upload_on_one_stream_registration_on_another(nn):
    """The upload does not wait for its copies: a registration (and a query)
    issued at once on another stream must still see the whole tree."""
    import torch
    c = W.scene_case()
    ref_t = nn.kdtree_build(c.target, c.leaf_size)
    nn.kdtree_upload(ref_t)
    ref = nn.icp_align(ref_t, dev(c.source), 10, 0.0, 1.0)
    q = dev(c.source)
    ref_idx = torch.empty(len(c.source), dtype=torch.int32, device="cuda")
    ref_d2 = torch.empty(len(c.source), dtype=torch.float32, device="cuda")
    nn.nn_query(ref_t, q, ref_idx, ref_d2)
    torch.cuda.synchronize()
    up, use = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        t = nn.kdtree_build(c.target, c.leaf_size)
        nn.kdtree_upload(t, stream=up)
        idx = torch.empty_like(ref_idx)
        d2 = torch.empty_like(ref_d2)
        nn.nn_query(t, q, idx, d2, stream=use)
        r = nn.icp_align(t, dev(c.source), 10, 0.0, 1.0, stream=use)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(r["T"], ref["T"])
        assert torch.equal(idx, ref_idx) and torch.equal(d2, ref_d2)
        t.free()


@pytest.mark.parametrize("name", ["tiny", "scene", "lidar"])
def test_prelaunched_passes_match_plain_launches(nn, name):
    """Queuing each pass before its transform is solved (the default) changes
    when the kernels start, not what they compute: bit-identical transforms,
    per-iteration records and final mse; also with timing and an initial
    transform, and over several registrations on one stream."""
    import torch
    c = W.CASES[name]()
    t = nn.kdtree_build(c.target, c.leaf_size)
    nn.kdtree_upload(t)
    src = dev(c.source)
    dmax = c.max_corr_dist[0]
    init = np.eye(4)
    init[:3, 3] = [0.01, -0.02, 0.005]
    for kw in ({}, {"timing": True}, {"init_T": init}):
        a = nn.icp_align(t, src, c.max_iter, c.eps, dmax, trace=True, prelaunch=False, warn_overlap=False, **kw)
        for mode in ({"persistent": False}, {}):      # passes pre-launched one by one; one persistent kernel
            b = nn.icp_align(t, src, c.max_iter, c.eps, dmax, trace=True, warn_overlap=False, **mode, **kw)
            np.testing.assert_array_equal(a["T"], b["T"])
            assert a["iters"] == b["iters"] and a["final_mse"] == b["final_mse"]
            assert a["final_n_accepted"] == b["final_n_accepted"]
            for ra, rb in zip(a["trace"], b["trace"]):
                assert (ra["mse"], ra["n_accepted"]) == (rb["mse"], rb["n_accepted"])
                np.testing.assert_array_equal(ra["T"], rb["T"])
            if kw.get("timing"):
                assert all(r["kernel_ms"] > 0 for r in b["trace"])
    s = torch.cuda.Stream()
    outs = [nn.icp_align(t, src, 8, 0.0, dmax, stream=s, warn_overlap=False) for _ in range(3)]
    s2 = torch.cuda.Stream()
    outs += [nn.icp_align(t, src, 8, 0.0, dmax, stream=x, warn_overlap=False) for x in (s, s2, s, s2)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        np.testing.assert_array_equal(o["T"], outs[0]["T"])


def test_pass_command_wait_is_bounded(nn):
    """A pre-launched pass whose command never comes gives up after its wait
    limit and publishes the abort marker; the stop command makes it return
    without a result; the identity command makes it run.  The context stays
    usable throughout."""
    c = W.scene_case()
    t = nn.kdtree_build(c.target, c.leaf_size)
    nn.kdtree_upload(t)
    src = dev(c.source)
    assert nn.probe_command_wait(t, src, 2_000_000, 0) == 1
    assert nn.probe_command_wait(t, src, 2_000_000, 1) == 0
    assert nn.probe_command_wait(t, src, 2_000_000, 2) == 2
    assert nn.probe_command_wait(t, c.source[:1000], 2_000_000, 0) == 1   # host source, one block
    for bad in ((0, 0), (2_000_000_000, 0), (1000, 3)):
        with pytest.raises(nn.IcpnnError):
            nn.probe_command_wait(t, src, *bad)
    a = nn.icp_align(t, src, 10, 0.0, c.max_corr_dist[0], prelaunch=False)
    b = nn.icp_align(t, src, 10, 0.0, c.max_corr_dist[0])
    np.testing.assert_array_equal(a["T"], b["T"])


def test_residual_and_prelaunched_registrations_alternate(nn):
    """Residual registrations and pre-launched ones share the thread's mapped
    buffer (result slot, command regions): a registration of either kind
    leaves nothing behind that changes the other's result."""
    c = W.tiny_case()
    t = nn.kdtree_build(c.target, c.leaf_size)
    nn.kdtree_upload(t)
    src = dev(c.source)
    ref = nn.icp_align(t, src, 10, 0.0, math.inf, prelaunch=False)
    ref_r = nn.icp_align(t, src, 10, 0.0, math.inf, residual_reject=True)
    for _ in range(6):
        r = nn.icp_align(t, src, 10, 0.0, math.inf, residual_reject=True)
        np.testing.assert_array_equal(r["T"], ref_r["T"])
        r = nn.icp_align(t, src, 10, 0.0, math.inf)
        np.testing.assert_array_equal(r["T"], ref["T"])


@pytest.mark.parametrize("persistent", [True, False])
@pytest.mark.parametrize("skip", [0, 5])
def test_registration_survives_a_pass_that_gives_up_waiting(nn, skip, persistent):
    """Fault injected on the host: the transform command of one pre-launched
    pass (the first, or the sixth) is written 80 ms late, beyond the pass's
    50 ms wait.  The pass gives up and publishes its abort marker; the
    registration runs that pass again as an ordinary launch, continues with
    ordinary launches, and ends bit-identical to a run that never
    pre-launched."""
    import time
    c = W.scene_case()
    t = nn.kdtree_build(c.target, c.leaf_size)
    nn.kdtree_upload(t)
    src = dev(c.source)
    dmax = c.max_corr_dist[0]
    ref = nn.icp_align(t, src, 12, 0.0, dmax, trace=True, prelaunch=False)
    nn.probe_delay_commands(skip, 1, 80_000_000)
    try:
        t0 = time.perf_counter()
        res = nn.icp_align(t, src, 12, 0.0, dmax, trace=True, persistent=persistent)
        elapsed = time.perf_counter() - t0
    finally:
        nn.probe_delay_commands(0, 0, 0)
    assert elapsed > 0.05
    np.testing.assert_array_equal(res["T"], ref["T"])
    assert res["iters"] == ref["iters"] and res["final_mse"] == ref["final_mse"]
    assert [r["mse"] for r in res["trace"]] == [r["mse"] for r in ref["trace"]]
    again = nn.icp_align(t, src, 12, 0.0, dmax, persistent=persistent)   # pre-launches again
    np.testing.assert_array_equal(again["T"], ref["T"])
    with pytest.raises(nn.IcpnnError):
        nn.probe_delay_commands(-1, 1, 0)


@pytest.mark.parametrize("persistent", [True, False])
@pytest.mark.parametrize("skip", [0, 4])
def test_registration_survives_a_stalled_host(nn, skip, persistent):
    """Fault injected on the host: between queuing pass k+1 and reading pass
    k the host sleeps 250 ms, beyond twice the 50 ms command wait (as when the
    host thread is descheduled, or a profiler serialises the launches).  Pass
    k has published, pass k+1 gives up waiting; pass k's result must still be
    read, pass k+1 run again as an ordinary launch, and the registration end
    bit-identical to one that never pre-launched."""
    import time
    c = W.scene_case()
    t = nn.kdtree_build(c.target, c.leaf_size)
    nn.kdtree_upload(t)
    src = dev(c.source)
    dmax = c.max_corr_dist[0]
    ref = nn.icp_align(t, src, 12, 0.0, dmax, trace=True, prelaunch=False)
    nn.probe_delay_collect(skip, 1, 250_000_000)
    try:
        t0 = time.perf_counter()
        res = nn.icp_align(t, src, 12, 0.0, dmax, trace=True, persistent=persistent)
        elapsed = time.perf_counter() - t0
    finally:
        nn.probe_delay_collect(0, 0, 0)
    assert elapsed > 0.25
    np.testing.assert_array_equal(res["T"], ref["T"])
    assert res["iters"] == ref["iters"] and res["final_mse"] == ref["final_mse"]
    assert [r["mse"] for r in res["trace"]] == [r["mse"] for r in ref["trace"]]
    assert [r["n_accepted"] for r in res["trace"]] == [r["n_accepted"] for r in ref["trace"]]
    again = nn.icp_align(t, src, 12, 0.0, dmax, persistent=persistent)   # pre-launches again
    np.testing.assert_array_equal(again["T"], ref["T"])


@pytest.mark.parametrize("residual", [False, True])
def test_back_to_back_registrations_with_a_late_first_command(nn, residual):
    """A registration ends by telling its persistent kernel to stop; that stop
    stays in the thread's command block.  The next registration's kernel must
    not take it for its own first command: here the first command is written
    5 ms after the launch (inside the 50 ms wait), so the new kernel certainly
    polls before it arrives."""
    c = W.tiny_case()
    t = nn.kdtree_build(c.target, c.leaf_size)
    nn.kdtree_upload(t)
    src = dev(c.source)
    kw = dict(residual_reject=residual, warn_overlap=False)
    ref = nn.icp_align(t, src, 8, 0.0, math.inf, prelaunch=False, **kw)
    for _ in range(3):
        nn.icp_align(t, src, 8, 0.0, math.inf, **kw)
        nn.probe_delay_commands(0, 1, 5_000_000)
        try:
            r = nn.icp_align(t, src, 8, 0.0, math.inf, **kw)
        finally:
            nn.probe_delay_commands(0, 0, 0)
        np.testing.assert_array_equal(r["T"], ref["T"])
        assert r["final_mse"] == ref["final_mse"]


def test_persistent_registration_on_many_sizes(nn):
    """The persistent kernel runs the per-pass kernel's grid (one partial per
    block, the same reduction levels), so its registration is bit-identical
    to ordinary launches for one-level reductions (<= 56 blocks), two-level
    ones with a ragged last group, and grids that loop over chunks."""
    c = W.scene_case()
    t = nn.kdtree_build(c.target, c.leaf_size)
    nn.kdtree_upload(t)
    for n in (5, 300, 14 * 256 * 8 + 1, 57 * 256, 100_000):
        src = dev(c.source[:n])
        dmax = math.inf if n < 1000 else 1.0
        a = nn.icp_align(t, src, 6, 0.0, dmax, trace=True, prelaunch=False, warn_overlap=False)
        b = nn.icp_align(t, src, 6, 0.0, dmax, trace=True, warn_overlap=False)
        np.testing.assert_array_equal(a["T"], b["T"])
        assert a["final_mse"] == b["final_mse"]
        assert [r["mse"] for r in a["trace"]] == [r["mse"] for r in b["trace"]]
    big = np.ascontiguousarray(np.tile(c.source, (8, 1)) + np.float32(0.001))    # 800k: chunks per warp > 1
    a = nn.icp_align(t, dev(big), 4, 0.0, 1.0, prelaunch=False, warn_overlap=False)
    b = nn.icp_align(t, dev(big), 4, 0.0, 1.0, warn_overlap=False)
    np.testing.assert_array_equal(a["T"], b["T"])
    assert a["final_mse"] == b["final_mse"]


def test_large_coarse_to_fine(nn, oracle_mod, large_oracle):
    """4M target / 2M source, two stages (2.0 m then 0.3 m), at full size.
    The first pass of each stage and its last pass are compared over the whole
    2M-point source: per-point indices and distances bit-identical, same
    accepted count and mse, moments within tolerance, and the oracle's solve
    from the last pass lands on the library's result.  (The oracle's searches
    are split over the host cores; each query's search is unchanged.)"""
    c = large_oracle["case"]
    ot = large_oracle["tree"]
    workers = large_oracle["workers"]
    t = nn.kdtree_build(c.target, c.leaf_size)
    nn.kdtree_upload(t)
    src_d = dev(c.source)
    T = None
    for dmax in c.max_corr_dist:
        res = nn.icp_align(t, src_d, c.max_iter, c.eps, dmax, init_T=T, trace=True)
        tr = res["trace"]
        for k in sorted({0, len(tr) - 1}):
            Tk = tr[k]["T"]
            m, idx, d2 = lib_step(nn, t, c.source, Tk, dmax)
            # the first pass evaluates the identity: the raw source's neighbours
            pre = large_oracle["identity_nn"] if np.array_equal(Tk, np.eye(4)) else None
            st = oracle_mod.icp_step(ot, c.source, Tk, dmax, workers=workers, nn=pre)
            np.testing.assert_array_equal(idx, st["idx"])
            np.testing.assert_array_equal(d2.view(np.uint32), st["d2"].view(np.uint32))
            check_moments(m, st, c.extent)
            assert tr[k]["n_accepted"] == st["n_accepted"]
            assert abs(tr[k]["mse"] - st["mse"]) <= 1e-6 * st["mse"]
            if k == len(tr) - 1:
                check_transform(res["T"], oracle_mod.solve_from_step(st, c.source, ot), c.extent)
        T = res["T"]
    assert abs(np.linalg.det(T[:3, :3]) - 1) < 1e-12


def test_errors(nn):
    c = W.tiny_case()
    t = nn.kdtree_build(c.target, c.leaf_size)
    nn.kdtree_upload(t)
    far = dev(c.source + np.float32(100.0))
    with pytest.raises(nn.IcpnnError) as e:
        nn.icp_align(t, far, 5, 1e-6, 0.1)
    assert e.value.status == "DEGENERATE"
    bad = c.source.copy()
    bad[3, 0] = np.nan
    with pytest.raises(nn.IcpnnError) as e:
        nn.icp_align(t, dev(bad), 5, 1e-6, math.inf)
    assert e.value.status == "NONFINITE"
    with pytest.raises(nn.IcpnnError) as e:
        nn.icp_align(t, dev(c.source), 0, 1e-6, math.inf)
    assert e.value.status == "INVALID_ARG"
    with pytest.raises(nn.IcpnnError) as e:
        nn.icp_align(t, dev(c.source), 5, -1.0, math.inf)
    assert e.value.status == "INVALID_ARG"
    # a failed call leaves the library usable, on its stream and on another
    # (a pass queued ahead of the failure is stopped, not left waiting)
    res = nn.icp_align(t, dev(c.source), 5, 0.0, math.inf)
    assert res["iters"] == 5
    import torch
    s = torch.cuda.Stream()
    with pytest.raises(nn.IcpnnError):
        nn.icp_align(t, far, 5, 1e-6, 0.1, stream=s)
    res2 = nn.icp_align(t, dev(c.source), 5, 0.0, math.inf)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(res2["T"], res["T"])


def test_round_robin_tree_gives_the_same_registration(nn, oracle_mod):
    """Section 4.2's alternative axis rule changes the tree, not the nearest
    neighbours nor the reduction order: the registration is bit-identical."""
    c = W.lidar_case()
    src = dev(c.source)
    trees = []
    for rr in (False, True):
        t = nn.kdtree_build(c.target, c.leaf_size, round_robin=rr)
        nn.kdtree_upload(t)
        trees.append(t)
    a = nn.icp_align(trees[0], src, c.max_iter, c.eps, c.max_corr_dist[0])
    b = nn.icp_align(trees[1], src, c.max_iter, c.eps, c.max_corr_dist[0])
    np.testing.assert_array_equal(a["T"], b["T"])
    assert a["iters"] == b["iters"] and a["final_mse"] == b["final_mse"]


def test_section6_uniform200k_regression(nn, oracle_mod):
    """The page's simulation regression (section 6) at its full 200k size:
    parity with the oracle, and the convergence curve it describes (a large
    first error, a steep drop, then a jump-free approach to the noise floor)."""
    c = W.uniform200k_case()
    t, ot = setup(nn, oracle_mod, c)
    res = nn.icp_align(t, dev(c.source), c.max_iter, c.eps, math.inf, trace=True)
    _trace_parity(nn, oracle_mod, c, t, ot, c.source, math.inf, res, sample_iters=[0, 3, 6, 29])
    Ts = [r["T"] for r in res["trace"]] + [res["T"]]
    rot = np.array([rot_angle(T[:3, :3], c.T_gt[:3, :3]) for T in Ts])
    tra = np.array([np.linalg.norm(T[:3, 3] - c.T_gt[:3, 3]) for T in Ts])
    assert rot[8] < 0.01 * rot[0] and tra[8] < 0.01 * tra[0]
    for k in range(8, len(rot) - 1):
        assert rot[k + 1] <= rot[k] * 1.05 + 1e-6
    assert rot[-1] < 1e-4 and tra[-1] < 1e-3
