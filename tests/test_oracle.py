"""Pins for the CPU oracle: each check ties it to something other than itself
(hand-derived values, an independent library routine, closed forms,
invariants, brute force on tiny inputs).

Source of the method: "Implementing ICP with CUDA-KDTree"
(pwwt.cn/news/5235220), sections 2.1 (objective, SVD step), 2.2 / 3.1 / 4.2 /
5.2 (tree), 3.2 (distance, search), 3.3 (loop), 4.6 (stopping rule) and 6
(simulation regression).
"""
import math

import numpy as np
import pytest

import workloads as W
from conftest import read_fixture


# ------------------------------------------------------------ NN ----------

def _hand_nn():
    rows = read_fixture("nn_hand.txt")
    tgt = np.array([[float(v) for v in r[2:5]] for r in rows if r[0] == "target"], np.float32)
    q = np.array([[float(v) for v in r[1:4]] for r in rows if r[0] == "query"], np.float32)
    exp_idx = np.array([int(r[5]) for r in rows if r[0] == "query"], np.int32)
    exp_d2 = np.array([float(r[6]) for r in rows if r[0] == "query"], np.float32)
    return tgt, q, exp_idx, exp_d2


def test_brute_force_matches_hand_fixture(oracle_mod):
    tgt, q, exp_idx, exp_d2 = _hand_nn()
    idx, d2 = oracle_mod.nn_brute(tgt, q)
    np.testing.assert_array_equal(idx, exp_idx)
    np.testing.assert_array_equal(np.isnan(d2), np.isnan(exp_d2))
    fin = ~np.isnan(exp_d2)
    np.testing.assert_array_equal(d2[fin], exp_d2[fin])


@pytest.mark.parametrize("leaf", [1, 2, 8])
def test_tree_matches_hand_fixture(oracle_mod, leaf):
    tgt, q, exp_idx, exp_d2 = _hand_nn()
    tree = oracle_mod.KDTree(tgt, leaf)
    idx, d2 = tree.query(q)
    np.testing.assert_array_equal(idx, exp_idx)
    fin = ~np.isnan(exp_d2)
    np.testing.assert_array_equal(d2[fin], exp_d2[fin])
    assert np.isnan(d2[~fin]).all()


def test_brute_force_agrees_with_scipy_ckdtree(oracle_mod):
    """Independent library (double precision) agrees wherever float32 rounding
    cannot reorder the two nearest candidates."""
    spatial = pytest.importorskip("scipy.spatial")
    rng = np.random.default_rng(7)
    ref = rng.normal(size=(3000, 3)).astype(np.float32) * np.float32(4.0)
    q = rng.normal(size=(2000, 3)).astype(np.float32) * np.float32(4.0)
    idx, d2 = oracle_mod.nn_brute(ref, q)
    dd, ii = spatial.cKDTree(ref.astype(np.float64)).query(q.astype(np.float64), k=2)
    clear_gap = (dd[:, 1] ** 2 - dd[:, 0] ** 2) > 1e-4 * (dd[:, 1] ** 2 + 1e-30)
    assert clear_gap.mean() > 0.95
    np.testing.assert_array_equal(idx[clear_gap], ii[clear_gap, 0])
    np.testing.assert_allclose(d2.astype(np.float64), dd[:, 0] ** 2, rtol=1e-6, atol=1e-12)


def test_query_on_target_points_gives_zero_and_lowest_duplicate(oracle_mod):
    base = W.uniform_cloud(500, 11)
    ref = np.vstack([base, base[::3]])          # indices >= 500 duplicate earlier ones
    idx, d2 = oracle_mod.nn_brute(ref, ref)
    assert (d2 == 0).all()
    expect = np.arange(len(ref))
    expect[500:] = np.arange(0, 500, 3)
    np.testing.assert_array_equal(idx, expect)


def _tie_clouds():
    g = W.grid_cloud(9, 0.5, origin=(-2.0, -2.0, -2.0))                 # 729 lattice points
    rng = np.random.default_rng(3)
    dup = np.vstack([g, g[rng.permutation(len(g))[:200]]])             # duplicated points
    q_lat = W.grid_cloud(17, 0.25, origin=(-2.0, -2.0, -2.0))          # lattice + midpoints: many ties
    clustered = W.gaussian_mixture(3000, rng, rng.uniform(-5, 5, (6, 3)), rng.uniform(0.05, 0.5, 6))
    flat = W.uniform_cloud(2000, 5)
    flat[:, 2] = 0.0                                                    # a plane: zero-variance axis
    line = np.zeros((300, 3), np.float32)
    line[:, 0] = np.repeat(np.arange(100, dtype=np.float32), 3)        # collinear, triplicated
    return {
        "grid": (g, q_lat),
        "dup": (dup, q_lat),
        "clustered": (clustered, W.uniform_cloud(2000, 9, -6, 6)),
        "flat": (flat, W.uniform_cloud(1000, 13)),
        "line": (line, W.uniform_cloud(500, 17, -5, 105)),
    }


@pytest.mark.parametrize("name", ["grid", "dup", "clustered", "flat", "line"])
@pytest.mark.parametrize("leaf", [1, 3, 8, 16, 64])
def test_tree_search_equals_brute_force(oracle_mod, name, leaf):
    ref, q = _tie_clouds()[name]
    tree = oracle_mod.KDTree(ref, leaf)
    i_t, d_t = tree.query(q)
    i_b, d_b = oracle_mod.nn_brute(ref, q)
    np.testing.assert_array_equal(i_t, i_b)
    np.testing.assert_array_equal(d_t.view(np.uint32), d_b.view(np.uint32))


def test_tie_fixture_needs_far_side_equal_distance(oracle_mod):
    """The lattice queries include cases where the lowest-indexed of several
    equally near points lies beyond a splitting plane exactly at the best
    distance, so a search that prunes on delta^2 >= best (the page's strict
    test) would return a different index: the pruning reading is exercised."""
    ref, q = _tie_clouds()["grid"]
    tree = oracle_mod.KDTree(ref, 1)
    ex = tree.export()
    i_b, d_b = oracle_mod.nn_brute(ref, q)
    # emulate the strict rule on the oracle's own node array
    def strict_search(qp):
        best = [np.float32(np.inf), 2**31 - 1]

        def rec(n):
            if ex["left"][n] < 0:
                for k in range(ex["start"][n], ex["end"][n]):
                    p = ex["leaf_index"][k]
                    dv = ref[p] - qp
                    d = np.float32(np.float32(dv[0] * dv[0]) + np.float32(dv[1] * dv[1]))
                    d = np.float32(d + np.float32(dv[2] * dv[2]))
                    if d < best[0] or (d == best[0] and p < best[1]):
                        best[0], best[1] = d, p
                return
            a = qp[ex["split_dim"][n]]
            s = ex["split_val"][n]
            near, far = (ex["left"][n], ex["right"][n]) if a < s else (ex["right"][n], ex["left"][n])
            rec(near)
            dl = np.float32(a - s)
            if np.float32(dl * dl) < best[0]:
                rec(far)
        rec(0)
        return best[1]
    sample = np.arange(0, len(q), 7)
    strict = np.array([strict_search(q[i]) for i in sample])
    assert (strict != i_b[sample]).any()


# ------------------------------------------------------------ tree --------

def _check_tree(ref, leaf, max_depth, ex, depth_reported, round_robin=False):
    n = len(ref)
    assert sorted(ex["leaf_index"].tolist()) == list(range(n))
    covered = np.zeros(n, int)
    max_seen = [0]

    def rec(node, lo, hi, depth):
        max_seen[0] = max(max_seen[0], depth)
        assert ex["start"][node] == lo and ex["end"][node] == hi
        members = ex["leaf_index"][lo:hi]
        count = hi - lo
        if ex["left"][node] < 0:
            assert ex["right"][node] < 0
            assert count <= leaf or depth == max_depth
            covered[lo:hi] += 1
            return
        assert count > leaf and depth < max_depth
        assert ex["left"][node] == node + 1                      # preorder: left child next
        d = ex["split_dim"][node]
        s = ex["split_val"][node]
        pts = ref[members].astype(np.float64)
        if round_robin:
            assert d == depth % 3                                # section 4.2 alternative
        else:
            var = pts.var(axis=0)                                # numpy population variance
            assert d == int(np.flatnonzero(var >= var.max() * (1 - 1e-9))[0])
        m = count // 2
        keys_l = [(ref[p, d], p) for p in members[:m]]
        keys_r = [(ref[p, d], p) for p in members[m:]]
        assert max(keys_l) < min(keys_r)                         # partition by (coord, index)
        assert s == min(keys_r)[0]                               # split = coordinate of the median
        rec(ex["left"][node], lo, lo + m, depth + 1)
        rec(ex["right"][node], lo + m, hi, depth + 1)

    rec(0, 0, n, 0)
    assert (covered == 1).all()
    assert max_seen[0] == depth_reported


@pytest.mark.parametrize("name", ["grid", "dup", "clustered", "flat", "line"])
@pytest.mark.parametrize("leaf", [1, 8, 12])
def test_tree_invariants(oracle_mod, name, leaf):
    ref, _ = _tie_clouds()[name]
    tree = oracle_mod.KDTree(ref, leaf)
    _check_tree(ref, leaf, oracle_mod.DEPTH_CAP, tree.export(), tree.depth)


def test_depth_cap_makes_big_leaves(oracle_mod):
    ref = W.uniform_cloud(1000, 21)
    tree = oracle_mod.KDTree(ref, 1, max_depth=4)
    ex = tree.export()
    _check_tree(ref, 1, 4, ex, tree.depth)
    leaves = ex["left"] < 0
    sizes = ex["end"][leaves] - ex["start"][leaves]
    assert tree.depth == 4 and leaves.sum() == 16 and sizes.sum() == 1000
    assert sizes.min() == 1000 // 16 and sizes.max() == -(-1000 // 16)
    q = W.uniform_cloud(300, 22)
    np.testing.assert_array_equal(tree.query(q)[0], oracle_mod.nn_brute(ref, q)[0])


def test_tree_depth_matches_median_arithmetic(oracle_mod):
    """With median splits the node sizes at depth k are floor/ceil(n / 2^k), so
    the depth is the first k with ceil(n / 2^k) <= leaf_size."""
    for n, leaf in [(100_000, 12), (4096, 8), (1000, 16), (7, 1), (1, 8)]:
        ref = W.uniform_cloud(n, n)
        tree = oracle_mod.KDTree(ref, leaf)
        k = 0
        while -(-n // 2 ** k) > leaf:
            k += 1
        assert tree.depth == k, (n, leaf)


# ------------------------------------------------------------ transform ---

def test_transform_exact_cases(oracle_mod):
    s = W.grid_cloud(4, 0.5, origin=(-1, -1, -1))
    I = np.eye(3, dtype=np.float32)
    np.testing.assert_array_equal(oracle_mod.transform(I, np.zeros(3), s), s)
    Rz = np.array([[0, -1, 0], [1, 0, 0], [0, 0, 1]], np.float32)   # 90 deg about z
    t = np.array([0.5, -2.0, 4.0], np.float32)
    expect = np.stack([-s[:, 1] + t[0], s[:, 0] + t[1], s[:, 2] + t[2]], 1)
    np.testing.assert_array_equal(oracle_mod.transform(Rz, t, s), expect)


def test_transform_error_bound_vs_double(oracle_mod):
    rng = np.random.default_rng(5)
    R = W.axis_angle_matrix(W.random_unit_vector(rng), 0.7).astype(np.float32)
    t = np.array([3.5, -1.25, 20.0], np.float32)
    s = (rng.normal(size=(5000, 3)) * 30).astype(np.float32)
    p = oracle_mod.transform(R, t, s).astype(np.float64)
    exact = s.astype(np.float64) @ R.astype(np.float64).T + t.astype(np.float64)
    # four roundings of terms no larger than |R||s| + |t|
    bound = 4 * 2.0 ** -24 * (np.abs(s.astype(np.float64)) @ np.abs(R.astype(np.float64)).T + np.abs(t)) * 1.01
    assert (np.abs(p - exact) <= bound).all()


# ------------------------------------------------------------ Kabsch ------

def _hand_kabsch(case):
    rows = read_fixture("kabsch_hand.txt")
    pairs = np.array([[float(v) for v in r[2:8]] for r in rows if r[0] == "pair" and r[1] == case])
    exp = [r for r in rows if r[0] == "expect" and r[1] == case][0]
    vals = np.array([float(v) for v in exp[2:]])
    return pairs[:, :3], pairs[:, 3:], vals[:9].reshape(3, 3), vals[9:]


@pytest.mark.parametrize("case", ["A", "B"])
def test_kabsch_hand_fixture(oracle_mod, case):
    S, Q, R_exp, t_exp = _hand_kabsch(case)
    R, t, _ = oracle_mod.kabsch(S, Q)
    np.testing.assert_allclose(R, R_exp, atol=1e-12)
    np.testing.assert_allclose(t, t_exp, atol=1e-12)
    assert abs(np.linalg.det(R) - 1.0) < 1e-12


def test_kabsch_recovers_random_rigid_motion(oracle_mod):
    rng = np.random.default_rng(8)
    for _ in range(20):
        R_true = W.axis_angle_matrix(W.random_unit_vector(rng), rng.uniform(0, math.pi))
        t_true = rng.normal(size=3) * 10
        S = rng.normal(size=(50, 3)) * 5
        Q = S @ R_true.T + t_true
        R, t, _ = oracle_mod.kabsch(S, Q)
        # arccos((tr - 1) / 2) only resolves angles down to ~1e-8 rad near 0,
        # so compare the matrices themselves
        assert np.abs(R - R_true).max() < 1e-12
        np.testing.assert_allclose(t, t_true, atol=1e-10)
        np.testing.assert_allclose(R.T @ R, np.eye(3), atol=1e-12)
        assert abs(np.linalg.det(R) - 1) < 1e-12


def test_kabsch_is_optimal_and_proper_for_mirrored_cloud(oracle_mod):
    """A mirrored non-planar cloud has no exact proper fit: the result must be
    a rotation (det +1) with residual no larger than any other rotation's."""
    rng = np.random.default_rng(9)
    S = rng.normal(size=(40, 3)) * np.array([3.0, 2.0, 1.0])
    Q = S * np.array([-1.0, 1.0, 1.0])
    R, t, _ = oracle_mod.kabsch(S, Q)
    assert abs(np.linalg.det(R) - 1) < 1e-12

    def E(R_, t_):
        return float(np.sum((S @ R_.T + t_ - Q) ** 2))
    e0 = E(R, t)
    for _ in range(200):
        Rp = W.axis_angle_matrix(W.random_unit_vector(rng), rng.uniform(0, 0.3)) @ R
        tp = Q.mean(0) - Rp @ S.mean(0)
        assert E(Rp, tp) >= e0 - 1e-9


def test_kabsch_degenerate_inputs(oracle_mod):
    with pytest.raises(oracle_mod.DegenerateError):
        oracle_mod.kabsch(np.zeros((2, 3)), np.zeros((2, 3)))
    line = np.outer(np.arange(10.0), [1.0, 2.0, 3.0])
    with pytest.raises(oracle_mod.DegenerateError):
        oracle_mod.kabsch(line, line + 1.0)


# ------------------------------------------------------------ ICP ---------

def test_icp_tiny_recovers_ground_truth(oracle_mod):
    c = W.tiny_case()
    tree = oracle_mod.KDTree(c.target, c.leaf_size)
    r = oracle_mod.icp_align(tree, c.source, c.max_iter, c.eps, c.max_corr_dist[0])
    assert r["iters"] < c.max_iter
    # noise 0.002 per coordinate over 4096 pairs: errors far below the noise level
    assert oracle_mod.rotation_error(r["T"][:3, :3], c.T_gt[:3, :3]) < 3e-4
    assert np.linalg.norm(r["T"][:3, 3] - c.T_gt[:3, 3]) < 5e-4
    assert abs(r["final_mse"] - 3 * 0.002 ** 2) < 0.5 * 3 * 0.002 ** 2
    R = r["T"][:3, :3]
    np.testing.assert_allclose(R.T @ R, np.eye(3), atol=1e-12)
    assert abs(np.linalg.det(R) - 1) < 1e-12


def test_icp_energy_decreases_without_rejection(oracle_mod):
    """Section 2.1: the two alternating steps never increase E.  Checked per
    iteration in double: the solve cannot raise E on the same pairs, and the
    next correspondence pass cannot raise it either (slack for float32)."""
    c = W.tiny_case()
    tree = oracle_mod.KDTree(c.target, c.leaf_size)
    r = oracle_mod.icp_align(tree, c.source, c.max_iter, 0.0, math.inf)
    src = c.source.astype(np.float64)
    tr = r["trace"]
    for k in range(len(tr) - 1):
        st = oracle_mod.icp_step(tree, c.source, tr[k]["T"], math.inf)
        Q = c.target[st["idx"]].astype(np.float64)
        T1 = tr[k + 1]["T"]
        e_before = np.sum((src @ tr[k]["T"][:3, :3].T + tr[k]["T"][:3, 3] - Q) ** 2)
        e_solved = np.sum((src @ T1[:3, :3].T + T1[:3, 3] - Q) ** 2)
        assert e_solved <= e_before * (1 + 1e-9)
        assert tr[k + 1]["mse"] * len(src) <= e_solved * (1 + 1e-5) + 1e-9


def test_icp_noise_free_converges_exactly(oracle_mod):
    rng = np.random.default_rng(12)
    target = W.uniform_cloud(3000, 12)
    R_true = W.axis_angle_matrix(W.random_unit_vector(rng), math.radians(6))
    t_true = np.array([0.03, 0.02, -0.04])
    src = ((target.astype(np.float64) - t_true) @ R_true).astype(np.float32)
    tree = oracle_mod.KDTree(target, 8)
    r = oracle_mod.icp_align(tree, src, 40, 1e-12, math.inf)
    assert oracle_mod.rotation_error(r["T"][:3, :3], R_true) < 1e-6
    assert np.linalg.norm(r["T"][:3, 3] - t_true) < 1e-6
    assert r["final_mse"] < 1e-12


def test_icp_rejection_counts_follow_threshold(oracle_mod):
    c = W.tiny_case()
    tree = oracle_mod.KDTree(c.target, c.leaf_size)
    st_all = oracle_mod.icp_step(tree, c.source, np.eye(4), math.inf)
    dmax = float(np.sqrt(np.median(st_all["d2"].astype(np.float64))))
    st = oracle_mod.icp_step(tree, c.source, np.eye(4), dmax)
    assert st["n_accepted"] == int(np.sum(st_all["d2"].astype(np.float64) <= dmax * dmax))
    assert 0 < st["n_accepted"] < len(c.source)


def test_icp_degenerate_when_nothing_accepted(oracle_mod):
    c = W.tiny_case()
    tree = oracle_mod.KDTree(c.target, c.leaf_size)
    with pytest.raises(oracle_mod.DegenerateError):
        oracle_mod.icp_align(tree, c.source + np.float32(100.0), 5, 1e-6, 0.1)


def test_rotation_error_formula():
    import oracle
    R = W.axis_angle_matrix([0, 0, 1], 0.25)
    assert abs(oracle.rotation_error(R, np.eye(3)) - 0.25) < 1e-12


# ------------------------------------------------------------ residual rejection

def _with_outliers(c, frac=0.03, seed=4):
    return W.with_outliers(c.source, frac, 0.15, seed)


def test_residual_rejection_drops_planted_outliers(oracle_mod):
    """Section 4.4: pairs beyond 3 sigma after the solve are dropped and the
    solve repeated.  Points displaced by 0.15 m in a cloud aligned to 0.002 m
    must be the ones dropped, and the recovered motion must improve."""
    c = W.tiny_case()
    src, bad = _with_outliers(c)
    tree = oracle_mod.KDTree(c.target, c.leaf_size)
    st = oracle_mod.icp_step(tree, src, c.T_gt, math.inf)
    T1 = oracle_mod.solve_from_step(st, src, tree)
    rr = oracle_mod.residual_reject(st, src, tree, T1, 3.0)
    dropped = np.flatnonzero(st["accepted"] & ~rr["kept"])
    assert len(dropped) > 0
    assert np.isin(dropped, bad).mean() > 0.95            # what it drops are outliers
    assert rr["n_kept"] + len(dropped) == st["n_accepted"]
    e_all = oracle_mod.rotation_error(T1[:3, :3], c.T_gt[:3, :3])
    e_rej = oracle_mod.rotation_error(rr["T"][:3, :3], c.T_gt[:3, :3])
    assert e_rej < 0.5 * e_all
    assert np.linalg.norm(rr["T"][:3, 3] - c.T_gt[:3, 3]) < np.linalg.norm(T1[:3, 3] - c.T_gt[:3, 3])


def test_residual_rule_and_sigma(oracle_mod):
    """sigma^2 is the mean squared residual of the accepted pairs under the
    first solve, recomputed here in double from the pairs themselves; the kept
    set is exactly the pairs within 3 sigma."""
    c = W.tiny_case()
    src, _ = _with_outliers(c, 0.02, 9)
    tree = oracle_mod.KDTree(c.target, c.leaf_size)
    st = oracle_mod.icp_step(tree, src, np.eye(4), math.inf)
    T1 = oracle_mod.solve_from_step(st, src, tree)
    rr = oracle_mod.residual_reject(st, src, tree, T1, 3.0)
    acc = st["accepted"]
    S = src[acc].astype(np.float64)
    Q = c.target[st["idx"][acc]].astype(np.float64)
    res = S @ T1[:3, :3].T + T1[:3, 3] - Q
    e2 = np.sum(res * res, axis=1)
    assert abs(rr["sigma2"] - e2.mean()) <= 1e-5 * e2.mean()
    near = np.abs(e2 - 9 * e2.mean()) < 1e-5 * e2.mean()
    np.testing.assert_array_equal(rr["kept"][acc][~near], (e2 <= 9 * e2.mean())[~near])


def test_icp_with_residual_rejection_recovers_through_outliers(oracle_mod):
    c = W.tiny_case()
    src, _ = _with_outliers(c, 0.05, 11)
    tree = oracle_mod.KDTree(c.target, c.leaf_size)
    plain = oracle_mod.icp_align(tree, src, c.max_iter, c.eps, math.inf)
    robust = oracle_mod.icp_align(tree, src, c.max_iter, c.eps, math.inf, residual_sigma=3.0)
    e_plain = oracle_mod.rotation_error(plain["T"][:3, :3], c.T_gt[:3, :3])
    e_rob = oracle_mod.rotation_error(robust["T"][:3, :3], c.T_gt[:3, :3])
    assert e_rob < e_plain
    assert all(r["n_inliers"] < r["n_accepted"] for r in robust["trace"])


# ------------------------------------------------------------ voxel grid

def _hand_voxel():
    from conftest import read_fixture
    rows = read_fixture("voxel_hand.txt")
    pts = np.array([[float(v) for v in r[1:4]] for r in rows if r[0] == "point"], np.float32)
    exp = np.array([[float(v) for v in r[1:4]] for r in rows if r[0] == "expect"], np.float64)
    return pts, exp.astype(np.float32)


def test_voxel_hand_fixture(oracle_mod):
    pts, exp = _hand_voxel()
    np.testing.assert_array_equal(oracle_mod.voxel_downsample(pts, 0.5), exp)


@pytest.mark.parametrize("v", [0.05, 0.1, 0.37])
def test_voxel_against_numpy_grouping(oracle_mod, v):
    """Voxel membership and order from numpy's float32 floor and unique; means
    from numpy in double (summation order may differ: within 1 float ulp)."""
    rng = np.random.default_rng(17)
    pts = (rng.normal(size=(20000, 3)) * np.array([2.0, 1.0, 0.5])).astype(np.float32)
    pts[::97] = pts[1::97]                                   # duplicates
    got = oracle_mod.voxel_downsample(pts, v)
    keys = np.floor(pts / np.float32(v)).astype(np.int64)
    uniq, inv = np.unique(keys, axis=0, return_inverse=True)
    inv = inv.reshape(-1)
    sums = np.zeros((len(uniq), 3))
    np.add.at(sums, inv, pts.astype(np.float64))
    means = (sums / np.bincount(inv)[:, None]).astype(np.float32)
    assert got.shape == means.shape
    np.testing.assert_array_almost_equal_nulp(got, means, nulp=1)


def test_voxel_degenerate_inputs(oracle_mod):
    assert oracle_mod.voxel_downsample(np.zeros((0, 3), np.float32), 0.1).shape == (0, 3)
    one = np.array([[1.5, -2.5, 3.25]], np.float32)
    np.testing.assert_array_equal(oracle_mod.voxel_downsample(one, 0.1), one)
    same = np.tile(np.array([[0.01, 0.02, 0.03]], np.float32), (1000, 1))
    assert oracle_mod.voxel_downsample(same, 1.0).shape == (1, 3)
    allnan = np.full((5, 3), np.nan, np.float32)
    assert oracle_mod.voxel_downsample(allnan, 1.0).shape == (0, 3)


# ------------------------------------------------------------ round robin, section 6

@pytest.mark.parametrize("name", ["grid", "clustered", "flat", "line"])
def test_round_robin_tree_invariants_and_search(oracle_mod, name):
    ref, q = _tie_clouds()[name]
    tree = oracle_mod.KDTree(ref, 4, round_robin=True)
    _check_tree(ref, 4, oracle_mod.DEPTH_CAP, tree.export(), tree.depth, round_robin=True)
    i_t, d_t = tree.query(q)
    i_b, d_b = oracle_mod.nn_brute(ref, q)
    np.testing.assert_array_equal(i_t, i_b)
    np.testing.assert_array_equal(d_t.view(np.uint32), d_b.view(np.uint32))


def test_section6_regression_curve(oracle_mod):
    """The page's simulation regression (section 6), at 40k points: a large
    error on the first iteration, a steep drop within five, then a slow,
    jump-free approach to the noise floor; the final motion near the truth."""
    c = W.uniform200k_case(40_000)
    tree = oracle_mod.KDTree(c.target, c.leaf_size)
    r = oracle_mod.icp_align(tree, c.source, c.max_iter, c.eps, math.inf)
    Ts = [x["T"] for x in r["trace"]] + [r["T"]]
    rot = np.array([oracle_mod.rotation_error(T[:3, :3], c.T_gt[:3, :3]) for T in Ts])
    tra = np.array([np.linalg.norm(T[:3, 3] - c.T_gt[:3, 3]) for T in Ts])
    assert rot[5] < 0.1 * rot[0] and tra[5] < 0.2 * tra[0]
    for k in range(5, len(rot) - 1):
        assert rot[k + 1] <= rot[k] * 1.05 + 1e-6
        assert tra[k + 1] <= tra[k] * 1.05 + 1e-6
    assert rot[-1] < 1e-4 and tra[-1] < 1e-3


def test_threaded_query_equals_serial(oracle_mod):
    """Splitting the queries over host threads changes nothing in the result."""
    ref = W.uniform_cloud(20000, 91)
    q = W.uniform_cloud(7001, 92, -1.1, 1.1)
    tree = oracle_mod.KDTree(ref, 12)
    i1, d1 = tree.query(q)
    i4, d4 = tree.query(q, workers=4)
    np.testing.assert_array_equal(i1, i4)
    np.testing.assert_array_equal(d1.view(np.uint32), d4.view(np.uint32))
