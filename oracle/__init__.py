"""CPU oracle for KD-tree ICP registration -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the CPU-baseline leg of the benchmark use
this package; the library never does, and it shares no code with the CUDA
path.  The float32 steps (nearest neighbour, KD-tree search, transform) are
plain C in ``icp_oracle.c``; the double-precision Kabsch solve and the ICP
loop are NumPy, with LAPACK's SVD (``numpy.linalg.svd``) as the SVD step.

Source: "Implementing ICP with CUDA-KDTree" (pwwt.cn/news/5235220).

* ``kabsch``   -- section 2.1: centroids of both point sets, de-meaned
                  coordinates, H, SVD, rotation from U and V, translation from
                  the centroid difference.  Convention (the page writes
                  "R = U V^T" without fixing which way H is formed):
                  H = sum (s - mu_s)(q - mu_q)^T, H = U S V^T,
                  R = V diag(1, 1, sign det(V U^T)) U^T, t = mu_q - R mu_s.
                  The reflection guard is the textbook Kabsch/Umeyama one
                  (not on the page).
* ``icp_step`` -- one iteration of the section 3.3 main loop: transform the
                  *original* source with the accumulated (R, t), find the
                  nearest target point of every transformed point, drop pairs
                  farther than the maximum correspondence distance (section
                  4.4), reduce the pairs (original s_i, matched q_i) to
                  centroids and H.
* ``icp_align`` -- the loop with the section 4.6 stopping rule: stop once the
                  change of the mean squared correspondence distance has
                  stayed below eps for two consecutive iterations, or at
                  max_iter.
* ``voxel_downsample`` -- section 4.3: one centroid per occupied voxel,
                  applied before the tree is built.
* ``residual_reject`` -- section 4.4's second defence against outliers:
                  after the solve, compute every accepted pair's residual,
                  drop pairs beyond n_sigma standard deviations and solve
                  once more (the page recommends 3 sigma, combined with the
                  maximum correspondence distance).

Readings (the page is silent or loose on these):
  - eps is absolute, on mse_k = (sum of accepted d2) / (number accepted);
  - "held for two rounds" = |mse_{k-1} - mse_k| < eps and
    |mse_{k-2} - mse_{k-1}| < eps;
  - the kernel-side transform uses the float32 rounding of the double
    (R, t); pairs use the original float32 source coordinates, widened to
    double;
  - a pair is accepted iff it has a match and double(d2) <= dmax^2 (no
    rejection when dmax is infinite or <= 0);
  - fewer than 3 accepted pairs, or H of rank < 2 (sigma_2 <= 1e-12 sigma_1),
    is degenerate;
  - the reported error is the mse under the returned transform (one extra
    correspondence pass, no solve);
  - residual rejection: residual e_i = |R' s_i + t' - q_i| of each accepted
    pair under the first solve (R', t') of the iteration, evaluated like the
    search (float32 transform of the original s_i with float32(R', t'),
    float32 squared distance); sigma^2 = mean of e_i^2 over the accepted pairs
    (the residual vectors of a least-squares rigid fit have zero mean, so
    this is their variance); keep pairs with e_i^2 <= (n_sigma sigma)^2,
    compared in double; the iteration's transform is the solve over the kept
    pairs; the stopping rule still uses the mse of the correspondence pass.

Parity pins (tests/test_oracle.py): hand-derived NN fixture, scipy cKDTree
cross-check, tree search == brute force on tie-heavy clouds, tree
invariants, exact transform cases, exact recovery of known rigid motions,
orthonormality / det +1, reflection guard, monotone ICP energy and
ground-truth recovery on the tiny case.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "icp_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libicp_oracle.so")
_lib = None

DEPTH_CAP = 20  # section 5.2 of the page


class DegenerateError(RuntimeError):
    pass


class NonFiniteError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile icp_oracle.c into libicp_oracle.so next to it."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB_PATH)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    i32 = ctypes.c_int32
    lib.orc_nn_brute.argtypes = [P, i64, P, i64, P, P]
    lib.orc_nn_brute.restype = None
    lib.orc_transform.argtypes = [P, P, P, i64, P]
    lib.orc_transform.restype = None
    lib.orc_tree_build.argtypes = [P, i64, i32, i32, i32, ctypes.POINTER(P)]
    lib.orc_tree_build.restype = ctypes.c_int
    lib.orc_tree_free.argtypes = [P]
    lib.orc_tree_free.restype = None
    lib.orc_tree_num_nodes.argtypes = [P]
    lib.orc_tree_num_nodes.restype = i64
    lib.orc_tree_depth.argtypes = [P]
    lib.orc_tree_depth.restype = i32
    lib.orc_tree_export.argtypes = [P] * 8
    lib.orc_tree_export.restype = None
    lib.orc_tree_nn.argtypes = [P, P, i64, P, P, P, P]
    lib.orc_tree_nn.restype = None
    lib.orc_pair_dist2.argtypes = [P, P, i64, P]
    lib.orc_pair_dist2.restype = None
    lib.orc_voxel_downsample.argtypes = [P, i64, ctypes.c_float, P]
    lib.orc_voxel_downsample.restype = i64
    _lib = lib
    return lib


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32).reshape(-1, 3))


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


# ------------------------------------------------------------------ NN ----

def nn_brute(reference, queries):
    """Exact 1-NN by exhaustive search: (idx int32, d2 float32)."""
    lib = _load()
    ref = _f32(reference)
    q = _f32(queries)
    idx = np.empty(len(q), np.int32)
    d2 = np.empty(len(q), np.float32)
    lib.orc_nn_brute(_ptr(ref), len(ref), _ptr(q), len(q), _ptr(idx), _ptr(d2))
    return idx, d2


def pair_dist2(q, p) -> np.ndarray:
    """float32 squared distance of each pair (q_i, p_i), search arithmetic."""
    lib = _load()
    q = _f32(q)
    p = _f32(p)
    out = np.empty(len(q), np.float32)
    lib.orc_pair_dist2(_ptr(q), _ptr(p), len(q), _ptr(out))
    return out


def voxel_downsample(points, voxel: float) -> np.ndarray:
    """Section 4.3 voxel-grid filter: centroids of the occupied voxels of side
    `voxel` (float32), ordered by voxel index (see icp_oracle.c)."""
    lib = _load()
    pts = _f32(points)
    out = np.empty((max(len(pts), 1), 3), np.float32)
    m = lib.orc_voxel_downsample(_ptr(pts), len(pts), float(np.float32(voxel)), _ptr(out))
    if m < 0:
        raise ValueError("oracle voxel downsampling failed")
    return out[:m].copy()


def transform(R, t, source) -> np.ndarray:
    """p = R s + t in float32, fixed evaluation order (see icp_oracle.c)."""
    lib = _load()
    R32 = np.ascontiguousarray(np.asarray(R, np.float32).reshape(9))
    t32 = np.ascontiguousarray(np.asarray(t, np.float32).reshape(3))
    s = _f32(source)
    out = np.empty_like(s)
    lib.orc_transform(_ptr(R32), _ptr(t32), _ptr(s), len(s), _ptr(out))
    return out


class KDTree:
    """The oracle's own KD-tree (page layout: 24-byte nodes in preorder)."""

    def __init__(self, points, leaf_size: int, max_depth: int = DEPTH_CAP, round_robin: bool = False):
        lib = _load()
        self.points = _f32(points)
        self.leaf_size = int(leaf_size)
        self.max_depth = int(max_depth)
        self.round_robin = bool(round_robin)
        h = ctypes.c_void_p()
        rc = lib.orc_tree_build(_ptr(self.points), len(self.points), self.leaf_size,
                                self.max_depth, int(self.round_robin), ctypes.byref(h))
        if rc != 0:
            raise ValueError(f"oracle tree build failed ({rc})")
        self._h = h
        self.n_nodes = int(lib.orc_tree_num_nodes(h))
        self.depth = int(lib.orc_tree_depth(h))

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and _lib is not None:
            _lib.orc_tree_free(h)
            self._h = None

    def export(self) -> dict:
        m = self.n_nodes
        out = {
            "split_val": np.empty(m, np.float32),
            "split_dim": np.empty(m, np.int32),
            "left": np.empty(m, np.int32),
            "right": np.empty(m, np.int32),
            "start": np.empty(m, np.int32),
            "end": np.empty(m, np.int32),
            "leaf_index": np.empty(len(self.points), np.int32),
        }
        _lib.orc_tree_export(self._h, *[_ptr(out[k]) for k in
                                        ("split_val", "split_dim", "left", "right",
                                         "start", "end", "leaf_index")])
        return out

    def query(self, queries, counts: bool = False, workers: int = 1):
        """Exact 1-NN of every query.  workers > 1 splits the queries into
        contiguous chunks searched by that many host threads (each query's
        search is the same; only the timing changes)."""
        q = _f32(queries)
        idx = np.empty(len(q), np.int32)
        d2 = np.empty(len(q), np.float32)
        nodes = np.empty(len(q), np.int64) if counts else None
        pts = np.empty(len(q), np.int64) if counts else None

        def run_range(a, b):
            # ctypes releases the GIL for the duration of the C call
            _lib.orc_tree_nn(self._h, _ptr(q[a:b]), b - a, _ptr(idx[a:b]), _ptr(d2[a:b]),
                             _ptr(nodes[a:b]) if counts else None, _ptr(pts[a:b]) if counts else None)

        if workers > 1 and len(q) >= 2 * workers:
            from concurrent.futures import ThreadPoolExecutor
            bounds = np.linspace(0, len(q), workers + 1).astype(np.int64)
            with ThreadPoolExecutor(workers) as ex:
                list(ex.map(lambda k: run_range(int(bounds[k]), int(bounds[k + 1])), range(workers)))
        elif len(q):
            run_range(0, len(q))
        return (idx, d2, nodes, pts) if counts else (idx, d2)


# -------------------------------------------------------------- Kabsch ----

def kabsch(S, Q):
    """Rigid (R, t) minimising sum ||R s_i + t - q_i||^2 over pairs (s_i, q_i).

    Returns (R, t, info) with info = {mu_s, mu_q, H, sigma}."""
    S = np.asarray(S, np.float64).reshape(-1, 3)
    Q = np.asarray(Q, np.float64).reshape(-1, 3)
    if len(S) < 3:
        raise DegenerateError("fewer than 3 correspondences")
    mu_s = S.mean(axis=0)
    mu_q = Q.mean(axis=0)
    H = (S - mu_s).T @ (Q - mu_q)
    U, sig, Vt = np.linalg.svd(H)
    if not (sig[0] > 0.0) or sig[1] <= 1e-12 * sig[0]:
        raise DegenerateError("cross-covariance of rank < 2")
    V = Vt.T
    d = 1.0 if np.linalg.det(V @ U.T) >= 0.0 else -1.0
    R = V @ np.diag([1.0, 1.0, d]) @ U.T
    t = mu_q - R @ mu_s
    return R, t, {"mu_s": mu_s, "mu_q": mu_q, "H": H, "sigma": sig}


def as_kernel_rt(T):
    """The float32 (R, t) a correspondence pass uses for the double transform T."""
    T = np.asarray(T, np.float64)
    return T[:3, :3].astype(np.float32), T[:3, 3].astype(np.float32)


def accept_mask(idx, d2, max_corr_dist):
    ok = idx >= 0
    if max_corr_dist is not None and np.isfinite(max_corr_dist) and max_corr_dist > 0:
        ok &= d2.astype(np.float64) <= float(max_corr_dist) ** 2
    return ok


# ----------------------------------------------------------------- ICP ----

def icp_step(tree: KDTree, source, T, max_corr_dist, workers: int = 1, nn=None):
    """One correspondence + reduction pass under transform T (double 4x4).

    nn: optional (idx, d2) already found by this tree for exactly the points
    this pass queries (the float32 transform of the source under T), to skip
    the search.

    Returns a dict: idx, d2 (per source point), accepted mask, n_accepted,
    mse, mu_s, mu_q, H (None when nothing is accepted)."""
    src = _f32(source)
    if not np.all(np.isfinite(src)):
        raise NonFiniteError("non-finite source point")
    if nn is not None:
        idx, d2 = nn
    else:
        R32, t32 = as_kernel_rt(T)
        p = transform(R32, t32, src)
        idx, d2 = tree.query(p, workers=workers)
    acc = accept_mask(idx, d2, max_corr_dist)
    n_acc = int(acc.sum())
    out = {"idx": idx, "d2": d2, "accepted": acc, "n_accepted": n_acc,
           "mse": float(np.sum(d2[acc].astype(np.float64)) / n_acc) if n_acc else float("nan"),
           "mu_s": None, "mu_q": None, "H": None}
    if n_acc:
        S = src[acc].astype(np.float64)
        Q = tree.points[idx[acc]].astype(np.float64)
        out["mu_s"] = S.mean(axis=0)
        out["mu_q"] = Q.mean(axis=0)
        out["H"] = (S - out["mu_s"]).T @ (Q - out["mu_q"])
    return out


def solve_from_step(step, source, tree: KDTree):
    acc = step["accepted"]
    if step["n_accepted"] < 3:
        raise DegenerateError("fewer than 3 accepted correspondences")
    S = _f32(source)[acc]
    Q = tree.points[step["idx"][acc]]
    R, t, _ = kabsch(S, Q)
    T = np.eye(4)
    T[:3, :3] = R
    T[:3, 3] = t
    return T


def residual_reject(step, source, tree: KDTree, T1, n_sigma: float):
    """Residuals of the accepted pairs under the first solve T1, the sigma
    rule, and the solve over the kept pairs.  Returns dict(T, kept (mask over
    the source), n_kept, sigma2, e2 (per accepted pair))."""
    acc = step["accepted"]
    src = _f32(source)
    S = src[acc]
    Q = tree.points[step["idx"][acc]]
    R32, t32 = as_kernel_rt(T1)
    e2 = pair_dist2(Q, transform(R32, t32, S))
    sigma2 = float(np.sum(e2.astype(np.float64)) / len(e2))
    keep_acc = e2.astype(np.float64) <= (n_sigma * n_sigma) * sigma2
    kept = np.zeros(len(src), bool)
    kept[np.flatnonzero(acc)[keep_acc]] = True
    if keep_acc.sum() < 3:
        raise DegenerateError("fewer than 3 pairs left after residual rejection")
    R, t, _ = kabsch(S[keep_acc], Q[keep_acc])
    T = np.eye(4)
    T[:3, :3] = R
    T[:3, 3] = t
    return {"T": T, "kept": kept, "n_kept": int(keep_acc.sum()), "sigma2": sigma2, "e2": e2}


def icp_align(tree: KDTree, source, max_iter: int, eps: float, max_corr_dist,
              init_T=None, residual_sigma: float = 0.0, workers: int = 1):
    """Section 3.3 loop with the section 4.6 stopping rule; residual_sigma > 0
    adds the section 4.4 residual rejection and re-solve to every iteration.

    Returns dict(T, iters, final_mse, trace) where trace[k] = dict(T (used for
    pass k), mse, n_accepted, n_inliers)."""
    T = np.eye(4) if init_T is None else np.asarray(init_T, np.float64).copy()
    trace = []
    mses = []
    iters = 0
    for k in range(max_iter):
        st = icp_step(tree, source, T, max_corr_dist, workers)
        if st["n_accepted"] < 3:
            raise DegenerateError("fewer than 3 accepted correspondences")
        T_next = solve_from_step(st, source, tree)
        n_in = st["n_accepted"]
        if residual_sigma > 0:
            rr = residual_reject(st, source, tree, T_next, residual_sigma)
            T_next = rr["T"]
            n_in = rr["n_kept"]
        trace.append({"T": T.copy(), "mse": st["mse"], "n_accepted": st["n_accepted"],
                      "n_inliers": n_in})
        mses.append(st["mse"])
        T = T_next
        iters = k + 1
        if (k >= 2 and abs(mses[-2] - mses[-1]) < eps
                and abs(mses[-3] - mses[-2]) < eps):
            break
    fin = icp_step(tree, source, T, max_corr_dist, workers)
    return {"T": T, "iters": iters, "final_mse": fin["mse"], "final_n_accepted": fin["n_accepted"],
            "trace": trace}


def rotation_error(R, R_true) -> float:
    """Angle (rad) of R^T R_true, from arccos((trace - 1) / 2) (section 6)."""
    c = (np.trace(np.asarray(R).T @ np.asarray(R_true)) - 1.0) / 2.0
    return float(np.arccos(np.clip(c, -1.0, 1.0)))


def traversal_bytes(nodes_visited, points_visited, node_bytes=8, point_bytes=16,
                    query_bytes=16, result_bytes=8):
    """Algorithmic bytes a single-query search touches: its query record, its
    result, every node it enters and every reference point it measures."""
    return (query_bytes + result_bytes + node_bytes * np.asarray(nodes_visited)
            + point_bytes * np.asarray(points_visited))
