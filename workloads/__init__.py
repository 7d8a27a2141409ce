"""Seeded synthetic point clouds for KD-tree ICP registration.

This module only *generates inputs*: point clouds, ground-truth rigid
transforms and the per-case parameters (leaf size, iteration cap, convergence
threshold, maximum correspondence distance).  It contains none of the
registration arithmetic itself (no nearest-neighbour search, no transform of
the method, no SVD solve), so that both the CPU oracle and the CUDA path can
consume the same inputs without sharing any code.

The real datasets of "Implementing ICP with CUDA-KDTree" (pwwt.cn/news/5235220,
introduction: four PCD clouds shipped with the project) are not available;
the generators below stand in for them.  Every generator draws from
``numpy.random.default_rng`` (PCG64) seeded with ``1000 + case number``, and
uses independent spawned sub-streams for independent draws.

Cases (sizes are the full workloads; ``scale`` shrinks the point counts for
small parity tests while keeping the structure):

1. ``tiny``     4,096 uniform points in [-1,1]^3, 10 deg / (0.05,-0.03,0.08)
                offset, N(0, 0.002) noise, leaf 8, 30 iterations, eps 1e-6,
                no distance rejection.
2. ``scene``    100k <-> 100k samples of a ground plane (40x40 m), 20 boxes and
                10 cylinders, N(0, 0.01 m) noise, offset <= 15 deg / <= 1 m,
                leaf 12, 50 iterations, max correspondence 1.0 m.
3. ``lidar``    two simulated 64-beam x 2048-column scans over a 270 deg
                sector, poses 2 m / 5 deg apart, sectors offset by 67.5 deg
                (25 % non-overlap), N(0, 0.02 m) range noise, leaf 16,
                max correspondence 0.5 m, 50 iterations.
4. ``gmm``      1M queries and 1M references from one 100-component isotropic
                Gaussian mixture (NN only), leaf 16.
5. ``large``    4M-point target, 2M-point source on the scene surfaces,
                20 deg / 3 m offset, leaf 16, max correspondence 2.0 m then
                0.3 m, 60 iterations per stage.
6. ``uniform200k`` the simulation regression of the page's section 6: 200k
                points uniform in [-25, 25]^3, source = target under a random
                rigid motion (2 deg about a random axis, |t| = 0.2 m: inside
                point-to-point ICP's basin for a 0.85 m point spacing) plus
                N(0, voxel / 10) noise with voxel 0.1 m, leaf 16, 30
                iterations, no distance rejection.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

SEED_BASE = 1000

# Convergence threshold on the change of the mean squared correspondence
# distance for the metre-scale scenes.  "Implementing ICP with CUDA-KDTree"
# section 4.6 recommends 1e-5 or 1e-4 for float32 clouds tens of metres wide.
SCENE_EPS = 1e-5


@dataclasses.dataclass
class RegistrationCase:
    """One registration problem: target, source and the parameters to run it."""

    name: str
    target: np.ndarray          # (m, 3) float32, C-contiguous
    source: np.ndarray          # (n, 3) float32, C-contiguous
    T_gt: np.ndarray            # (4, 4) float64: target ~= T_gt * source
    leaf_size: int
    max_iter: int
    eps: float
    max_corr_dist: tuple        # one entry per coarse-to-fine stage; inf = no rejection
    extent: float               # diagonal of the target's bounding box (m)
    info: dict = dataclasses.field(default_factory=dict)


@dataclasses.dataclass
class QueryCase:
    """A nearest-neighbour-only problem."""

    name: str
    reference: np.ndarray       # (m, 3) float32
    queries: np.ndarray         # (n, 3) float32
    leaf_size: int
    extent: float


# --------------------------------------------------------------------------
# small helpers for building inputs
# --------------------------------------------------------------------------

def _rngs(case_no: int, k: int):
    ss = np.random.SeedSequence(SEED_BASE + case_no)
    return [np.random.default_rng(s) for s in ss.spawn(k)]


def random_unit_vector(rng) -> np.ndarray:
    v = rng.normal(size=3)
    return v / np.linalg.norm(v)


def axis_angle_matrix(axis, angle_rad: float) -> np.ndarray:
    """Rotation matrix for ``angle_rad`` about the unit vector ``axis`` (Rodrigues)."""
    a = np.asarray(axis, dtype=np.float64)
    a = a / np.linalg.norm(a)
    K = np.array([[0.0, -a[2], a[1]], [a[2], 0.0, -a[0]], [-a[1], a[0], 0.0]])
    return np.eye(3) + math.sin(angle_rad) * K + (1.0 - math.cos(angle_rad)) * (K @ K)


def rigid(R, t) -> np.ndarray:
    T = np.eye(4)
    T[:3, :3] = R
    T[:3, 3] = t
    return T


def _apply_inverse(T: np.ndarray, pts: np.ndarray) -> np.ndarray:
    """Map world points into the frame that ``T`` maps to world (input synthesis)."""
    R = T[:3, :3]
    t = T[:3, 3]
    return (pts - t) @ R  # row-vector form of R^T (p - t)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def bbox_diagonal(pts: np.ndarray) -> float:
    if len(pts) == 0:
        return 0.0
    lo = pts.min(axis=0).astype(np.float64)
    hi = pts.max(axis=0).astype(np.float64)
    return float(np.linalg.norm(hi - lo))


# --------------------------------------------------------------------------
# generic clouds used by edge-case tests
# --------------------------------------------------------------------------

def uniform_cloud(n: int, seed: int, lo=-1.0, hi=1.0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return _f32(rng.uniform(lo, hi, size=(n, 3)))


def grid_cloud(k: int, spacing: float = 1.0, origin=(0.0, 0.0, 0.0)) -> np.ndarray:
    """k^3 points on an axis-aligned lattice: a cloud full of exact distance ties."""
    r = np.arange(k, dtype=np.float64) * spacing
    g = np.stack(np.meshgrid(r, r, r, indexing="ij"), axis=-1).reshape(-1, 3)
    return _f32(g + np.asarray(origin))


def gaussian_mixture(n: int, rng, centres: np.ndarray, sigmas: np.ndarray) -> np.ndarray:
    comp = rng.integers(0, len(centres), size=n)
    pts = centres[comp] + rng.normal(size=(n, 3)) * sigmas[comp, None]
    return _f32(pts)


def with_outliers(points: np.ndarray, frac: float, sigma: float, seed: int):
    """Copy of a cloud with a fraction of its points displaced by N(0, sigma)
    per coordinate (gross outliers for the residual rejection); returns
    (cloud, indices of the displaced points)."""
    rng = np.random.default_rng(seed)
    pts = np.array(points, dtype=np.float32, copy=True)
    bad = rng.choice(len(pts), int(frac * len(pts)), replace=False)
    pts[bad] += rng.normal(0.0, sigma, size=(len(bad), 3)).astype(np.float32)
    return pts, bad


# --------------------------------------------------------------------------
# case 1: tiny uniform cube
# --------------------------------------------------------------------------

def tiny_case(n: int = 4096) -> RegistrationCase:
    r_tgt, r_axis, r_noise, r_perm = _rngs(1, 4)
    target = r_tgt.uniform(-1.0, 1.0, size=(n, 3))
    R = axis_angle_matrix(random_unit_vector(r_axis), math.radians(10.0))
    T_gt = rigid(R, [0.05, -0.03, 0.08])
    src = _apply_inverse(T_gt, target) + r_noise.normal(0.0, 0.002, size=(n, 3))
    src = src[r_perm.permutation(n)]
    target = _f32(target)
    return RegistrationCase("tiny", target, _f32(src), T_gt, leaf_size=8, max_iter=30,
                            eps=1e-6, max_corr_dist=(math.inf,),
                            extent=bbox_diagonal(target))


# --------------------------------------------------------------------------
# box / cylinder / plane scenes (cases 2, 3, 5)
# --------------------------------------------------------------------------

@dataclasses.dataclass
class Scene:
    boxes: np.ndarray      # (B, 6): cx, cy, sx, sy, sz, unused (boxes rest on z = 0)
    cyls: np.ndarray       # (C, 4): cx, cy, r, h
    half_plane: float      # ground plane is [-half, half]^2 at z = 0 (inf = unbounded)


def make_scene(rng, n_boxes=20, n_cyls=10, half_plane=20.0, spread=18.0,
               keep_clear=None) -> Scene:
    """Random axis-aligned boxes (sides U(1,4) m) and vertical cylinders
    (r U(0.2,1) m, h U(2,6) m) standing on the ground plane, centres
    U(-spread, spread)^2.  ``keep_clear`` is a list of (x, y, radius) discs no
    primitive may overlap (used to keep LiDAR poses outside obstacles)."""

    def clear(cx, cy, rad):
        if keep_clear is None:
            return True
        return all(math.hypot(cx - x, cy - y) > rad + r for (x, y, r) in keep_clear)

    boxes = []
    while len(boxes) < n_boxes:
        cx, cy = rng.uniform(-spread, spread, size=2)
        sx, sy, sz = rng.uniform(1.0, 4.0, size=3)
        if clear(cx, cy, 0.5 * math.hypot(sx, sy)):
            boxes.append((cx, cy, sx, sy, sz, 0.0))
    cyls = []
    while len(cyls) < n_cyls:
        cx, cy = rng.uniform(-spread, spread, size=2)
        r = rng.uniform(0.2, 1.0)
        h = rng.uniform(2.0, 6.0)
        if clear(cx, cy, r):
            cyls.append((cx, cy, r, h))
    return Scene(np.array(boxes), np.array(cyls), half_plane)


def _inside_footprint(scene: Scene, x, y):
    inside = np.zeros(x.shape, dtype=bool)
    for cx, cy, sx, sy, _, _ in scene.boxes:
        inside |= (np.abs(x - cx) <= sx / 2) & (np.abs(y - cy) <= sy / 2)
    for cx, cy, r, _ in scene.cyls:
        inside |= (x - cx) ** 2 + (y - cy) ** 2 <= r * r
    return inside


def sample_scene_surfaces(scene: Scene, n: int, rng, noise_sigma: float) -> np.ndarray:
    """Area-weighted uniform samples of the visible surfaces: the ground plane
    outside the primitives' footprints, the four sides and the top of every
    box, the side and top cap of every cylinder; plus isotropic N(0, sigma)."""
    surfaces = []  # (area, sampler(k) -> (k,3))
    L = 2.0 * scene.half_plane
    foot = sum(b[2] * b[3] for b in scene.boxes) + sum(math.pi * c[2] ** 2 for c in scene.cyls)

    def plane(k):
        out = np.empty((0, 3))
        while len(out) < k:
            m = int((k - len(out)) * 1.3) + 16
            x = rng.uniform(-scene.half_plane, scene.half_plane, m)
            y = rng.uniform(-scene.half_plane, scene.half_plane, m)
            keep = ~_inside_footprint(scene, x, y)
            out = np.vstack([out, np.stack([x[keep], y[keep], np.zeros(keep.sum())], 1)])
        return out[:k]

    surfaces.append((L * L - foot, plane))
    for cx, cy, sx, sy, sz, _ in scene.boxes:
        def face(k, cx=cx, cy=cy, sx=sx, sy=sy, sz=sz, which=0):
            u = rng.uniform(-0.5, 0.5, k)
            v = rng.uniform(0.0, 1.0, k)
            if which == 0:
                return np.stack([cx + sx / 2 + 0 * u, cy + u * sy, v * sz], 1)
            if which == 1:
                return np.stack([cx - sx / 2 + 0 * u, cy + u * sy, v * sz], 1)
            if which == 2:
                return np.stack([cx + u * sx, cy + sy / 2 + 0 * u, v * sz], 1)
            if which == 3:
                return np.stack([cx + u * sx, cy - sy / 2 + 0 * u, v * sz], 1)
            w = rng.uniform(-0.5, 0.5, k)
            return np.stack([cx + u * sx, cy + w * sy, np.full(k, sz)], 1)
        for which, area in enumerate([sy * sz, sy * sz, sx * sz, sx * sz, sx * sy]):
            surfaces.append((area, lambda k, f=face, w=which: f(k, which=w)))
    for cx, cy, r, h in scene.cyls:
        def side(k, cx=cx, cy=cy, r=r, h=h):
            a = rng.uniform(0, 2 * math.pi, k)
            return np.stack([cx + r * np.cos(a), cy + r * np.sin(a), rng.uniform(0, h, k)], 1)

        def cap(k, cx=cx, cy=cy, r=r, h=h):
            a = rng.uniform(0, 2 * math.pi, k)
            rr = r * np.sqrt(rng.uniform(0, 1, k))
            return np.stack([cx + rr * np.cos(a), cy + rr * np.sin(a), np.full(k, h)], 1)
        surfaces.append((2 * math.pi * r * h, side))
        surfaces.append((math.pi * r * r, cap))

    areas = np.array([a for a, _ in surfaces])
    counts = rng.multinomial(n, areas / areas.sum())
    parts = [f(int(k)) for (_, f), k in zip(surfaces, counts) if k > 0]
    pts = np.vstack(parts)
    pts = pts[rng.permutation(len(pts))]
    return pts + rng.normal(0.0, noise_sigma, size=pts.shape)


def scene_case(n_target: int = 100_000, n_source: int = 100_000) -> RegistrationCase:
    r_scene, r_tgt, r_src, r_pose = _rngs(2, 4)
    scene = make_scene(r_scene)
    target = sample_scene_surfaces(scene, n_target, r_tgt, 0.01)
    world_src = sample_scene_surfaces(scene, n_source, r_src, 0.01)
    angle = math.radians(r_pose.uniform(0.0, 15.0))
    R = axis_angle_matrix(random_unit_vector(r_pose), angle)
    t = random_unit_vector(r_pose) * r_pose.uniform(0.0, 1.0)
    T_gt = rigid(R, t)
    source = _apply_inverse(T_gt, world_src)
    target = _f32(target)
    return RegistrationCase("scene", target, _f32(source), T_gt, leaf_size=12, max_iter=50,
                            eps=SCENE_EPS, max_corr_dist=(1.0,), extent=bbox_diagonal(target),
                            info={"angle_deg": math.degrees(angle), "t_norm": float(np.linalg.norm(t))})


def scene_frames(n_frames: int, n_target: int = 100_000, n_source: int = 100_000):
    """The scene of case 2 (same target) with n_frames independent sources:
    frame 0 is case 2's own source, frame k > 0 an independent resample of the
    same surfaces under its own offset (<= 15 deg, <= 1 m), drawn from the
    sub-stream ``SeedSequence(1002).spawn(4 + k)[-1]``.  Returns (case, [frame
    sources], [frame ground truths])."""
    case = scene_case(n_target, n_source)
    r_scene = _rngs(2, 4)[0]
    scene = make_scene(r_scene)
    srcs, gts = [case.source], [case.T_gt]
    for k in range(1, n_frames):
        rng = np.random.default_rng(np.random.SeedSequence(SEED_BASE + 2).spawn(4 + k)[-1])
        world = sample_scene_surfaces(scene, n_source, rng, 0.01)
        angle = math.radians(rng.uniform(0.0, 15.0))
        R = axis_angle_matrix(random_unit_vector(rng), angle)
        t = random_unit_vector(rng) * rng.uniform(0.0, 1.0)
        T = rigid(R, t)
        srcs.append(_f32(_apply_inverse(T, world)))
        gts.append(T)
    return case, srcs, gts


def uniform200k_case(n: int = 200_000) -> RegistrationCase:
    r_tgt, r_pose, r_noise = _rngs(6, 3)
    target = r_tgt.uniform(-25.0, 25.0, size=(n, 3))
    R = axis_angle_matrix(random_unit_vector(r_pose), math.radians(2.0))
    t = random_unit_vector(r_pose) * 0.2
    T_gt = rigid(R, t)
    src = _apply_inverse(T_gt, target) + r_noise.normal(0.0, 0.1 / 10.0, size=(n, 3))
    target = _f32(target)
    return RegistrationCase("uniform200k", target, _f32(src), T_gt, leaf_size=16, max_iter=30,
                            eps=0.0, max_corr_dist=(math.inf,), extent=bbox_diagonal(target))


def large_case(n_target: int = 4_000_000, n_source: int = 2_000_000) -> RegistrationCase:
    r_scene, r_tgt, r_src, r_pose = _rngs(5, 4)
    scene = make_scene(r_scene)
    target = sample_scene_surfaces(scene, n_target, r_tgt, 0.01)
    world_src = sample_scene_surfaces(scene, n_source, r_src, 0.01)
    R = axis_angle_matrix(random_unit_vector(r_pose), math.radians(20.0))
    t = random_unit_vector(r_pose) * 3.0
    T_gt = rigid(R, t)
    source = _apply_inverse(T_gt, world_src)
    target = _f32(target)
    return RegistrationCase("large", target, _f32(source), T_gt, leaf_size=16, max_iter=60,
                            eps=SCENE_EPS, max_corr_dist=(2.0, 0.3), extent=bbox_diagonal(target))


# ---- case 3: simulated spinning LiDAR -------------------------------------

def _ray_cast(scene: Scene, origin: np.ndarray, dirs: np.ndarray) -> np.ndarray:
    """Range to the first hit of each ray (inf where nothing is hit)."""
    ox, oy, oz = origin
    dx, dy, dz = dirs[:, 0], dirs[:, 1], dirs[:, 2]
    best = np.full(len(dirs), np.inf)
    with np.errstate(divide="ignore", invalid="ignore"):
        tp = np.where(dz < 0, -oz / dz, np.inf)
        if math.isfinite(scene.half_plane):
            hx, hy = ox + tp * dx, oy + tp * dy
            tp = np.where((np.abs(hx) <= scene.half_plane) & (np.abs(hy) <= scene.half_plane), tp, np.inf)
        best = np.minimum(best, tp)
        for cx, cy, sx, sy, sz, _ in scene.boxes:
            lo = np.array([cx - sx / 2, cy - sy / 2, 0.0])
            hi = np.array([cx + sx / 2, cy + sy / 2, sz])
            t0 = np.full(len(dirs), -np.inf)
            t1 = np.full(len(dirs), np.inf)
            for a, (o, d) in enumerate(((ox, dx), (oy, dy), (oz, dz))):
                ta = (lo[a] - o) / d
                tb = (hi[a] - o) / d
                tmin = np.where(d == 0, np.where((o >= lo[a]) & (o <= hi[a]), -np.inf, np.inf), np.minimum(ta, tb))
                tmax = np.where(d == 0, np.where((o >= lo[a]) & (o <= hi[a]), np.inf, -np.inf), np.maximum(ta, tb))
                t0 = np.maximum(t0, tmin)
                t1 = np.minimum(t1, tmax)
            hit = (t0 <= t1) & (t0 > 0)
            best = np.minimum(best, np.where(hit, t0, np.inf))
        for cx, cy, r, h in scene.cyls:
            px, py = ox - cx, oy - cy
            a = dx * dx + dy * dy
            b = 2 * (px * dx + py * dy)
            c = px * px + py * py - r * r
            disc = b * b - 4 * a * c
            ts = (-b - np.sqrt(np.maximum(disc, 0))) / (2 * a)
            z = oz + ts * dz
            side_hit = (disc >= 0) & (a > 0) & (ts > 0) & (z >= 0) & (z <= h)
            best = np.minimum(best, np.where(side_hit, ts, np.inf))
            tc = np.where(dz != 0, (h - oz) / dz, np.inf)
            cxh, cyh = px + tc * dx, py + tc * dy
            cap_hit = (tc > 0) & (cxh * cxh + cyh * cyh <= r * r)
            best = np.minimum(best, np.where(cap_hit, tc, np.inf))
    return best


def lidar_scan(scene: Scene, pose_xy, yaw: float, sector_start: float, rng,
               beams=64, columns=2048, height=1.8, range_sigma=0.02):
    """One spinning scan expressed in the sensor frame (x forward, z up)."""
    el = np.radians(np.linspace(-25.0, -1.3, beams))
    az = sector_start + np.radians(270.0) * (np.arange(columns) + 0.5) / columns
    E, A = np.meshgrid(el, az, indexing="ij")
    d_sensor = np.stack([np.cos(E) * np.cos(A), np.cos(E) * np.sin(A), np.sin(E)], -1).reshape(-1, 3)
    c, s = math.cos(yaw), math.sin(yaw)
    Rz = np.array([[c, -s, 0], [s, c, 0], [0, 0, 1.0]])
    d_world = d_sensor @ Rz.T
    origin = np.array([pose_xy[0], pose_xy[1], height])
    rng_true = _ray_cast(scene, origin, d_world)
    keep = np.isfinite(rng_true) & (rng_true >= 1.0) & (rng_true <= 80.0)
    rng_meas = rng_true[keep] + rng.normal(0.0, range_sigma, size=int(keep.sum()))
    pts = d_sensor[keep] * rng_meas[:, None]
    T_world_sensor = rigid(Rz, origin)
    return pts, T_world_sensor


def lidar_case(beams: int = 64, columns: int = 2048) -> RegistrationCase:
    r_scene, r_a, r_b, r_pose = _rngs(3, 4)
    yaw_a = r_pose.uniform(-math.pi, math.pi)
    move = random_unit_vector(r_pose)
    move[2] = 0.0
    move /= np.linalg.norm(move)
    pa = np.array([0.0, 0.0])
    pb = pa + 2.0 * move[:2]
    yaw_b = yaw_a + math.radians(5.0)
    scene = make_scene(r_scene, half_plane=math.inf,
                       keep_clear=[(pa[0], pa[1], 3.0), (pb[0], pb[1], 3.0)])
    start = r_pose.uniform(-math.pi, math.pi)
    tgt, T_wa = lidar_scan(scene, pa, yaw_a, start, r_a, beams, columns)
    src, T_wb = lidar_scan(scene, pb, yaw_b, start + math.radians(67.5), r_b, beams, columns)
    T_gt = np.linalg.inv(T_wa) @ T_wb      # source (scan B frame) -> target (scan A frame)
    target = _f32(tgt)
    return RegistrationCase("lidar", target, _f32(src), T_gt, leaf_size=16, max_iter=50,
                            eps=SCENE_EPS, max_corr_dist=(0.5,), extent=bbox_diagonal(target),
                            info={"rays": beams * columns, "n_target": len(tgt), "n_source": len(src),
                                  "sector_overlap": 1.0 - 67.5 / 270.0})


# ---- case 4: Gaussian mixture, NN only -------------------------------------

def gmm_case(n_queries: int = 1_000_000, n_reference: int = 1_000_000) -> QueryCase:
    r_mix, r_ref, r_q = _rngs(4, 3)
    centres = r_mix.uniform(-50.0, 50.0, size=(100, 3))
    sigmas = r_mix.uniform(0.5, 3.0, size=100)
    ref = gaussian_mixture(n_reference, r_ref, centres, sigmas)
    q = gaussian_mixture(n_queries, r_q, centres, sigmas)
    return QueryCase("gmm", ref, q, leaf_size=16, extent=bbox_diagonal(ref))


CASES = {
    "tiny": tiny_case,
    "scene": scene_case,
    "lidar": lidar_case,
    "gmm": gmm_case,
    "large": large_case,
    "uniform200k": uniform200k_case,
}
