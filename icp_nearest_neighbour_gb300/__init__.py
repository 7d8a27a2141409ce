"""Python binding of libicpnn (KD-tree nearest neighbour + ICP on one GB300).

Argument marshalling only: every step of the computation runs in the C/CUDA
library (``libicpnn.so``, built in-tree by ``_build.build()``).  There is no
fallback: if the library is missing or fails to load, importing the functions
raises.  Functions carry the C names without the ``icpnn_`` prefix; see
``include/icpnn.h`` for the full contract of each call.

Arrays may be NumPy arrays (host memory) or torch tensors (host or CUDA
memory); points are (n, 3) float32, C-contiguous.  PyTorch is used only to
hold device memory and to name the stream.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from ._build import LIB as _LIB_PATH, build as _build_library

__all__ = [
    "IcpnnError", "KDTree", "Moments", "IterRecord", "load", "kdtree_build", "kdtree_upload",
    "kdtree_free", "kdtree_info", "kdtree_export", "nn_query", "icp_step", "icp_step_noalloc",
    "kabsch", "icp_align", "icp_align_batch", "voxel_downsample",
    "last_error", "launch_count", "MORTON_SORT", "TRACE_TIMING", "RESIDUAL_REJECT", "NO_PRELAUNCH", "NO_PERSISTENT", "MAX_DEPTH",
    "NOALLOC_MAX_POINTS", "OVERLAP_WARN_RATIO", "LowOverlapWarning",
]

MORTON_SORT = 1
TRACE_TIMING = 2
RESIDUAL_REJECT = 4
SPLIT_ROUND_ROBIN = 8
NO_PRELAUNCH = 16
NO_PERSISTENT = 32
MAX_DEPTH = 20
NOALLOC_MAX_POINTS = 1 << 20
OVERLAP_WARN_RATIO = 0.8

STATUS = {
    0: "OK", -1: "INVALID_ARG", -2: "NOT_UPLOADED", -3: "CUDA", -4: "DEGENERATE",
    -5: "TREE_DEPTH", -6: "NONFINITE", -7: "NO_MEMORY",
}


class IcpnnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code
        self.status = STATUS.get(code, str(code))


class LowOverlapWarning(UserWarning):
    """A registration ended with fewer than OVERLAP_WARN_RATIO of the source
    points matched within the maximum correspondence distance."""


class Moments(ctypes.Structure):
    _fields_ = [("n_accepted", ctypes.c_int64), ("n_nonfinite", ctypes.c_int64),
                ("mu_src", ctypes.c_double * 3), ("mu_tgt", ctypes.c_double * 3),
                ("H", ctypes.c_double * 9), ("sum_d2", ctypes.c_double), ("mse", ctypes.c_double)]

    def as_dict(self):
        return {"n_accepted": self.n_accepted, "n_nonfinite": self.n_nonfinite,
                "mu_src": np.array(self.mu_src[:]), "mu_tgt": np.array(self.mu_tgt[:]),
                "H": np.array(self.H[:]).reshape(3, 3), "sum_d2": self.sum_d2, "mse": self.mse}


class IterRecord(ctypes.Structure):
    _fields_ = [("iter", ctypes.c_int32), ("flags", ctypes.c_int32), ("n_accepted", ctypes.c_int64),
                ("n_inliers", ctypes.c_int64), ("mse", ctypes.c_double), ("sigma2", ctypes.c_double),
                ("T", ctypes.c_double * 16), ("kernel_ms", ctypes.c_float), ("residual_ms", ctypes.c_float)]


_lib = None


def load(build_if_missing: bool = False):
    """Load libicpnn.so (building it first only when asked).  The environment
    variable ICPNN_LIBRARY may name another build of the library to load."""
    global _lib
    if _lib is not None:
        return _lib
    path = os.environ.get("ICPNN_LIBRARY", _LIB_PATH)
    if build_if_missing and path == _LIB_PATH:
        _build_library()
    if not os.path.exists(path):
        raise RuntimeError(f"libicpnn.so not built ({path}); run __graft_entry__.build() "
                           "or python -m icp_nearest_neighbour_gb300._build")
    lib = ctypes.CDLL(path)
    P, i64, i32, u32, f64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32,
                             ctypes.c_double)
    sig = {
        "icpnn_kdtree_build": ([P, i64, i32, i32, u32, ctypes.POINTER(P)], ctypes.c_int),
        "icpnn_kdtree_build_device": ([P, i64, i32, i32, u32, ctypes.POINTER(P), P], ctypes.c_int),
        "icpnn_kdtree_upload": ([P, P], ctypes.c_int),
        "icpnn_kdtree_free": ([P], None),
        "icpnn_kdtree_info": ([P, P, P, P, P, P], ctypes.c_int),
        "icpnn_kdtree_export": ([P, i64, P, P, P, P, P, P, P], ctypes.c_int),
        "icpnn_nn_query": ([P, P, i64, P, P, u32, P], ctypes.c_int),
        "icpnn_icp_step": ([P, P, i64, P, P, f64, P, P, P, P], ctypes.c_int),
        "icpnn_icp_step_noalloc": ([P, P, i64, P, P, f64, P, P, P, P], ctypes.c_int),
        "icpnn_kabsch": ([P, P], ctypes.c_int),
        "icpnn_icp_align": ([P, P, i64, i32, f64, f64, P, P, P, P, P, P, i32, u32, P], ctypes.c_int),
        "icpnn_icp_align_batch": ([P, i32, P, P, i32, f64, f64, P, P, P, P, P, P, u32, i32, P], ctypes.c_int),
        "icpnn_voxel_downsample": ([P, i64, ctypes.c_float, P, P, P], ctypes.c_int),
        "icpnn_last_error": ([], ctypes.c_char_p),
        "icpnn_launch_count": ([], i64),
        "icpnn_version": ([], i32),
        "icpnn_probe_l2_read": ([P, i64, i32, P, P], ctypes.c_int),
        "icpnn_probe_command_wait": ([P, P, i64, ctypes.c_uint64, i32, P, P], ctypes.c_int),
        "icpnn_probe_delay_commands": ([i32, i32, ctypes.c_uint64], ctypes.c_int),
        "icpnn_probe_delay_collect": ([i32, i32, ctypes.c_uint64], ctypes.c_int),
        "icpnn_probe_read_result": ([P, i64, ctypes.c_uint64, P, P, P], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def last_error() -> str:
    return load().icpnn_last_error().decode()


def launch_count() -> int:
    return int(load().icpnn_launch_count())


def _check(rc: int):
    if rc != 0:
        raise IcpnnError(rc, last_error())


# ---------------------------------------------------------------- marshalling

def _is_torch(x) -> bool:
    return type(x).__module__.startswith("torch")


def _ptr(x, dtype, shape_last=None, name="array"):
    """Address of a contiguous array of the given numpy dtype (None -> NULL)."""
    if x is None:
        return None
    if _is_torch(x):
        import torch
        tdt = {np.float32: torch.float32, np.int32: torch.int32, np.float64: torch.float64}[dtype]
        if x.dtype != tdt or not x.is_contiguous():
            raise TypeError(f"{name}: expected a contiguous {tdt} tensor")
        if shape_last is not None and (x.dim() != 2 or x.shape[1] != shape_last):
            raise TypeError(f"{name}: expected shape (n, {shape_last})")
        return ctypes.c_void_p(x.data_ptr())
    if not isinstance(x, np.ndarray) or x.dtype != dtype or not x.flags.c_contiguous:
        raise TypeError(f"{name}: expected a C-contiguous numpy {np.dtype(dtype)} array")
    if shape_last is not None and (x.ndim != 2 or x.shape[1] != shape_last):
        raise TypeError(f"{name}: expected shape (n, {shape_last})")
    return ctypes.c_void_p(x.ctypes.data)


def _stream(stream):
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available():
                return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        except ImportError:
            pass
        return None
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


# ---------------------------------------------------------------- tree

class KDTree:
    """Owner of an ``icpnn_tree`` handle."""

    def __init__(self, handle):
        self._h = handle

    @property
    def handle(self):
        if self._h is None:
            raise ValueError("tree has been freed")
        return self._h

    def free(self):
        if self._h is not None and _lib is not None:
            _lib.icpnn_kdtree_free(self._h)
        self._h = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass

    def info(self):
        return kdtree_info(self)


def kdtree_build(points, leaf_size: int, max_depth: int = -1, round_robin: bool = False) -> KDTree:
    """Host build of the target tree; round_robin picks the x, y, z, ... axis rule."""
    pts = np.ascontiguousarray(points, dtype=np.float32).reshape(-1, 3)
    lib = load()
    h = ctypes.c_void_p()
    _check(lib.icpnn_kdtree_build(_ptr(pts, np.float32, 3, "points"), len(pts), int(leaf_size),
                                  int(max_depth), SPLIT_ROUND_ROBIN if round_robin else 0, ctypes.byref(h)))
    return KDTree(h)


def kdtree_build_device(points, leaf_size: int, max_depth: int = -1, round_robin: bool = False,
                        stream=None) -> KDTree:
    """Device build of the same tree (points: a CUDA tensor, or host array);
    the tree is left on the device, already uploaded."""
    if not _is_torch(points):
        points = np.ascontiguousarray(points, dtype=np.float32).reshape(-1, 3)
    lib = load()
    h = ctypes.c_void_p()
    _check(lib.icpnn_kdtree_build_device(_ptr(points, np.float32, 3, "points"), int(points.shape[0]),
                                         int(leaf_size), int(max_depth),
                                         SPLIT_ROUND_ROBIN if round_robin else 0, ctypes.byref(h),
                                         _stream(stream)))
    return KDTree(h)


def probe_l2_read(buf, repeats: int, sink, stream=None):
    """Measurement helper: `repeats` L1-bypassing read passes over a device
    buffer (a CUDA tensor whose byte size is a multiple of 16) in one launch."""
    _check(load().icpnn_probe_l2_read(ctypes.c_void_p(buf.data_ptr()), buf.numel() * buf.element_size(),
                                      int(repeats), ctypes.c_void_p(sink.data_ptr()), _stream(stream)))


def probe_command_wait(tree: KDTree, src, wait_ns: int, mode: int, stream=None) -> int:
    """Test helper: one pre-launched pass whose blocks wait at most wait_ns for
    their command; mode 0 sends none, 1 the stop command, 2 the identity.
    Returns what the pass published: 0 nothing, 1 the abort marker, 2 its result."""
    out = ctypes.c_int32(-1)
    _check(load().icpnn_probe_command_wait(tree.handle, _ptr(src, np.float32, 3, "src"), int(src.shape[0]),
                                           int(wait_ns), int(mode), ctypes.byref(out), _stream(stream)))
    return out.value


def probe_delay_commands(skip: int, count: int, delay_ns: int):
    """Test helper: on this thread, write the next `count` transform commands to
    pre-launched passes (after `skip` normal ones) only after sleeping delay_ns."""
    _check(load().icpnn_probe_delay_commands(int(skip), int(count), int(delay_ns)))


def probe_delay_collect(skip: int, count: int, delay_ns: int):
    """Test helper: on this thread, start the next `count` reads of a
    pre-launched pass's result (after `skip` normal ones) only after sleeping
    delay_ns, between queuing the successor pass and reading the result."""
    _check(load().icpnn_probe_delay_collect(int(skip), int(count), int(delay_ns)))


RESULT_WORDS = 38  # 64-bit words of a pass's published result


def probe_read_result(words, seq: int):
    """Test helper: the host's reader of a pass's published result applied to
    `words` (RESULT_WORDS uint64 on the host).  Returns (slots, pass_ms) once
    every word carries pass `seq`'s tag, else None."""
    w = np.ascontiguousarray(words, dtype=np.uint64)
    slots = np.zeros(18, dtype=np.float64)
    ms = ctypes.c_float(0.0)
    complete = ctypes.c_int32(0)
    _check(load().icpnn_probe_read_result(w.ctypes.data_as(ctypes.c_void_p), int(w.size), int(seq),
                                          slots.ctypes.data_as(ctypes.c_void_p), ctypes.byref(ms),
                                          ctypes.byref(complete)))
    return (slots, float(ms.value)) if complete.value else None


def kdtree_upload(tree: KDTree, stream=None):
    _check(load().icpnn_kdtree_upload(tree.handle, _stream(stream)))


def kdtree_free(tree: KDTree):
    tree.free()


def kdtree_info(tree: KDTree) -> dict:
    n = ctypes.c_int64()
    leaf = ctypes.c_int32()
    md = ctypes.c_int32()
    depth = ctypes.c_int32()
    nodes = ctypes.c_int64()
    _check(load().icpnn_kdtree_info(tree.handle, ctypes.byref(n), ctypes.byref(leaf), ctypes.byref(md),
                                    ctypes.byref(depth), ctypes.byref(nodes)))
    return {"n_points": n.value, "leaf_size": leaf.value, "max_depth": md.value, "depth": depth.value,
            "n_nodes": nodes.value}


def kdtree_export(tree: KDTree) -> dict:
    info = kdtree_info(tree)
    m, n = info["n_nodes"], info["n_points"]
    out = {"split_val": np.empty(m, np.float32), "split_dim": np.empty(m, np.int32),
           "left": np.empty(m, np.int32), "right": np.empty(m, np.int32), "start": np.empty(m, np.int32),
           "end": np.empty(m, np.int32), "leaf_index": np.empty(n, np.int32)}
    keys = ["split_val", "split_dim", "left", "right", "start", "end", "leaf_index"]
    _check(load().icpnn_kdtree_export(tree.handle, m, *[ctypes.c_void_p(out[k].ctypes.data) for k in keys]))
    return out


# ---------------------------------------------------------------- query / ICP

def nn_query(tree: KDTree, xyz, idx, dist2, flags: int = 0, stream=None):
    """Fill idx (int32, n) and dist2 (float32, n) with each query's exact nearest target point.

    flags=MORTON_SORT reorders the queries along a Morton curve first; the
    results are the same.  The sort costs about as much as it saves for a
    one-shot query of up to ~1M incoherent points; icp_align always sorts its
    source once and reuses the order in every pass."""
    n = int(xyz.shape[0])
    _check(load().icpnn_nn_query(tree.handle, _ptr(xyz, np.float32, 3, "xyz"), n,
                                 _ptr(idx, np.int32, None, "idx"), _ptr(dist2, np.float32, None, "dist2"),
                                 int(flags), _stream(stream)))


def icp_step(tree: KDTree, src, R, t, max_corr_dist: float = float("inf"), idx=None, dist2=None,
             stream=None) -> dict:
    """One fused correspondence pass under float32 (R, t); returns the moments as a dict."""
    R32 = np.ascontiguousarray(R, dtype=np.float32).reshape(9)
    t32 = np.ascontiguousarray(t, dtype=np.float32).reshape(3)
    m = Moments()
    _check(load().icpnn_icp_step(tree.handle, _ptr(src, np.float32, 3, "src"), int(src.shape[0]),
                                 ctypes.c_void_p(R32.ctypes.data), ctypes.c_void_p(t32.ctypes.data),
                                 float(max_corr_dist), _ptr(idx, np.int32, None, "idx"),
                                 _ptr(dist2, np.float32, None, "dist2"), ctypes.byref(m), _stream(stream)))
    return m.as_dict()


def icp_step_noalloc(tree: KDTree, src, R, t, max_corr_dist: float = float("inf"), idx=None,
                     dist2=None, stream=None) -> dict:
    """The same pass as icp_step without any allocation (device buffers only,
    at most NOALLOC_MAX_POINTS points); for callers that cannot allocate."""
    R32 = np.ascontiguousarray(R, dtype=np.float32).reshape(9)
    t32 = np.ascontiguousarray(t, dtype=np.float32).reshape(3)
    m = Moments()
    _check(load().icpnn_icp_step_noalloc(tree.handle, _ptr(src, np.float32, 3, "src"), int(src.shape[0]),
                                         ctypes.c_void_p(R32.ctypes.data), ctypes.c_void_p(t32.ctypes.data),
                                         float(max_corr_dist), _ptr(idx, np.int32, None, "idx"),
                                         _ptr(dist2, np.float32, None, "dist2"), ctypes.byref(m),
                                         _stream(stream)))
    return m.as_dict()


def kabsch(moments: dict) -> np.ndarray:
    """Host solve from a moments dict (as returned by icp_step): 4x4 transform."""
    m = Moments()
    m.n_accepted = int(moments["n_accepted"])
    m.n_nonfinite = int(moments.get("n_nonfinite", 0))
    m.mu_src[:] = [float(v) for v in moments["mu_src"]]
    m.mu_tgt[:] = [float(v) for v in moments["mu_tgt"]]
    m.H[:] = [float(v) for v in np.asarray(moments["H"]).reshape(9)]
    T = np.zeros(16)
    _check(load().icpnn_kabsch(ctypes.byref(m), ctypes.c_void_p(T.ctypes.data)))
    return T.reshape(4, 4)


def _overlap(n_accepted: int, n: int, warn: bool) -> dict:
    ratio = n_accepted / n if n else float("nan")
    low = bool(ratio < OVERLAP_WARN_RATIO)
    if low and warn:
        import warnings
        warnings.warn(f"registration overlap {ratio:.3f} is below {OVERLAP_WARN_RATIO}: "
                      f"{n_accepted} of {n} source points matched", LowOverlapWarning, stacklevel=3)
    return {"final_n_accepted": int(n_accepted), "overlap": ratio, "low_overlap": low}


def icp_align(tree: KDTree, src, max_iter: int, eps: float, max_corr_dist: float = float("inf"),
              init_T=None, trace: bool = False, timing: bool = False, residual_reject: bool = False,
              prelaunch: bool = True, persistent: bool = True, warn_overlap: bool = True,
              stream=None) -> dict:
    """Register src onto the tree's points; returns dict(T, final_mse, iters,
    final_n_accepted, overlap, low_overlap, trace).
    residual_reject adds the 3-sigma residual rejection and re-solve to every iteration;
    by default the registration runs as one persistent kernel; persistent=False
    pre-launches the passes one at a time instead, and prelaunch=False launches
    each pass only after its transform is solved (the results are the same bits).
    overlap = final_n_accepted / n; below OVERLAP_WARN_RATIO a LowOverlapWarning is
    issued (unless warn_overlap=False), as the page's section 6 advises."""
    T = np.zeros(16)
    fmse = ctypes.c_double()
    iters = ctypes.c_int32()
    n_fin = ctypes.c_int64()
    init = None
    if init_T is not None:
        init_arr = np.ascontiguousarray(init_T, dtype=np.float64).reshape(16)
        init = ctypes.c_void_p(init_arr.ctypes.data)
    cap = int(max_iter) if (trace or timing) else 0
    recs = (IterRecord * max(cap, 1))()
    flags = ((TRACE_TIMING if timing else 0) | (RESIDUAL_REJECT if residual_reject else 0)
             | (0 if prelaunch else NO_PRELAUNCH) | (0 if persistent else NO_PERSISTENT))
    _check(load().icpnn_icp_align(tree.handle, _ptr(src, np.float32, 3, "src"), int(src.shape[0]),
                                  int(max_iter), float(eps), float(max_corr_dist), init,
                                  ctypes.c_void_p(T.ctypes.data), ctypes.byref(fmse), ctypes.byref(iters),
                                  ctypes.byref(n_fin), ctypes.cast(recs, ctypes.c_void_p) if cap else None,
                                  cap, flags, _stream(stream)))
    out = {"T": T.reshape(4, 4), "final_mse": fmse.value, "iters": iters.value}
    out.update(_overlap(n_fin.value, int(src.shape[0]), warn_overlap))
    if cap:
        out["trace"] = [{"iter": r.iter, "n_accepted": r.n_accepted, "n_inliers": r.n_inliers,
                         "mse": r.mse, "sigma2": r.sigma2, "T": np.array(r.T[:]).reshape(4, 4),
                         "kernel_ms": r.kernel_ms, "residual_ms": r.residual_ms}
                        for r in recs[:min(iters.value, cap)]]
    return out


def icp_align_batch(tree: KDTree, srcs, max_iter: int, eps: float, max_corr_dist: float = float("inf"),
                    init_T=None, residual_reject: bool = False, max_concurrent: int = 4,
                    prelaunch: bool = True, stream=None) -> dict:
    """Register several sources against one tree, several frames in flight.

    Returns dict(T (n, 4, 4), final_mse (n,), iters (n,), final_n_accepted (n,),
    overlap (n,), status (n,))."""
    n = len(srcs)
    ptrs = (ctypes.c_void_p * n)(*[_ptr(x, np.float32, 3, f"srcs[{i}]").value for i, x in enumerate(srcs)])
    counts = np.ascontiguousarray([int(x.shape[0]) for x in srcs], dtype=np.int64)
    T = np.zeros((n, 16))
    fmse = np.zeros(n)
    iters = np.zeros(n, np.int32)
    n_fin = np.zeros(n, np.int64)
    status = np.zeros(n, np.int32)
    init = None
    if init_T is not None:
        init_arr = np.ascontiguousarray(init_T, dtype=np.float64).reshape(n * 16)
        init = ctypes.c_void_p(init_arr.ctypes.data)
    rc = load().icpnn_icp_align_batch(tree.handle, n, ctypes.cast(ptrs, ctypes.c_void_p),
                                      ctypes.c_void_p(counts.ctypes.data), int(max_iter), float(eps),
                                      float(max_corr_dist), init, ctypes.c_void_p(T.ctypes.data),
                                      ctypes.c_void_p(fmse.ctypes.data), ctypes.c_void_p(iters.ctypes.data),
                                      ctypes.c_void_p(n_fin.ctypes.data), ctypes.c_void_p(status.ctypes.data),
                                      (RESIDUAL_REJECT if residual_reject else 0)
                                      | (0 if prelaunch else NO_PRELAUNCH), int(max_concurrent),
                                      _stream(stream))
    out = {"T": T.reshape(n, 4, 4), "final_mse": fmse, "iters": iters, "final_n_accepted": n_fin,
           "overlap": n_fin / counts, "status": status}
    if rc != 0:
        err = IcpnnError(rc, last_error())
        err.result = out
        raise err
    return out


def voxel_downsample(xyz, voxel_size: float, stream=None):
    """Voxel-grid filter (centroid per occupied voxel).  A CUDA tensor in gives
    a CUDA tensor out, a NumPy array gives a NumPy array; shape (m, 3)."""
    n = int(xyz.shape[0])
    if _is_torch(xyz) and xyz.is_cuda:
        import torch
        out = torch.empty((max(n, 1), 3), dtype=torch.float32, device=xyz.device)
    else:
        out = np.empty((max(n, 1), 3), np.float32)
    m = ctypes.c_int64()
    _check(load().icpnn_voxel_downsample(_ptr(xyz, np.float32, 3, "xyz"), n, float(voxel_size),
                                         _ptr(out, np.float32, 3, "out"), ctypes.byref(m), _stream(stream)))
    return out[:m.value]
