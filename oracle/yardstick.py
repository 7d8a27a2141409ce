"""Algorithmic work per query, counted by the oracle's reference search (near
child first, far child unless fl(delta^2) > best, no box tests, no radius
seeding) -- the fixed yardstick the benchmark divides by kernel time to get
achieved bandwidth and distance evaluations.  Part of the test
infrastructure: it calls only the oracle and the input generators.

Per query the search enters N_node nodes and measures N_pt reference points.
Bytes (8-byte compact node, 16-byte point record):
    ICP pass   16 (source record) + 8 N_node + 16 N_pt
    NN query   16 (query record) + 8 (index, dist2 result) + 8 N_node + 16 N_pt
Floating-point work: 8 N_pt float32 operations (3 subtractions, 3
multiplications, 2 additions per distance).

Per workload the statistics run over every query of the passes listed:
    tiny, scene, lidar, uniform200k -- every pass of the oracle's own
        registration (each iteration's pass and the final one);
    gmm   -- the 1M x 1M nearest-neighbour query;
    large -- the 4M / 2M registration's first pass (identity) and a pass at
        the ground-truth transform (where both stages end), over the whole
        source.

Usage: python -m oracle.yardstick [name ...]   (JSON on stdout; the scene
takes about a minute of CPU, all workloads together tens of minutes)
"""
from __future__ import annotations

import json
import math
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import oracle  # noqa: E402
import workloads  # noqa: E402

WORKERS = max(1, min(64, os.cpu_count() or 1))


def _stats(nodes: np.ndarray, pts: np.ndarray, kind: str) -> dict:
    extra = 16 if kind == "icp" else 24
    b = extra + 8 * nodes + 16 * pts
    return {
        "queries": int(len(nodes)),
        "mean_nodes_per_query": float(nodes.mean()),
        "p99_nodes_per_query": float(np.percentile(nodes, 99)),
        "mean_points_per_query": float(pts.mean()),
        "p99_points_per_query": float(np.percentile(pts, 99)),
        "bytes_per_query": float(b.mean()),
        "p99_bytes_per_query": float(np.percentile(b, 99)),
        "fp32_flops_per_query": float(8 * pts.mean()),
    }


def _pass_counts(tree, source, Ts):
    nodes, pts = [], []
    for T in Ts:
        R32, t32 = oracle.as_kernel_rt(T)
        p = oracle.transform(R32, t32, source)
        _, _, nv, pv = tree.query(p, counts=True, workers=WORKERS)
        nodes.append(nv)
        pts.append(pv)
    return np.concatenate(nodes), np.concatenate(pts)


def registration_work(name: str) -> dict:
    c = workloads.CASES[name]()
    tree = oracle.KDTree(c.target, c.leaf_size)
    dmax = c.max_corr_dist[0]
    res = oracle.icp_align(tree, c.source, c.max_iter, c.eps, dmax, workers=WORKERS)
    Ts = [r["T"] for r in res["trace"]] + [res["T"]]          # every pass, final one included
    nodes, pts = _pass_counts(tree, c.source, Ts)
    out = {"workload": name, "kind": "icp pass", "passes": len(Ts), "solves": res["iters"],
           "n_source": len(c.source)}
    out.update(_stats(nodes, pts, "icp"))
    return out


def gmm_work() -> dict:
    c = workloads.gmm_case()
    tree = oracle.KDTree(c.reference, c.leaf_size)
    _, _, nv, pv = tree.query(c.queries, counts=True, workers=WORKERS)
    out = {"workload": "gmm", "kind": "nn query", "n_queries": len(c.queries)}
    out.update(_stats(nv, pv, "nn"))
    return out


def large_work() -> dict:
    c = workloads.large_case()
    tree = oracle.KDTree(c.target, c.leaf_size)
    out = {"workload": "large", "kind": "icp pass", "n_source": len(c.source)}
    for label, T in (("identity", np.eye(4)), ("ground_truth", c.T_gt)):
        nodes, pts = _pass_counts(tree, c.source, [T])
        out[label] = _stats(nodes, pts, "icp")
    return out


def work(name: str) -> dict:
    if name == "gmm":
        return gmm_work()
    if name == "large":
        return large_work()
    return registration_work(name)


NAMES = ("tiny", "scene", "lidar", "gmm", "large", "uniform200k")


if __name__ == "__main__":
    names = sys.argv[1:] or list(NAMES)
    print(json.dumps({n: work(n) for n in names}, indent=1))
