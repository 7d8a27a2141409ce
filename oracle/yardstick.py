"""Algorithmic work per query of the 100k <-> 100k scene registration, counted
by the oracle's reference search (near child first, far child unless
fl(delta^2) > best) -- the fixed yardstick the benchmark divides by kernel
time to get achieved bandwidth.  Part of the test infrastructure: it calls
only the oracle and the input generators.

Per query of an ICP pass the bytes are
    16 (source record) + 8 * nodes entered + 16 * points measured
(8-byte compact node, 16-byte point record); per query of a plain NN query
add the 8-byte (index, dist2) result and count a 16-byte query record.

Usage: python -m oracle.yardstick   (prints JSON; about a minute of CPU)
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


def scene_registration_work():
    c = workloads.scene_case()
    tree = oracle.KDTree(c.target, c.leaf_size)
    dmax = c.max_corr_dist[0]
    res = oracle.icp_align(tree, c.source, c.max_iter, c.eps, dmax)
    Ts = [r["T"] for r in res["trace"]] + [res["T"]]          # every pass, final one included
    nodes_tot = 0
    pts_tot = 0
    per_pass = []
    for T in Ts:
        R32, t32 = oracle.as_kernel_rt(T)
        p = oracle.transform(R32, t32, c.source)
        _, _, nv, pv = tree.query(p, counts=True)
        nodes_tot += int(nv.sum())
        pts_tot += int(pv.sum())
        per_pass.append((float(nv.mean()), float(pv.mean())))
    n_q = len(c.source) * len(Ts)
    mean_nodes = nodes_tot / n_q
    mean_pts = pts_tot / n_q
    return {
        "workload": "scene 100k<->100k, leaf 12, max_iter 50, dmax 1.0 m, eps 1e-5",
        "passes": len(Ts),
        "solves": res["iters"],
        "mean_nodes_per_query": mean_nodes,
        "mean_points_per_query": mean_pts,
        "icp_bytes_per_query": 16 + 8 * mean_nodes + 16 * mean_pts,
        "first_pass": per_pass[0],
        "last_pass": per_pass[-1],
    }


if __name__ == "__main__":
    print(json.dumps(scene_registration_work(), indent=1))
