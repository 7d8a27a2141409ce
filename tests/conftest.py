import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device and the compiled library")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes of CPU oracle time)")


def read_fixture(name):
    """Rows of a golden text fixture, comments and blank lines dropped."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def large_oracle(oracle_mod):
    """The 4M-target / 2M-source workload with the oracle's tree and the
    oracle's nearest neighbour of every raw source point (its searches split
    over the host cores), computed once per session: the NN-only check and
    the first ICP pass (identity transform) share it."""
    import workloads as W
    c = W.large_case()
    ot = oracle_mod.KDTree(c.target, c.leaf_size)
    workers = max(1, min(64, os.cpu_count() or 1))
    idx, d2 = ot.query(c.source, workers=workers)
    return {"case": c, "tree": ot, "workers": workers, "identity_nn": (idx, d2)}
