import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a) and the built libq4.so")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def parse_values(text: str) -> np.ndarray:
    """Parse a whitespace list of floats where "v*n" repeats v n times."""
    out = []
    for tok in text.split():
        if "*" in tok:
            v, n = tok.split("*")
            out.extend([float(v)] * int(n))
        else:
            out.append(float(tok))
    return np.array(out, dtype=np.float32)


def read_golden(name: str):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if not line.strip() or line.lstrip().startswith("#"):
                continue
            rows.append([p.strip() for p in line.split("|")])
    return rows


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle
