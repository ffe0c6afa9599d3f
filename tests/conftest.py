import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def read_golden(name):
    """Parse a tests/golden fixture: '# comment' lines, then 'NAME rows cols'
    headers followed by that many rows of numbers, or 'key value' pairs."""
    path = os.path.join(ROOT, "tests", "golden", name)
    mats, scalars = {}, {}
    with open(path) as f:
        lines = [ln.strip() for ln in f if ln.strip() and not ln.lstrip().startswith("#")]
    i = 0
    while i < len(lines):
        parts = lines[i].split()
        if len(parts) == 3 and parts[1].isdigit() and parts[2].isdigit():
            r, c = int(parts[1]), int(parts[2])
            rows = [[float(v) for v in lines[i + 1 + t].split()] for t in range(r)]
            assert all(len(row) == c for row in rows)
            mats[parts[0]] = rows
            i += 1 + r
        else:
            scalars[parts[0]] = float(parts[1])
            i += 1
    return mats, scalars
