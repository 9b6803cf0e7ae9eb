import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA path through the C-ABI)")


def read_golden(name):
    """Parse a tests/golden fixture: '#' comments, 'key = value' lines, blocks split by 'name ='."""
    blocks, cur = [], {}
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if "=" in line:
                k, v = (p.strip() for p in line.split("=", 1))
                if k == "name" and cur:
                    blocks.append(cur)
                    cur = {}
                cur[k] = v
            else:
                rows.append(line.split())
    if cur:
        blocks.append(cur)
    return blocks, rows


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()


def pytest_terminal_summary(terminalreporter):
    try:
        from gpu_helpers import ERRORS
    except Exception:
        return
    real = [(lab, e) for lab, e in ERRORS if lab not in ("mismatch", "row")]
    if real:
        worst = sorted(real, key=lambda x: -x[1])[:5]
        terminalreporter.write_line(
            f"attention comparisons: {len(real)}, worst relative errors: "
            + ", ".join(f"{lab or '?'}={e:.2e}" for lab, e in worst))
