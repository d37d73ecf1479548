import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size parity cases (minutes)")


def load_golden(name: str) -> dict:
    """Parse a tests/golden fixture: 'x:' / 'y:' rows plus key: value settings."""
    xs, ys, meta = [], [], {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(":")
            if key == "x":
                xs.append([float(v) for v in rest.split()])
            elif key == "y":
                ys.append([float(v) for v in rest.split()])
            else:
                meta[key] = rest.strip()
    return {"x": xs, "y": ys, **meta}


@pytest.fixture(scope="session")
def orc():
    import oracle

    return oracle.default()
