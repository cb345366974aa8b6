import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long CPU-only check")


def golden_values():
    vals = {}
    with open(os.path.join(ROOT, "tests", "golden", "pages_values.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                parts = line.split()
                vals[parts[0]] = float(parts[1])
    return vals
