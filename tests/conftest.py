import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_sessionfinish(session, exitstatus):
    """With LLAMA_PARITY_LOG=<file>: write every GPU-vs-oracle comparison of the session as TSV
    (what, max and p99 of |gpu-ref|/(1+|ref|), the gate it was held to)."""
    path = os.environ.get("LLAMA_PARITY_LOG")
    util = sys.modules.get("gpu_util")
    if not path or util is None:
        return
    with open(path, "w", encoding="utf-8") as f:
        f.write("what\tmax\tp99\tgate\n")
        for what, mx, p99, gate in util.PARITY_LOG:
            f.write(f"{what}\t{mx:.3e}\t{p99:.3e}\t{gate}\n")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def golden(name):
    """Parse a tests/golden fixture: '#' lines are the citation, other lines 'key v1 v2 ...'."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = [float(v) for v in vals]
    return out


@pytest.fixture(scope="session")
def cuda_dev():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")
