import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def ensure_built():
    """Compile the CUDA library if it is missing or stale (nvcc cross-compiles without a GPU)."""
    import importlib.util
    path = os.path.join(ROOT, "routing_shared_expert_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("_moe_gb300_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def read_golden(name):
    """Parse a golden fixture: '# ...' comments, then 'key v1 v2 ...' lines.

    Repeated keys accumulate into a list of rows.  Values 'a/b' are fractions.
    """
    from fractions import Fraction
    out = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            parsed = [float(Fraction(v)) if "/" in v else float(v) for v in vals]
            if key in out:
                if not isinstance(out[key][0], list):
                    out[key] = [out[key]]
                out[key].append(parsed)
            else:
                out[key] = parsed
    return out


@pytest.fixture
def golden():
    return read_golden
