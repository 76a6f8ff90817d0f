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


def pytest_terminal_summary(terminalreporter):
    """Print every parity case's measured error next to its bar (and write the table to the
    file named by MOE_PARITY_LOG, when set)."""
    mod = sys.modules.get("tests.gpu_helpers")
    rows = getattr(mod, "ERRORS", None) if mod is not None else None
    if not rows:
        return
    lines = ["parity: max|y - y_ref| / rms(y_ref) against the bar",
             f"{'case':<44} {'error':>10} {'bar':>9} {'error/bar':>9}"]
    for case, err, bar in rows:
        lines.append(f"{case:<44} {err:10.3e} {bar:9.1e} {err / bar:9.2f}")
    terminalreporter.write_line("")
    for ln in lines:
        terminalreporter.write_line(ln)
    path = os.environ.get("MOE_PARITY_LOG")
    if path:
        with open(path, "w") as fh:
            fh.write("\n".join(lines) + "\n")
