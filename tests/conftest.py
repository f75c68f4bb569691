import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter):
    """Largest worst-case |gpu - ref| / tolerance ratios the GPU parity tests
    reached (1.0 is the bound).  Written as JSON too when NVFP4_PARITY_LOG
    names a file."""
    try:
        from gpu_util import WORST_RATIOS
    except ImportError:
        return
    if not WORST_RATIOS:
        return
    rows = sorted(WORST_RATIOS, key=lambda r: -r[3])
    tr = terminalreporter
    tr.write_sep("-", "parity: worst |gpu - ref| / tolerance per comparison (bound 1.0)")
    tr.write_line("comparisons: %d, elements: %d, largest ratio: %.4g" % (
        len(rows), sum(r[2] for r in rows), rows[0][3]))
    for test, what, n, worst in rows[:15]:
        tr.write_line("  %.4g  %s  (%s, %d elements)" % (worst, test, what, n))
    path = os.environ.get("NVFP4_PARITY_LOG")
    if path:
        import json
        with open(path, "w") as f:
            json.dump([{"test": t, "what": w, "elements": n, "worst_ratio": r} for t, w, n, r in rows], f,
                      indent=0)
