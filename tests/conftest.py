import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs on the GB300 box)")


@pytest.fixture(scope="session")
def golden():
    import json

    def load(name):
        with open(os.path.join(ROOT, "tests", "golden", name)) as f:
            return json.load(f)

    return load


def pytest_terminal_summary(terminalreporter):
    """Print the parity maxima of every workload compared in this session
    (element-wise abs and relative error, and the row-wise figure)."""
    try:
        from tests.helpers import PARITY_REPORT
    except Exception:
        return
    agg = {}
    for what, n, a, r, row, refv in PARITY_REPORT:
        if what.startswith("expected-fail:"):  # the bar's own negative tests
            continue
        key = what or "?"
        cur = agg.get(key)
        if cur is None:
            agg[key] = [n, a, r, row, refv]
        else:
            cur[0] += n
            cur[1] = max(cur[1], a)
            if r > cur[2]:
                cur[2], cur[4] = r, refv
            cur[3] = max(cur[3], row)
    if not agg:
        return
    tr = terminalreporter
    tr.write_line("parity vs the fp64 oracle (bars: abs 1e-2 or the bf16 rounding 2^-8|ref| "
                  "where larger, element rel 2e-2 with a 1e-2 floor, row rel 2e-2)")
    for key in sorted(agg):
        n, a, r, row, refv = agg[key]
        tr.write_line(f"  {key:<40s} n={n:<9d} abs={a:.2e} rel={r:.2e} (ref {refv:+.2e}) "
                      f"row={row:.2e}")
    tot = max(agg.values(), key=lambda v: v[2])
    tr.write_line(f"  ALL: {len(agg)} workloads, {sum(v[0] for v in agg.values())} elements, "
                  f"max abs {max(v[1] for v in agg.values()):.2e}, max rel {tot[2]:.2e}, "
                  f"max row rel {max(v[3] for v in agg.values()):.2e}")
