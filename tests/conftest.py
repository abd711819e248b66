import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size parity case")


def pytest_terminal_summary(terminalreporter):
    """End-to-end comparisons measured against the plain per-element rule
    (tests/harness.py PLAIN_RECORDS), whatever tolerance each check applied."""
    h = sys.modules.get("harness")
    recs = getattr(h, "PLAIN_RECORDS", None) if h else None
    if not recs:
        return
    tr = terminalreporter
    tr.write_sep("-", "end-to-end results against the plain per-element rule")
    tr.write_line("(bf16: 1e-2 + 1e-2|ref|; FP8 layer: 5e-2 |ref|) "
                  "tensor: elements beyond / elements, largest error/bound")
    for name, bad, n, worst in recs:
        tr.write_line(f"  {name}: {bad} / {n}, {worst:.3g}")
