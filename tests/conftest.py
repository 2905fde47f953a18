import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print every case's worst output and lse error next to its gate."""
    from _util import LSE_TOL, MARGINS, OUT_TOL
    if not MARGINS:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity margins (worst error per case; gates: out %.0e, lse %.0e)" % (OUT_TOL, LSE_TOL))
    for case in sorted(MARGINS):
        o, l = MARGINS[case]
        tr.write_line(f"{case:58s} out {o:.3e} ({o / OUT_TOL:5.1%} of gate)   lse {l:.3e} ({l / LSE_TOL:5.1%})")
