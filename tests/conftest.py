import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the built CUDA library")


def pytest_terminal_summary(terminalreporter):
    """Totals of the GPU-vs-oracle parity checks of this run (if any ran)."""
    try:
        from santa_harness import REPORTS
    except Exception:
        return
    if not REPORTS:
        return
    samples = sum(r.samples for _, r in REPORTS)
    excused = sum(r.excused for _, r in REPORTS)
    heads = sum(r.heads for _, r in REPORTS)
    worst = max(REPORTS, key=lambda nr: nr[1].max_out_err)
    most = max(REPORTS, key=lambda nr: nr[1].excused)
    tr = terminalreporter
    tr.write_sep("-", "parity vs the float64 oracle")
    tr.write_line(f"checks={len(REPORTS)} heads={heads} samples={samples} excused={excused} "
                  f"({excused / max(1, samples):.2e} of samples)")
    tr.write_line(f"max |out - oracle| = {worst[1].max_out_err:.2e} ({worst[0]}); "
                  f"most excused in one check: {most[1].excused} ({most[0]})")
