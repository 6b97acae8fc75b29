import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print the parity report of the GPU tests: per checked case, the
    excused boundary ids (inside the 1e-3 band / needing the u-rounding
    slack), the elements of u that rounded the other way (of those that may),
    and how far q spreads (median largest q, median count of q > 1e-4)."""
    mod = sys.modules.get("parity")
    rows = getattr(mod, "REPORT", None) if mod else None
    if not rows:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity report (excused ids: band / u-slack of compared)")
    for r in rows:
        parts = [r["case"]]
        if "band" in r:
            parts.append(f"ids {r['band']}/{r['slack']} of {r['compared']}")
        if "u_flips" in r:
            parts.append(f"u flips {r['u_flips']} of {r['u_ambiguous']} ambiguous")
        if "q_max_median" in r:
            parts.append(f"q max {r['q_max_median']:.3g} live {r['q_live_median']:g}")
        if "temperature" in r and r["temperature"] != 1.0:
            parts.append(f"T {r['temperature']:.3g}")
        tr.write_line("  " + " | ".join(parts))
    out = os.environ.get("LMHEAD_REPORT_DIR", "")
    if out and os.path.isdir(out):
        import json
        with open(os.path.join(out, "parity_report.json"), "w") as fh:
            json.dump(rows, fh, indent=1)
