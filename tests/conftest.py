import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def pytest_terminal_summary(terminalreporter):
    """Error statistics of every parity comparison of the run: per comparison
    the max error against its bound, the mean relative error and the LSE
    error, then the comparison closest to each bound."""
    mod = sys.modules.get("_helpers")
    stats = getattr(mod, "PARITY_STATS", None) if mod else None
    if not stats:
        return
    tr = terminalreporter
    tr.section("parity error statistics (error / bound)")
    worst = {"max": (0.0, ""), "mean": (0.0, ""), "lse": (0.0, "")}
    for label, s in stats:
        fm = s["max_err"] / s["max_bound"] if s["max_bound"] > 0 else 0.0
        fr = s["mean_rel"] / s["mean_bound"]
        fl = s["lse_err"] / s["lse_bound"]
        tr.write_line(f"{label}: max {s['max_err']:.3g}/{s['max_bound']:.3g} ({fm:.2f})  "
                      f"mean-rel {s['mean_rel']:.3g}/{s['mean_bound']:.3g} ({fr:.2f})  "
                      f"lse {s['lse_err']:.3g}/{s['lse_bound']:.3g} ({fl:.2f})  n={s['n']}")
        for k, f in (("max", fm), ("mean", fr), ("lse", fl)):
            if f > worst[k][0]:
                worst[k] = (f, label)
    for k, (f, label) in worst.items():
        tr.write_line(f"closest to the {k} bound: {f:.2f} of it ({label})")
