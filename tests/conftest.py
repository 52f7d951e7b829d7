import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103)")


def pytest_terminal_summary(terminalreporter):
    """Print the error statistics of every GPU-vs-oracle comparison."""
    try:
        from tests.parity import RECORDED
    except Exception:
        return
    if not RECORDED:
        return
    tr = terminalreporter
    tr.section("parity statistics (GPU vs fp64 oracle)")
    for what, st in RECORDED:
        tr.write_line(what + ": " + ", ".join(f"{k}={v:.3g}" for k, v in st.items()))
    out = os.environ.get("PARITY_STATS_OUT")
    if out:
        import json
        with open(out, "w") as fh:
            json.dump([{"what": w, **st} for w, st in RECORDED], fh, indent=1)
