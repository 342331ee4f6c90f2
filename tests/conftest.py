import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The parity figures behind the GPU tests' assertions: per test, the
    largest strict row-relative error (rows held to the relative bar), the
    near-zero rows' error against their absolute bound, and the plain maximum
    with no row exempt."""
    mod = sys.modules.get("tests.gpu_util")
    recs = getattr(mod, "RECORDS", None) if mod else None
    if not recs:
        return
    worst: dict = {}
    for name, e in recs:
        w = worst.setdefault(name, {"strict": 0.0, "near_zero": 0.0, "n_near": 0, "unexempt": 0.0, "n": 0})
        w["strict"] = max(w["strict"], e["strict"])
        w["near_zero"] = max(w["near_zero"], e["near_zero"])
        w["n_near"] = max(w["n_near"], e["n_near"])
        w["unexempt"] = max(w["unexempt"], e["unexempt"])
        w["n"] += 1
    tr = terminalreporter
    tr.section("parity (row-relative, no floor)")
    overall = max(w["strict"] for w in worst.values())
    tr.write_line(f"largest strict error over {len(recs)} compared tensors: {overall:.3e}")
    tr.write_line(f"{'strict':>10} {'near0/bnd':>10} {'n_near':>6} {'unexempt':>10}  test")
    for name, w in sorted(worst.items(), key=lambda kv: -kv[1]["strict"])[:40]:
        tr.write_line(f"{w['strict']:10.3e} {w['near_zero']:10.3e} {w['n_near']:6d} "
                      f"{w['unexempt']:10.3e}  {name}")
