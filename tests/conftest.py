"""Shared pytest setup: the ``gpu`` marker and import paths."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size parity case (minutes)")


def pytest_terminal_summary(terminalreporter):
    """The worst per-tensor and element-wise parity figures of the run."""
    try:
        import _parity
    except ImportError:
        return
    rec = [r for r in _parity.RECORD if r[2] is not None]
    if not rec:
        return
    tr = terminalreporter
    tr.section("parity figures (worst 12 element-wise; bound %.3f)" % _parity.ELEM_TOL)
    for name, rel, el in sorted(rec, key=lambda r: -r[2])[:12]:
        tr.write_line(f"{name:40s} per-tensor {rel:.3e}  element-wise {el:.3e}")
    tr.write_line(f"{len(rec)} tensor comparisons; worst per-tensor {max(r[1] for r in rec):.3e}, "
                  f"worst element-wise {max(r[2] for r in rec):.3e}")
