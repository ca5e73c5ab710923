import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workloads")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """A table of the GPU parity runs: each one's worst output error against the oracle on the
    GPU's index set (stored-precision keys), the same against float64 keys never stored, the
    selection near-ties reported and the measured hit rate."""
    try:
        from tests.gpu_harness import REPORTS
    except Exception:
        return
    if not REPORTS:
        return
    tr = terminalreporter
    tr.write_sep("-", "GPU parity against the oracle (max |out - oracle|; vs float64 keys never stored)")
    for r in REPORTS:
        a = "-" if r["alpha"] is None else f"{r['alpha']:.2f}"
        tr.write_line(f"{r['workload'][:64]:64s} t{r['steps']:<3d} u{r['units']:<3d} abs {r['max_abs']:.2e} "
                      f"rel {r['max_rel']:.1e} unrounded {r['vs_unrounded']:.2e} ties {r['ties']} a {a}")
