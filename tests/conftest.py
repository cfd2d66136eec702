import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    # Without a GPU, tests marked gpu are skipped rather than failed when they
    # are selected anyway (the GPU suite is run with -m gpu on a GB300).
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


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    # Routing-exemption counts per workload (tokens whose routing was accepted
    # inside a tie band, or re-derived from the GPU's x_hat), one JSON line so
    # that the tail of a quiet run keeps them.
    try:
        from tests.parity_util import RECORDS
    except Exception:  # pragma: no cover
        return
    if RECORDS:
        import json
        short = {name: {k: v for k, v in c.items()
                        if k in ("tokens", "set_ties", "set_ties_routed_apart", "order_ties_routed_apart",
                                 "xhat_rows_differ", "rerouted_by_xhat", "max_logit_err")}
                 for name, c in sorted(RECORDS.items())}
        terminalreporter.write_line("routing exemptions: " + json.dumps(short, separators=(",", ":")))
