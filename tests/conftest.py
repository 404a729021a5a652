import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The listed near-boundary decisions of the GPU parity tests, counted
    over the session (hash bits within 1e-4 of their hyperplane, NN choices
    within 1e-4 of tau or of the runner-up), and the worst attention error."""
    parity = sys.modules.get("parity")
    reps = getattr(parity, "ALL_REPORTS", None) if parity else None
    if not reps:
        return
    try:
        keys = ("listed_hash_bits", "differing_listed_bits", "listed_nn", "differing_listed_nn", "v_ulp_diffs")
        tot = {k: sum(getattr(r, k) for r in reps) for k in keys}
        errs = [v for r in reps for v in r.att.values()]
        worst = (max(e[0] for e in errs), max(e[1] for e in errs)) if errs else (0.0, 0.0)
        terminalreporter.write_line(
            "parity: listed hash bits {listed_hash_bits} (differing {differing_listed_bits}), listed NN decisions "
            "{listed_nn} (differing {differing_listed_nn}), stored values one ulp apart {v_ulp_diffs}; ".format(**tot)
            + f"worst attention error max {worst[0]:.3g} mean {worst[1]:.3g} over {len(errs)} comparisons")
    except Exception as e:  # a summary must never fail the run
        terminalreporter.write_line(f"parity summary unavailable: {e}")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)
