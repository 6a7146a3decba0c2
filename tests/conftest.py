import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    import torch

    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """The bare parity figures of every layer-output check of the session
    (max |err| / RMS(ref) against the exact oracle value, which bound each
    case asserted), one line per check; also written to
    $MOE_PARITY_LOG when that variable names a file."""
    try:
        from tolerances import parity_log
    except ImportError:
        return
    if not parity_log:
        return
    import json

    tr = terminalreporter
    tr.section("parity figures (layer outputs against the exact oracle value)")
    # the full-size workloads last, so that they end the log
    for what, r in sorted(parity_log, key=lambda x: x[0].startswith("full")):
        if r.get("dtype") == "f32":
            tr.write_line(f"{what}: f32 max|err|/max|ref| {r['max_err_over_max_ref']:.2e}")
            continue
        if "max_err_over_rms" not in r:
            continue
        tr.write_line(
            f"{what}: {r['dtype']} max|err|/RMS {r['max_err_over_rms']:.4f} "
            f"(stated {2e-2 if r['dtype'] == 'bf16' else 2.5e-3:g}; {r['n_above_stated']} of "
            f"{r['n']} above) rms|err|/RMS {r['rms_err_over_rms']:.2e} "
            f"max|ref|/RMS {r['max_abs_ref_over_rms']:.1f} secondary {r['max_err_over_secondary']:.2f} "
            f"[{r['check']}]")
    path = os.environ.get("MOE_PARITY_LOG")
    if path:
        with open(path, "w") as f:
            json.dump(parity_log, f, indent=1)
