import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

_BY_TEST = {}


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size sampled parity cases")


def _records():
    mod = sys.modules.get("tests.gpu_harness")
    return None if mod is None else mod.RECORDS


def pytest_runtest_setup(item):
    rec = _records()
    if rec is not None:
        rec.clear()


def pytest_runtest_teardown(item):
    rec = _records()
    if rec and item.get_closest_marker("gpu") is not None:  # the GPU-vs-oracle comparisons
        _BY_TEST[item.nodeid] = list(rec)
    if rec:
        rec.clear()


def pytest_terminal_summary(terminalreporter):
    """Measured errors of the parity comparisons: per test, the comparison closest to its
    bound; with DLLM_PARITY_LOG=<path>, every comparison as JSON."""
    if not _BY_TEST:
        return
    tr = terminalreporter
    tr.section("parity: measured error / bound (closest comparison per test)")
    for nodeid, rec in _BY_TEST.items():
        what, e, bound = max(rec, key=lambda r: (r[1] / r[2]) if r[2] else 0.0)
        tr.write_line(f"{e:10.3g} / {bound:<8.3g} {nodeid} :: {what}")
    path = os.environ.get("DLLM_PARITY_LOG")
    if path:
        with open(path, "w") as f:
            json.dump({k: [list(r) for r in v] for k, v in _BY_TEST.items()}, f, indent=0)
