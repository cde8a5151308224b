import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (runs the CUDA library)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


# worst err/bound ratio of each GPU parity case, gathered by the tests (see
# gpu_util.MARGINS) and reported at the end of the session
@pytest.fixture(scope="session")
def margins():
    import gpu_util
    return gpu_util.MARGINS


def pytest_terminal_summary(terminalreporter):
    gpu_util = sys.modules.get("gpu_util")
    rows = getattr(gpu_util, "MARGINS", None)
    if not rows:
        return
    worst = {}
    for r in rows:
        key = (r["test"], r["path"])
        if key not in worst or r["max_err_over_bound"] > worst[key]["max_err_over_bound"]:
            worst[key] = r
    terminalreporter.write_sep("-", "worst err/bound per test kind and path")
    for (test, path), r in sorted(worst.items()):
        terminalreporter.write_line(
            f"{test:12s} {path:16s} {r['max_err_over_bound']:.4f}  "
            f"({', '.join(f'{k}={v}' for k, v in r.items() if k not in ('test', 'path', 'max_err_over_bound'))})")
    out = os.environ.get("W4A16_MARGINS_FILE")  # where to keep them as JSON, if anywhere
    if out:
        import json
        with open(out, "w") as f:
            json.dump(rows, f)
