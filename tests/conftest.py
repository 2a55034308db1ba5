import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    # GPU tests need a device; on a host without one they are skipped, not failed,
    # unless the run asked for them explicitly with -m gpu.
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device on this host")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture
def tune():
    """Set the library's tuning knobs for one test: ``tune(tile=128, split_k=4)``
    (values may be ints or digit strings, None restores the planner's choice).
    Every knob is put back to its value from before the test afterwards."""
    import dense_fp32_matrix_06_gb300 as sg
    from dense_fp32_matrix_06_gb300 import _build
    _build.build()
    sg.load_library()
    saved = {k: sg.get_tuning(k) for k in sg.TUNING_KNOBS}

    def set_knobs(**knobs):
        for k, v in knobs.items():
            sg.set_tuning(k, None if v is None else int(v))

    yield set_knobs
    for k, v in saved.items():
        sg.set_tuning(k, v)
