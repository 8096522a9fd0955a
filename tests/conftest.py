import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built W12 library")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover - torch missing entirely
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture
def w12_opts():
    """Setter for the library's launch options (w12_set_option); every option
    it touched gets its previous value back when the test ends."""
    from lossless_bit_weight_encode_gb300 import w12
    saved = {}

    def setopt(**values):
        for name, v in values.items():
            if name not in saved:
                saved[name] = w12.w12_get_option(name)
            w12.w12_set_option(name, int(v))

    yield setopt
    for name, v in saved.items():
        w12.w12_set_option(name, v)
