import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(autouse=True)
def _device_error_word_stays_clear(request):
    """After every GPU test: no kernel of the library gave up on a bounded wait
    (the device error word, read and cleared through w4a16_read_error_word)."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import torch
    if not torch.cuda.is_available():
        return
    import bf16_activation_quantized_gb300 as w4
    word = w4.read_error_word(clear=True)
    assert word == 0, f"a kernel recorded error bits {word:#x} in the device error word"
