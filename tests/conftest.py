import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture
def kernel_forms():
    """Lets a GPU test force a kernel form with gdn_set_kernel_forms; the automatic choice is put
    back afterwards, so no other test sees the override."""
    import gated_deltanet_recurrence_gb300 as gdn
    yield gdn
    gdn.gdn_set_kernel_forms()
