import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103)")


@pytest.fixture(scope="session")
def built_lib():
    """Builds (if needed) and loads the CUDA library."""
    from mqa_attention_gb300 import build as b
    import mqa_attention_gb300 as m

    b.build()
    return m.lib()
