import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the compiled library")


@pytest.fixture
def tune():
    """Set library tuning knobs (bn=, pair=, split=, swap=, group_m=, pdl=) for one test; every knob is
    back on the automatic choice afterwards."""
    import moe_grouped_gemm_tma_gb300 as dg

    def set_knobs(**knobs):
        for k, v in knobs.items():
            dg.dg_tuning_set(k, v)

    try:
        yield set_knobs
    finally:
        dg.dg_tuning_reset()
