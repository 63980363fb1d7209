import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workload checks")


@pytest.fixture
def tune():
    """Overrides of the library's measured kernel choices (the tp_mlp_tuning.h hook) for one
    test: ``tune.set("raster", 1)``; every knob set is restored when the test ends."""
    import tensor_sharded_linear_bias_gb300 as tp

    class Tune:
        def __init__(self):
            self.saved = {}

        def set(self, knob, value):
            if knob not in self.saved:
                self.saved[knob] = tp.tp_tuning_get(knob)
            tp.tp_tuning_set(knob, int(value))

    t = Tune()
    yield t
    for k, v in t.saved.items():
        tp.tp_tuning_set(k, v)
