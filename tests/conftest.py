import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    # the exhaustive BF16 pins convert every bit pattern, NaNs included, to
    # wider floats: numpy's warning about those casts is expected
    config.addinivalue_line("filterwarnings",
                            "ignore:invalid value encountered in cast:RuntimeWarning")
