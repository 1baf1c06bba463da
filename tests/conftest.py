import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running full-size case")
    config.addinivalue_line("markers", "run_last: collected after every other test (a run stopping at the first "
                                       "failure has run the rest first)")


def pytest_collection_modifyitems(session, config, items):
    """Tests marked run_last go to the end of the run, in their own order."""
    last = [it for it in items if it.get_closest_marker("run_last")]
    if last:
        items[:] = [it for it in items if not it.get_closest_marker("run_last")] + last
