import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def pytest_sessionstart(session):
    # The package loads libzeroshard.so at import; build it (and the helper
    # libraries) if missing or older than its sources.
    import synth
    import oracle
    synth.build_host()
    oracle.build()
    from importlib import util
    spec = util.spec_from_file_location(
        "_zs_build", os.path.join(ROOT, "zero_mixed_precision_shard_gb300", "_build.py"))
    mod = util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
