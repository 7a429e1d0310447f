"""Shared pytest configuration: the ``gpu`` marker and import paths."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (parity tests through the C ABI)")
    config.addinivalue_line("markers", "slow: full-size cases")


# The oracle's property tests draw their cases with hypothesis.  Where it is
# not installed (the GPU hosts have no wheelhouse) the file is left out of
# collection instead of being reported as a skipped module in a run that
# selects GPU tests only; the CPU suite, where hypothesis is present, runs it.
try:
    import hypothesis  # noqa: F401
    collect_ignore = []
except ImportError:
    collect_ignore = ["test_oracle_properties.py"]
