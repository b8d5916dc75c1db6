import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA library)")


def pytest_sessionstart(session):
    """PKV_ORACLE_MUTANT_SRC names a changed copy of the oracle's C source (the mutation
    test plants one mistake per copy): the oracle builds and loads that copy instead,
    in PKV_ORACLE_MUTANT_BUILD."""
    src = os.environ.get("PKV_ORACLE_MUTANT_SRC")
    if src:
        import oracle
        build = os.environ["PKV_ORACLE_MUTANT_BUILD"]
        oracle._SRC = src
        oracle._BUILD = build
        oracle._LIB_PATH = os.path.join(build, "liboracle_paged.so")
