import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_sessionstart(session):
    # The library is built in-tree (stamp-cached, a few seconds when stale).
    from paged_mla_decode_08_gb300.build import build
    build()
